"""Plain CPU oracle for the int4 group-128 weight-only GEMV / skinny GEMM.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  The library under int4_weight_only_q4_gb300/
never imports it, and it imports nothing from the library: the two share no
code, tables or constants beyond the seeded inputs of ``synthetic``.

Everything is computed in float64 with numpy, one obvious step at a time, in
the order the method is described on the rumik-oss-1 int4 engine page
(rtts.neoandmatrix.me):

  * "Step 3: an int4 file and a first kernel": every projection's rows are cut
    into runs of 128 columns, each run carrying one fp16 scale and one fp16
    minimum; the 4-bit codes are packed in pairs.  Dequantisation is
    w = code * scale + min.
  * "Step 7: why the GEMV was stuck": the GEMV is y = W x; known-answer inputs
    (e.g. all-zero codes leave only the minimum term) catch a min term that
    is counted the wrong number of times.
  * "Step 4": per-frame argmax sampling over the head logits.

and on the pure-C TTS engine page (wpnews.pro, section on batching): a
batched matvec is B independent matvecs that reuse each weight row.

Readings where the pages are silent (each is listed in the design notes):
  * scale = (max - min) / 15 with 15 = 2**4 - 1 code steps; min = group min.
  * max, min and (max - min) / 15 are taken in float64 from the fp32 weights
    and rounded to fp16 once, directly from float64, nearest-even.
  * code = clamp(rint((w - min_h) / scale_h), 0, 15) in float64 with the
    STORED fp16 scale/min; rint is round-half-to-even.  scale_h == 0 gives
    code 0 (then every dequantised value equals min_h).
  * nibble order: byte j of a row holds column 2j in bits 0-3 and column
    2j+1 in bits 4-7 (low nibble first).
  * a group whose scale or min does not fit in fp16 is rejected.
  * argmax returns the lowest index among equal maxima.

Pins: tests/test_oracle_pins.py checks every function here against brute force
written differently, Python's own fp16 packer, closed forms and hand-derived
known-answer fixtures (tests/golden/).
"""
from __future__ import annotations

import numpy as np

GROUP = 128
LEVELS = 15  # 4-bit codes 0..15


class QuantiseRangeError(ValueError):
    """A group's scale or minimum is not representable in fp16."""


# ---------------------------------------------------------------- fp16 helpers
def f16_bits_rne(d) -> np.ndarray:
    """Round float64 values to IEEE binary16, nearest-even; return uint16 bits.

    Written from the binary16 definition: 1 sign bit, 5 exponent bits (bias 15),
    10 fraction bits; subnormals are multiples of 2**-24.  Overflow raises
    QuantiseRangeError (the quantiser never wants an infinite scale).
    """
    d = np.asarray(d, dtype=np.float64)
    if not np.all(np.isfinite(d)):
        raise QuantiseRangeError("non-finite value")
    sign = np.signbit(d).astype(np.uint32) << 15
    a = np.abs(d)
    out = np.zeros(a.shape, dtype=np.uint32)

    sub = a < 2.0 ** -14
    # subnormal (and zero): value = q * 2**-24, q in [0, 1024]; q == 1024 is the
    # smallest normal, whose bit pattern 0x0400 is exactly q.
    q_sub = np.rint(a[sub] * 2.0 ** 24)
    out[sub] = q_sub.astype(np.uint32)

    nrm = ~sub
    if np.any(nrm):
        m, e = np.frexp(a[nrm])           # a = m * 2**e, m in [0.5, 1)
        E = e.astype(np.int64) - 1        # a = 1.f * 2**E
        sig = np.rint(np.ldexp(a[nrm], (10 - E).astype(np.int64)))  # in [1024, 2048]
        carry = sig >= 2048.0
        sig = np.where(carry, 1024.0, sig)
        E = E + carry
        if np.any(E > 15):
            raise QuantiseRangeError("fp16 overflow")
        out[nrm] = (((E + 15).astype(np.uint32) << 10) | (sig.astype(np.uint32) - 1024))
    return (out | sign).astype(np.uint16)


def f16_bits_to_f64(b) -> np.ndarray:
    """Exact value of binary16 bit patterns as float64 (no inf/nan expected)."""
    b = np.asarray(b, dtype=np.uint16).astype(np.int64)
    s = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    val = np.where(e == 0, f * 2.0 ** -24, np.ldexp(1024.0 + f, (e - 25).astype(np.int64)))
    return s * val


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact value of bf16 bit patterns (upper half of an fp32) as float64."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ quantiser
def quantise(w: np.ndarray):
    """fp32 weights [N, K] -> (codes uint8 [N, K] in 0..15, scale bits, min bits).

    Groups are 128 consecutive columns of one row; scale/min are uint16 fp16
    bit patterns of shape [N, K // 128].
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    if not np.all(np.isfinite(w)):
        raise QuantiseRangeError("non-finite weight")
    G = K // GROUP
    wg = w.astype(np.float64).reshape(N, G, GROUP)
    mn = wg.min(axis=2)
    mx = wg.max(axis=2)
    scale_bits = f16_bits_rne((mx - mn) / LEVELS)
    min_bits = f16_bits_rne(mn)
    scale = f16_bits_to_f64(scale_bits)[:, :, None]
    mnh = f16_bits_to_f64(min_bits)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((wg - mnh) / scale)
    q = np.where(scale > 0, q, 0.0)
    codes = np.clip(q, 0, LEVELS).astype(np.uint8).reshape(N, K)
    return codes, scale_bits, min_bits


# -------------------------------------------------------------- pack / unpack
def pack(codes: np.ndarray) -> np.ndarray:
    """codes uint8 [N, K] (0..15) -> bytes [N, K/2], column 2j low nibble, 2j+1 high."""
    c = np.asarray(codes, dtype=np.uint8)
    lo = c[:, 0::2]
    hi = c[:, 1::2]
    return (lo | (hi << 4)).astype(np.uint8)


def unpack(packed: np.ndarray) -> np.ndarray:
    """bytes [N, K/2] -> codes uint8 [N, K]."""
    p = np.asarray(packed, dtype=np.uint8)
    N, H = p.shape
    out = np.empty((N, 2 * H), dtype=np.uint8)
    out[:, 0::2] = p & 0x0F
    out[:, 1::2] = p >> 4
    return out


# --------------------------------------------------------------- dequantise
def dequantise(codes: np.ndarray, scale_bits: np.ndarray, min_bits: np.ndarray) -> np.ndarray:
    """w_hat[n, k] = code[n, k] * scale[n, k // 128] + min[n, k // 128], in float64."""
    codes = np.asarray(codes)
    N, K = codes.shape
    s = np.repeat(f16_bits_to_f64(scale_bits), GROUP, axis=1)
    m = np.repeat(f16_bits_to_f64(min_bits), GROUP, axis=1)
    return codes.astype(np.float64) * s + m


# ----------------------------------------------------------------- matvec
def matvec(w_hat: np.ndarray, x_bf16: np.ndarray) -> np.ndarray:
    """Y[b, n] = sum_k w_hat[n, k] * x[b, k] in float64; x given as bf16 bits [B, K]."""
    x = bf16_bits_to_f64(np.atleast_2d(x_bf16))
    return x @ w_hat.T


def gemv_packed(packed: np.ndarray, scale_bits, min_bits, x_bf16, rows=None, chunk=4096) -> np.ndarray:
    """Dequantise-then-matvec straight from the packed format.

    ``rows`` (optional index array) restricts the output to those rows; the
    work is done ``chunk`` rows at a time to bound memory.  Returns float64
    [B, len(rows)].
    """
    packed = np.asarray(packed)
    N = packed.shape[0]
    idx = np.arange(N) if rows is None else np.asarray(rows)
    x = np.atleast_2d(x_bf16)
    out = np.empty((x.shape[0], idx.size), dtype=np.float64)
    for s in range(0, idx.size, chunk):
        r = idx[s:s + chunk]
        w_hat = dequantise(unpack(packed[r]), np.asarray(scale_bits)[r], np.asarray(min_bits)[r])
        out[:, s:s + chunk] = matvec(w_hat, x)
    return out


def quantise_pack(w: np.ndarray):
    """Quantise then pack: the offline export job of the int4 file."""
    codes, sb, mb = quantise(w)
    return pack(codes), sb, mb


# ----------------------------------------------------------------- argmax
def argmax_first(y: np.ndarray) -> np.ndarray:
    """Per batch row of y [B, N]: index of the maximum, lowest index on ties."""
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    return np.argmax(y, axis=1).astype(np.int32)


# ------------------------------------------------------------ tolerances
def rel_err(y_test: np.ndarray, y_ref: np.ndarray) -> float:
    """max_n |y - y_ref| / max(|y_ref|, 0.01 * rms(y_ref)), per batch row.

    The element-wise relative error of the stated 2e-3 bound, with a floor of
    1% of the row's RMS so that outputs near zero do not divide by ~0.
    """
    y_test = np.atleast_2d(np.asarray(y_test, dtype=np.float64))
    y_ref = np.atleast_2d(np.asarray(y_ref, dtype=np.float64))
    worst = 0.0
    for t, r in zip(y_test, y_ref):
        rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
        den = np.maximum(np.abs(r), 0.01 * rms)
        den = np.where(den > 0, den, 1.0)
        if r.size:
            worst = max(worst, float(np.max(np.abs(t - r) / den)))
    return worst


def argmax_ambiguous(y_ref_row: np.ndarray, abs_bound: float) -> bool:
    """True when the top two logits are closer than ``abs_bound`` (either index is then correct)."""
    r = np.sort(np.asarray(y_ref_row, dtype=np.float64))
    return r.size > 1 and (r[-1] - r[-2]) <= abs_bound
