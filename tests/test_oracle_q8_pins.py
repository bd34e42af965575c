"""Pins of the int8 output-head oracle (oracle/q8_oracle.py) against things other than itself.

The format is the rumik-oss-1 write-up's int8 head ("Steps 9-10: streaming to the
speaker": the audio head in int8 with its own kernel; "Step 2": int8 weights as torchao
quantized tensors), read as one symmetric fp16 scale per output row.  References: Python's
own binary16 packer (struct 'e'), Python's round() (half-to-even), plain loops with
math.fsum (an exactly rounded sum), closed forms (ramps, one-hot activations, zero rows,
sign symmetry) and the round-trip bound.  The planted-mistake tests at the end copy the
quantiser with one plausible bug each and check that a pin fails on it.
"""
import math

import numpy as np
import pytest

import oracle.q8_oracle as Q8
import synthetic
from oracle.q4_oracle import QuantiseRangeError, argmax_first
from test_oracle_pins import py_f16_bits, py_f16_value


def brute_quantise_rows(w):
    """Plain loops: per row s = max |w|, scale = fp16(s/127) by struct, code = round-half-even."""
    N, K = w.shape
    codes = np.zeros((N, K), np.int8)
    sb = np.zeros(N, np.uint16)
    for n in range(N):
        s = max(abs(float(v)) for v in w[n])
        bits = py_f16_bits(s / 127.0)
        sb[n] = bits
        sh = py_f16_value(bits)
        for k in range(K):
            if sh == 0.0:
                c = 0
            else:
                c = round(float(w[n, k]) / sh)  # Python rounds halves to even
                c = max(-127, min(127, c))
            codes[n, k] = c
    return codes, sb


def brute_matvec(codes, sb, x_bits):
    x = synthetic_bf16_to_float(x_bits)
    N, K = codes.shape
    out = np.zeros((x.shape[0], N))
    for b in range(x.shape[0]):
        for n in range(N):
            sh = py_f16_value(int(sb[n]))
            out[b, n] = math.fsum(int(codes[n, k]) * sh * x[b, k] for k in range(K))
    return out


def synthetic_bf16_to_float(bits):
    bits = np.atleast_2d(np.asarray(bits, np.uint16))
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ quantiser
@pytest.mark.parametrize("N,K,seed", [(1, 128, 0), (3, 256, 1), (4, 130, 2), (2, 7, 3)])
def test_quantise_matches_brute_force(N, K, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((N, K)) * rng.choice([0.02, 0.3, 7.0], (N, 1))).astype(np.float32)
    codes, sb = Q8.quantise_rows(w)
    bc, bsb = brute_quantise_rows(w)
    assert np.array_equal(sb, bsb)
    assert np.array_equal(codes, bc)


def test_quantise_ties_go_to_even():
    # scale exactly 1.0 (max 127), entries at .5: rint(2.5) = 2, rint(-3.5) = -4, rint(0.5) = 0
    w = np.array([[127.0, 2.5, -3.5, 0.5, -0.5, 126.5]], np.float32)
    codes, sb = Q8.quantise_rows(w)
    assert py_f16_value(int(sb[0])) == 1.0
    assert codes[0].tolist() == [127, 2, -4, 0, 0, 126]


def test_ramp_row_is_exact():
    # codes -127..127 at an exact fp16 scale reproduce w exactly and the codes themselves
    scale = 0.0078125  # 2**-7
    ramp = np.arange(-127, 128, dtype=np.float64)
    w = (ramp * scale).astype(np.float32)[None, :]
    codes, sb = Q8.quantise_rows(w)
    assert py_f16_value(int(sb[0])) == scale
    assert codes[0].tolist() == list(range(-127, 128))
    assert np.array_equal(Q8.dequantise(codes, sb), w.astype(np.float64))


def test_zero_row_and_sign_symmetry():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((3, 384)) * 0.02).astype(np.float32)
    w[1] = 0.0
    codes, sb = Q8.quantise_rows(w)
    assert sb[1] == 0 and not codes[1].any()
    assert not Q8.dequantise(codes, sb)[1].any()
    c2, s2 = Q8.quantise_rows(-w)
    assert np.array_equal(s2, sb) and np.array_equal(c2, -codes)


def test_round_trip_bound():
    for seed in range(3):
        w, _ = synthetic.random_shape_problem(64, 3072, 1, seed=seed, outliers=True)
        codes, sb = Q8.quantise_rows(w)
        sh = np.array([py_f16_value(int(b)) for b in sb])
        s = np.max(np.abs(w.astype(np.float64)), axis=1)
        bound = sh / 2 + 127 * np.abs(sh - s / 127)
        err = np.abs(w.astype(np.float64) - codes.astype(np.float64) * sh[:, None])
        assert np.all(err <= bound[:, None] * (1 + 1e-12))
        assert np.abs(codes).max() <= 127


def test_unrepresentable_scale_rejected():
    w = np.zeros((2, 128), np.float32)
    w[1, 5] = 65504.0 * 127 * 1.01
    with pytest.raises(QuantiseRangeError):
        Q8.quantise_rows(w)
    with pytest.raises(QuantiseRangeError):
        Q8.quantise_rows(np.full((1, 128), np.nan, np.float32))


# ------------------------------------------------------------------ GEMV and argmax
def test_matvec_matches_brute_force():
    w, x = synthetic.random_shape_problem(6, 256, 3, seed=4, outliers=True)
    codes, sb = Q8.quantise_rows(w)
    y = Q8.matvec(codes, sb, x)
    assert np.allclose(y, brute_matvec(codes, sb, x), rtol=1e-13, atol=1e-15)
    rows = [5, 0, 3]
    assert np.array_equal(Q8.matvec(codes, sb, x, rows=rows), y[:, rows])


def test_one_hot_activation_selects_a_column():
    w, _ = synthetic.random_shape_problem(40, 384, 1, seed=5)
    codes, sb = Q8.quantise_rows(w)
    k = 77
    xf = np.zeros((1, 384), np.float32)
    xf[0, k] = 1.0
    y = Q8.matvec(codes, sb, synthetic.f32_to_bf16_bits(xf))
    want = [int(codes[n, k]) * py_f16_value(int(sb[n])) for n in range(40)]
    assert y[0].tolist() == want


def test_head_argmax_first_index_and_chunking():
    w, x = synthetic.random_shape_problem(300, 256, 2, seed=6)
    codes, sb = Q8.quantise_rows(w)
    codes[17] = codes[250]          # a tie in every batch row: rows 17 and 250 are equal
    sb[17] = sb[250]
    y, idx = Q8.head_argmax(codes, sb, x, chunk=64)
    assert np.array_equal(y, Q8.matvec(codes, sb, x))
    for b in range(2):
        best = max(range(300), key=lambda n: (y[b, n], -n))
        assert idx[b] == best
    assert np.array_equal(idx, argmax_first(y))


# ------------------------------------------------------------------ planted mistakes
# (Rounding s/127 through fp32 first is not among them: for a float32 s the quotient never lies
# strictly within half an fp32 ulp of an fp16 rounding midpoint, so that variant is equivalent.)
def _mutant(kind):
    def quantise(w):
        w64 = np.asarray(w, np.float32).astype(np.float64)
        s = np.max(np.abs(w64), axis=1)
        if kind == "per_tensor_scale":
            s = np.full_like(s, s.max())
        div = 128.0 if kind == "divide_by_128" else 127.0
        sbits = np.array([py_f16_bits(float(v / div)) for v in s], np.uint16)
        sh = np.array([py_f16_value(int(b)) for b in sbits])
        q = w64 / np.where(sh == 0, 1.0, sh)[:, None]
        if kind == "floor":
            q = np.floor(q)
        elif kind == "half_away":
            q = np.sign(q) * np.floor(np.abs(q) + 0.5)
        else:
            q = np.rint(q)
        if kind == "no_clip":
            codes = q.astype(np.int64).astype(np.int8)  # wraps past 127
        else:
            codes = np.clip(q, -127, 127).astype(np.int8)
        return np.where(sh[:, None] == 0, 0, codes).astype(np.int8), sbits
    return quantise


def _pins_pass(quantise):
    rng = np.random.default_rng(0)
    cases = [
        np.array([[127.0, 2.5, -3.5, 0.5, -0.5, 126.5]], np.float32),
        (np.arange(-127, 128) * 0.0078125).astype(np.float32)[None, :],
        (rng.standard_normal((3, 256)) * rng.choice([0.02, 0.3, 7.0], (3, 1))).astype(np.float32),
        # s/127 = 1.25 * 2**-24 rounds down to the smallest fp16 subnormal: codes must clamp at 127
        np.array([[1.25 * 127 * 2.0 ** -24, -1.0 * 127 * 2.0 ** -24, 0.0]], np.float32),
    ]
    for w in cases:
        c, sb = quantise(w)
        bc, bsb = brute_quantise_rows(w)
        if not (np.array_equal(c, bc) and np.array_equal(sb, bsb)):
            return False
    return True


def test_pins_accept_the_oracle():
    assert _pins_pass(Q8.quantise_rows)


@pytest.mark.parametrize("kind", ["floor", "half_away", "divide_by_128", "no_clip", "per_tensor_scale"])
def test_pins_catch_planted_mistake(kind):
    assert not _pins_pass(_mutant(kind))
