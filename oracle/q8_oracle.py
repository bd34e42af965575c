"""Plain CPU oracle for the int8 output-head GEMV / skinny GEMM and its argmax.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  The library under int4_weight_only_q4_gb300/
never imports it, and it imports nothing from the library.

The rumik-oss-1 int4 engine write-up (rtts.neoandmatrix.me) keeps every
projection in int4 except the output head: "Steps 9-10: streaming to the
speaker" moves the audio head to int8 with its own CUDA kernel, int4 having
cost that matrix clearly more accuracy than the others, and the closing advice
names the output head as the one matrix that needed int8.  "Step 2: int8 and int4 weights" obtains its int8 weights from
torchao's quantized tensors.  The pages give no further detail of the int8
format; the reading taken here (listed in the design notes) is torchao's int8
weight-only scheme:

  * one scale per output row (per channel), symmetric, no minimum;
  * s = max_k |w[n, k]| in float64, scale_h = fp16(s / 127) rounded once,
    nearest-even, directly from float64;
  * code = clamp(rint(w / scale_h), -127, 127) in float64 with the STORED fp16
    scale (rint = round-half-to-even); scale_h == 0 gives code 0;
  * a row whose scale does not fit in fp16 is rejected;
  * w_hat = code * scale_h, y = W_hat x in float64, argmax = lowest index
    among equal maxima (as for the int4 head).

Pins: tests/test_oracle_q8_pins.py (brute force written differently, the
round-trip bound, closed forms, planted mistakes).
"""
from __future__ import annotations

import numpy as np

from .q4_oracle import QuantiseRangeError, argmax_first, bf16_bits_to_f64, f16_bits_rne, f16_bits_to_f64

QMAX = 127  # symmetric int8 codes -127..127


def quantise_rows(w: np.ndarray):
    """fp32 [N, K] -> (codes int8 [N, K], scale bits uint16 [N])."""
    w = np.asarray(w, dtype=np.float32)
    if not np.all(np.isfinite(w)):
        raise QuantiseRangeError("non-finite weight")
    w64 = w.astype(np.float64)
    s = np.max(np.abs(w64), axis=1)                   # per-row absolute maximum
    scale_bits = f16_bits_rne(s / QMAX)                # raises if it overflows fp16
    scale_h = f16_bits_to_f64(scale_bits)
    codes = np.zeros(w.shape, dtype=np.int8)
    nz = scale_h != 0.0
    q = np.rint(w64[nz] / scale_h[nz, None])
    codes[nz] = np.clip(q, -QMAX, QMAX).astype(np.int8)
    return codes, scale_bits.astype(np.uint16)


def dequantise(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """w_hat = code * scale_h, exactly, in float64."""
    return codes.astype(np.float64) * f16_bits_to_f64(np.asarray(scale_bits, np.uint16))[:, None]


def matvec(codes: np.ndarray, scale_bits: np.ndarray, x_bits: np.ndarray, rows=None) -> np.ndarray:
    """Y[b, i] = sum_k w_hat[rows[i], k] * x[b, k] in float64 (rows: all by default)."""
    x = bf16_bits_to_f64(np.atleast_2d(np.asarray(x_bits, np.uint16)))
    if rows is not None:
        codes = codes[rows]
        scale_bits = np.asarray(scale_bits)[rows]
    return (dequantise(codes, scale_bits) @ x.T).T


def head_argmax(codes: np.ndarray, scale_bits: np.ndarray, x_bits: np.ndarray, chunk: int = 8192):
    """Logits of the whole head in row chunks, and the first index of each batch row's maximum."""
    N = codes.shape[0]
    parts = [matvec(codes[i:i + chunk], scale_bits[i:i + chunk], x_bits) for i in range(0, N, chunk)]
    y = np.concatenate(parts, axis=1)
    return y, argmax_first(y)
