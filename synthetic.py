"""Seeded synthetic inputs for the int4 group-128 GEMV workloads.

This module is shared by the oracle side (tests, oracle timing) and the CUDA
side (tests, bench, smoke).  It holds input generation only -- random weights,
random activations and the workload shapes -- and none of the method's
arithmetic (no quantisation, packing, dequantisation or dot products).

Workloads follow the rumik-oss-1 int4 engine write-up (rtts.neoandmatrix.me,
"Step 3: an int4 file and a first kernel" and "Step 4: our own engine speaks"):
per layer a fused qkv+gate+up projection of 25,088 rows, an o-projection and a
down projection, 36 layers, hidden size 3072 and intermediate 8192 as fixed by
the benchmark configurations; plus a wide 65,536-row output head.

Recipe (identical for every caller):
  rng  = numpy.random.default_rng(seed)            (PCG64)
  W    = rng.standard_normal((N, K), float32) * 0.02
  if outliers: rows = rng.choice(N, round(0.01*N), replace=False); W[rows] *= 8
  X    = rng.standard_normal((B, K), float32), rounded to bf16 (nearest-even)
The decode step's matrix for layer l, projection p (0 fused, 1 o, 2 down)
uses seed = base + 3*l + p.
"""
from __future__ import annotations

import numpy as np

GROUP = 128
HIDDEN = 3072
INTERMEDIATE = 8192
FUSED_ROWS = 25088          # q + k + v + gate + up, one int4 matrix per layer
LAYERS = 36
HEAD_ROWS = 65536

# name -> (N, K, outlier rows)
SHAPES = {
    "tiny": (256, 512, False),
    "fused": (FUSED_ROWS, HIDDEN, True),
    "oproj": (HIDDEN, HIDDEN, True),
    "down": (HIDDEN, INTERMEDIATE, True),
    "head": (HEAD_ROWS, HIDDEN, True),
}

# the three projections of one decode-step layer, in launch order
LAYER_PROJS = ("fused", "oproj", "down")


def weights(N: int, K: int, seed: int, outliers: bool) -> tuple[np.ndarray, np.random.Generator]:
    """fp32 [N, K] weights ~ N(0, 0.02), 1% of rows x8 when ``outliers``.

    Returns the generator too, so activations can be drawn after the weights
    from the same stream."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(0.02)
    if outliers:
        rows = rng.choice(N, int(round(0.01 * N)), replace=False)
        w[rows] *= np.float32(8.0)
    return w, rng


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(B: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """bf16 [B, K] activations ~ N(0, 1), as uint16 bit patterns."""
    return f32_to_bf16_bits(rng.standard_normal((B, K), dtype=np.float32))


def problem(name: str, B: int = 1, seed: int = 0):
    """(W fp32 [N,K], X bf16 bits [B,K]) for a named shape."""
    N, K, outl = SHAPES[name]
    w, rng = weights(N, K, seed, outl)
    return w, activations(B, K, rng)


def decode_step_seed(base: int, layer: int, proj: int) -> int:
    return base + 3 * layer + proj


def decode_step_matrix(layer: int, proj: int, B: int = 1, base: int = 0):
    """Weights and activations of one matrix of the synthetic decode step."""
    N, K, outl = SHAPES[LAYER_PROJS[proj]]
    w, rng = weights(N, K, decode_step_seed(base, layer, proj), outl)
    return w, activations(B, K, rng)


def random_shape_problem(N: int, K: int, B: int, seed: int, outliers: bool = False):
    w, rng = weights(N, K, seed, outliers)
    return w, activations(B, K, rng)


# ------------------------------------------------------------------ attention over a KV cache
# "Step 6: flash-decoding for long clips": one decode step's attention over a cache of about
# 2,000 positions, with 4 query heads per KV head.  The head layout is read from the shapes
# above: the o-projection's input of 3072 = 24 query heads x 128, so 6 KV heads.
Q_HEADS, KV_HEADS, HEAD_DIM = 24, 6, 128
CACHE_LEN = 2000


def attention_problem(B: int, Hq: int, Hkv: int, D: int, Lmax: int, lengths, seed: int,
                      q_std: float = 1.0):
    """(Q [B, Hq, D], K [B, Hkv, Lmax, D], V [B, Hkv, Lmax, D] as bf16 bits, lengths int32 [B]).

    Recipe: rng = default_rng(seed); Q = N(0, 1) * q_std, then K = N(0, 1), then V = N(0, 1),
    each drawn as float32 in that order and rounded to bf16 (nearest-even).  q_std sets how
    peaked the softmax is (scores have standard deviation q_std * sqrt(D) * scale)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, D), dtype=np.float32) * np.float32(q_std)
    k = rng.standard_normal((B, Hkv, Lmax, D), dtype=np.float32)
    v = rng.standard_normal((B, Hkv, Lmax, D), dtype=np.float32)
    lens = np.broadcast_to(np.asarray(lengths, np.int32), (B,)).copy()
    return f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v), lens
