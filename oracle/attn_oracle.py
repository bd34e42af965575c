"""Plain CPU oracle for one decode step of grouped-query attention over a KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  The library never imports it, and it imports
nothing from the library.

The rumik-oss-1 write-up, "Step 6: flash-decoding for long clips", cuts each KV
head's cache into pieces that are processed in parallel, lets the grouped query
heads of one KV head form the rows of a single matrix-multiply tile, and merges
the per-piece results with a separate small kernel.  Splitting a softmax-weighted sum
into chunks and merging them reaches the same value as the one-pass sum (up to
rounding), so this oracle is the definition of the attention output itself:

    O[b, h, :] = sum_p w_p V[b, h // g, p, :],
    w_p = exp(s_p) / sum_q exp(s_q),   s_p = scale * <Q[b, h, :], K[b, h // g, p, :]>,

over the cache positions p = 0 .. len[b]-1, with g = Hq / Hkv query heads per KV
head.  Readings where the page is silent (listed in the design notes):

  * query head h reads KV head h // g (consecutive query heads share a KV head);
  * only the first len[b] positions of a sequence's cache are attended; an
    empty cache (len[b] = 0) gives O = 0;
  * Q, K and V are bf16 values (handed over as their bit patterns), the
    arithmetic here is fp64; the maximum score is subtracted before exp, which
    changes nothing mathematically and keeps exp in range.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64 values (exact)."""
    b = np.asarray(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def head_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Attention of one query vector q [D] over keys k [L, D] and values v [L, D] (fp64):
    softmax(scale * k q) weighted sum of the rows of v; zeros for L = 0."""
    if k.shape[0] == 0:
        return np.zeros(v.shape[1])
    s = (k @ q) * scale
    w = np.exp(s - s.max())
    return (w @ v) / w.sum()


def decode_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, lengths, scale: float,
                     heads=None) -> np.ndarray:
    """O [B, Hq, D] (fp64) for Q [B, Hq, D] and caches K, V [B, Hkv, Lmax, D] (bf16 bits).

    ``heads`` (optional list of (b, h) pairs) restricts the work to those outputs; the
    rest of O stays zero."""
    Q = np.asarray(Q, np.uint16)
    B, Hq, D = Q.shape
    Hkv = K.shape[1]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    g = Hq // Hkv
    O = np.zeros((B, Hq, D))
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        n = int(lengths[b])
        kvh = h // g
        O[b, h] = head_attention(bf16_bits_to_f64(Q[b, h]), bf16_bits_to_f64(K[b, kvh, :n]),
                                 bf16_bits_to_f64(V[b, kvh, :n]), scale)
    return O
