"""Plain CPU oracle for top-k sampling with the Gumbel-max trick over the head's logits.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  The library never imports it, and it imports
nothing from the library.

The rumik-oss-1 write-up samples the next token on the GPU: "Step 4: our own
engine speaks" lists top-k sampling with the Gumbel-max trick, and "Steps 9-10:
streaming to the speaker" moves the sampler into kernels that rank candidates
by 64-bit integer keys built from each logit's bit pattern and its position.
Readings where the
pages are silent (listed in the design notes):

  * ranking: NaN above every number, then larger values, then the lower index
    among equal values (the same order as the argmax); the top k are the first
    k in that order, in that order (rank 0 = largest);
  * the caller supplies the randomness: noise[b, r] (fp32, Gumbel(0, 1)
    distributed, i.e. -log(-log(u)) for u uniform in (0, 1)) is added to the
    rank-r candidate;
  * score[r] = fp32(fp32(y * inv_temperature) + noise[r]), two roundings of
    IEEE binary32 arithmetic, so that the oracle and the GPU take the decision in
    the same precision; the token is the candidate with the highest score (NaN
    first, ties to the lower rank).
"""
from __future__ import annotations

import numpy as np


def rank_order(y_row: np.ndarray) -> np.ndarray:
    """Indices of one row sorted by the ranking above (NaN first, larger first, lower index first)."""
    y = np.asarray(y_row, np.float32)
    n = np.arange(y.size)
    nan = np.isnan(y)
    vals = np.where(nan, 0.0, y).astype(np.float64)
    # lexsort: last key is primary.  Primary: NaN first; then value descending; then index ascending.
    return np.lexsort((n, -vals, ~nan))


def top_k(y: np.ndarray, k: int) -> np.ndarray:
    """[B, k] indices of the k best-ranked logits per row, in rank order."""
    y = np.atleast_2d(y)
    return np.stack([rank_order(row)[:k] for row in y])


def gumbel_scores(y: np.ndarray, idx: np.ndarray, inv_temperature: float, noise: np.ndarray) -> np.ndarray:
    """float32 scores fp32(fp32(y[idx] * inv_temperature) + noise), one rounding per operation."""
    y = np.atleast_2d(np.asarray(y, np.float32))
    sel = np.take_along_axis(y, idx, axis=1)
    scaled = (sel * np.float32(inv_temperature)).astype(np.float32)
    return (scaled + np.asarray(noise, np.float32)).astype(np.float32)


def best_rank(scores_row: np.ndarray) -> int:
    """Rank with the highest score: NaN first, ties to the lower rank."""
    s = np.asarray(scores_row, np.float32)
    nan = np.flatnonzero(np.isnan(s))
    if nan.size:
        return int(nan[0])
    return int(np.argmax(s))  # numpy returns the first maximum


def sample(y: np.ndarray, k: int, inv_temperature: float, noise: np.ndarray):
    """(token [B], top-k indices [B, k]) for logits y [B, N] and noise [B, k]."""
    idx = top_k(y, k)
    sc = gumbel_scores(y, idx, inv_temperature, noise)
    tok = np.array([idx[b, best_rank(sc[b])] for b in range(idx.shape[0])], np.int64)
    return tok, idx


def gumbel_noise(u: np.ndarray) -> np.ndarray:
    """Gumbel(0, 1) noise from uniforms in (0, 1), in float64 then rounded to float32 (the inputs
    the tests hand to both sides)."""
    u = np.asarray(u, np.float64)
    return (-np.log(-np.log(u))).astype(np.float32)
