"""Pins of the sampler oracle (oracle/sampler_oracle.py) against things other than itself.

Top-k sampling with the Gumbel-max trick (rumik-oss-1 write-up, "Step 4: our own engine speaks";
"Steps 9-10": top-k by sorting 64-bit keys of float bits and index).  References: Python's own
sorted() on (value, index) keys, the closed forms of the trick (zero noise or k = 1 is the
greedy argmax; a dominant noise term selects its rank), numpy's argmax, and the Gumbel law itself
(frequencies of a seeded sample against softmax probabilities).  Planted mistakes at the end.
"""
import math

import numpy as np
import pytest

import oracle.sampler_oracle as S


def brute_rank(row):
    """Python sort on explicit keys: NaN first, value descending, index ascending."""
    def key(i):
        v = float(row[i])
        return (0, 0.0, i) if math.isnan(v) else (1, -v, i)
    return sorted(range(len(row)), key=key)


def test_rank_order_matches_python_sort():
    rng = np.random.default_rng(0)
    for trial in range(20):
        y = rng.standard_normal(300).astype(np.float32)
        y[rng.integers(0, 300, 40)] = y[rng.integers(0, 300, 40)]       # many ties
        if trial % 3 == 0:
            y[rng.integers(0, 300, 3)] = np.nan
        if trial % 4 == 0:
            y[rng.integers(0, 300, 5)] = -np.inf
        assert S.rank_order(y).tolist() == brute_rank(y)


def test_zero_noise_and_k1_are_greedy():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((4, 1000)).astype(np.float32)
    tok, idx = S.sample(y, 50, 1.0, np.zeros((4, 50), np.float32))
    assert tok.tolist() == np.argmax(y, axis=1).tolist()
    tok1, _ = S.sample(y, 1, 0.7, rng.standard_normal((4, 1)).astype(np.float32) * 100)
    assert tok1.tolist() == np.argmax(y, axis=1).tolist()
    assert idx[:, 0].tolist() == np.argmax(y, axis=1).tolist()


def test_dominant_noise_selects_its_rank():
    rng = np.random.default_rng(2)
    y = rng.standard_normal((3, 500)).astype(np.float32)
    noise = np.zeros((3, 20), np.float32)
    noise[0, 7] = noise[1, 19] = noise[2, 0] = 1e6
    tok, idx = S.sample(y, 20, 1.0, noise)
    assert tok.tolist() == [idx[0, 7], idx[1, 19], idx[2, 0]]


def test_score_rounding_is_two_float32_steps():
    # y * t is rounded to float32 before the noise is added (no fused multiply-add)
    y = np.array([[1 + 2.0 ** -23]], np.float32)
    t = np.float32(1 + 2.0 ** -23)
    noise = np.array([[-1.0]], np.float32)
    sc = S.gumbel_scores(y, np.array([[0]]), float(t), noise)
    prod = np.float32(np.float32(y[0, 0]) * t)
    assert sc[0, 0] == np.float32(prod + np.float32(-1.0))
    exact = float(y[0, 0]) * float(t) - 1.0          # what a fused multiply-add would keep
    assert float(sc[0, 0]) != exact


def test_ties_in_score_go_to_lower_rank():
    y = np.array([[3.0, 2.0, 1.0, 0.0]], np.float32)
    noise = np.array([[0.0, 1.0, 2.0, -5.0]], np.float32)   # scores 3, 3, 3, -5
    tok, idx = S.sample(y, 4, 1.0, noise)
    assert idx[0].tolist() == [0, 1, 2, 3] and tok[0] == 0


def test_gumbel_max_follows_softmax():
    # with Gumbel noise the frequencies approach softmax(y * inv_temperature) over the top k
    rng = np.random.default_rng(3)
    y = np.array([[2.0, 1.5, 1.0, 0.2, -1.0, -3.0]], np.float32)
    k, invt, n = 4, 1.3, 40000
    counts = np.zeros(6)
    u = rng.random((n, k))
    noise = S.gumbel_noise(np.clip(u, 1e-12, 1 - 1e-12))
    for i in range(n):
        tok, _ = S.sample(y, k, invt, noise[i:i + 1])
        counts[tok[0]] += 1
    p = np.exp(y[0, :k] * invt) / np.exp(y[0, :k] * invt).sum()
    assert np.all(np.abs(counts[:k] / n - p) < 0.01)
    assert counts[k:].sum() == 0


# ------------------------------------------------------------------ planted mistakes
def _mutant_sample(kind):
    def sample(y, k, invt, noise):
        y = np.atleast_2d(np.asarray(y, np.float32))
        out_t, out_i = [], []
        for b, row in enumerate(y):
            if kind == "stable_desc_by_value_only_last_index":
                order = sorted(range(row.size), key=lambda i: (-float(row[i]), -i))
            elif kind == "nan_last":
                order = sorted(range(row.size), key=lambda i: (1 if math.isnan(row[i]) else 0,
                                                               0.0 if math.isnan(row[i]) else -float(row[i]), i))
            else:
                order = brute_rank(row)
            idx = np.array(order[:k])
            if kind == "fma_score":
                sc = (row[idx].astype(np.float64) * float(invt) + noise[b].astype(np.float64))
            elif kind == "noise_by_index":
                sc = np.float32(row[idx] * np.float32(invt)) + noise[b][np.argsort(idx).argsort()]
            else:
                sc = (row[idx] * np.float32(invt)).astype(np.float32) + noise[b]
            out_i.append(idx)
            out_t.append(idx[int(np.argmax(sc))])
        return np.array(out_t), np.array(out_i)
    return sample


def _fma_case():
    """Logits (1 + a 2^-23, 0), scale 1 + b 2^-23 whose float32 product rounds up, noise (-1, n1) with
    n1 strictly between the exact and the rounded score of rank 0: two roundings pick rank 0, a
    fused multiply-add would pick rank 1."""
    eps = 2.0 ** -23
    for a in range(3000, 5000):
        for b in range(1500, 1600):
            frac = (a * b * eps) % 1.0
            if 0.65 < frac < 0.9:
                y0, t = np.float32(1 + a * eps), np.float32(1 + b * eps)
                exact = float(y0) * float(t) - 1.0
                rounded = float(np.float32(np.float32(y0 * t) - np.float32(1.0)))
                n1 = np.float32((exact + rounded) / 2)
                assert exact < float(n1) < rounded
                return (np.array([[y0, 0.0]], np.float32), 2, float(t), np.array([[-1.0, n1]], np.float32))
    raise AssertionError("no case found")


def _sampler_pins_pass(sample):
    cases = []
    y = np.array([[3.0, 2.0, 3.0, np.nan, 1.0, 2.0]], np.float32)
    cases.append((y, 4, 1.0, np.zeros((1, 4), np.float32)))
    cases.append(_fma_case())
    rng = np.random.default_rng(5)
    y3 = rng.standard_normal((1, 50)).astype(np.float32)
    n3 = np.zeros((1, 10), np.float32)
    n3[0, 9] = 1e6
    cases.append((y3, 10, 1.0, n3))
    for yy, k, t, nz in cases:
        tok, idx = sample(yy, k, t, nz)
        want_t, want_i = S.sample(yy, k, t, nz)
        ref_i = np.array([brute_rank(r)[:k] for r in yy])
        if not (np.array_equal(idx, ref_i) and np.array_equal(tok, want_t)):
            return False
    return True


def test_pins_accept_the_oracle():
    assert _sampler_pins_pass(S.sample)


@pytest.mark.parametrize("kind", ["stable_desc_by_value_only_last_index", "nan_last", "fma_score",
                                  "noise_by_index"])
def test_pins_catch_planted_mistake(kind):
    assert not _sampler_pins_pass(_mutant_sample(kind))
