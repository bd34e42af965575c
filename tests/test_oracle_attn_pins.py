"""Pins of the decode-attention oracle (oracle/attn_oracle.py) against things other than itself.

The operation is one decode step of grouped-query attention over a KV cache (rumik-oss-1
write-up, "Step 6: flash-decoding for long clips").  References: plain Python loops with
math.exp and math.fsum (an exactly rounded sum), closed forms (uniform keys or a zero scale give
the mean of the values; one position gives its value; two positions give the logistic weights;
a dominant key selects its value), invariants (order of the positions, what lies past the
length, a constant added to every key), and numpy's repeat for the head grouping.  Planted
mistakes at the end.
"""
import math

import numpy as np
import pytest

import oracle.attn_oracle as A
import synthetic


def f64(bits):
    return A.bf16_bits_to_f64(bits)


def brute_attention(Q, K, V, lengths, scale):
    """Python loops: scores by fsum, weights by math.exp, output by fsum."""
    B, Hq, D = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    q, k, v = f64(Q), f64(K), f64(V)
    O = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(lengths[b])
        for h in range(Hq):
            kv = h // g
            if n == 0:
                continue
            s = [scale * math.fsum(q[b, h, d] * k[b, kv, p, d] for d in range(D)) for p in range(n)]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            tot = math.fsum(w)
            for d in range(D):
                O[b, h, d] = math.fsum(w[p] * v[b, kv, p, d] for p in range(n)) / tot
    return O


def bits(a):
    return synthetic.f32_to_bf16_bits(np.asarray(a, np.float32))


# ------------------------------------------------------------------ brute force
@pytest.mark.parametrize("B,Hq,Hkv,D,L,lens,seed,qs", [
    (1, 4, 1, 8, 6, [6], 0, 1.0),
    (2, 4, 2, 16, 9, [9, 4], 1, 2.0),
    (3, 6, 3, 8, 7, [1, 7, 0], 2, 0.5),
    (2, 8, 2, 32, 20, [17, 20], 3, 3.0),
])
def test_matches_brute_force(B, Hq, Hkv, D, L, lens, seed, qs):
    Q, K, V, lengths = synthetic.attention_problem(B, Hq, Hkv, D, L, lens, seed, q_std=qs)
    scale = 1 / math.sqrt(D)
    got = A.decode_attention(Q, K, V, lengths, scale)
    want = brute_attention(Q, K, V, lengths, scale)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)


def test_heads_subset_matches_full():
    Q, K, V, lengths = synthetic.attention_problem(2, 8, 2, 16, 12, [12, 5], 4)
    full = A.decode_attention(Q, K, V, lengths, 0.25)
    sub = A.decode_attention(Q, K, V, lengths, 0.25, heads=[(1, 7), (0, 2)])
    assert np.array_equal(sub[1, 7], full[1, 7]) and np.array_equal(sub[0, 2], full[0, 2])
    assert not sub[0, 0].any()


# ------------------------------------------------------------------ closed forms
def test_uniform_keys_and_zero_scale_give_the_mean():
    rng = np.random.default_rng(5)
    Q = bits(rng.standard_normal((1, 4, 16)))
    V = bits(rng.standard_normal((1, 2, 10, 16)))
    Kd = bits(rng.standard_normal((1, 2, 10, 16)))
    Ku = np.repeat(Kd[:, :, :1], 10, axis=2)           # every key equal
    lens = np.array([7], np.int32)
    mean = np.array([[math.fsum(f64(V)[0, kv, p, d] for p in range(7)) / 7 for d in range(16)]
                     for kv in range(2)])
    for K, scale in ((Ku, 0.3), (Kd, 0.0)):
        O = A.decode_attention(Q, K, V, lens, scale)
        for h in range(4):
            assert np.allclose(O[0, h], mean[h // 2], rtol=1e-13, atol=1e-15)


def test_one_position_and_empty_cache():
    Q, K, V, _ = synthetic.attention_problem(2, 4, 2, 8, 5, [5, 5], 6)
    O = A.decode_attention(Q, K, V, np.array([1, 0], np.int32), 0.5)
    for h in range(4):
        assert np.array_equal(O[0, h], f64(V)[0, h // 2, 0])
        assert not O[1, h].any()


def test_two_positions_give_logistic_weights():
    Q, K, V, _ = synthetic.attention_problem(1, 2, 1, 32, 2, [2], 7, q_std=2.0)
    scale = 0.125
    O = A.decode_attention(Q, K, V, np.array([2], np.int32), scale)
    q, k, v = f64(Q)[0], f64(K)[0, 0], f64(V)[0, 0]
    for h in range(2):
        delta = scale * (math.fsum(q[h] * k[0]) - math.fsum(q[h] * k[1]))
        w0 = 1 / (1 + math.exp(-delta))
        assert np.allclose(O[0, h], w0 * v[0] + (1 - w0) * v[1], rtol=1e-12, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(8)
    D, L, star = 16, 50, 31
    Q = bits(np.ones((1, 1, D)))
    Kf = rng.standard_normal((1, 1, L, D)).astype(np.float32) * 0.1
    Kf[0, 0, star] = 8.0                              # score 128 * scale above the rest
    V = bits(rng.standard_normal((1, 1, L, D)))
    O = A.decode_attention(Q, bits(Kf), V, np.array([L], np.int32), 1.0)
    # the other weights are below L * exp(-(128 - 16 * 0.1 * 4)) ~ 1e-50
    assert np.allclose(O[0, 0], f64(V)[0, 0, star], rtol=0, atol=1e-40)


def test_huge_scores_stay_finite():
    Q = bits(np.full((1, 1, 8), 100.0))
    Kf = np.full((1, 1, 3, 8), 90.0, np.float32)
    Kf[0, 0, 1] = 100.0
    K = bits(Kf)
    V = bits(np.arange(24, dtype=np.float32).reshape(1, 1, 3, 8))
    O = A.decode_attention(Q, K, V, np.array([3], np.int32), 1.0)   # scores 72,000 / 80,000 / 72,000
    assert np.array_equal(O[0, 0], f64(V)[0, 0, 1])


# ------------------------------------------------------------------ invariants
def test_position_order_does_not_matter():
    Q, K, V, _ = synthetic.attention_problem(1, 8, 2, 32, 40, [40], 9, q_std=2.0)
    lens = np.array([33], np.int32)
    perm = np.random.default_rng(0).permutation(33)
    K2, V2 = K.copy(), V.copy()
    K2[:, :, :33] = K[:, :, perm]
    V2[:, :, :33] = V[:, :, perm]
    assert np.allclose(A.decode_attention(Q, K, V, lens, 0.2), A.decode_attention(Q, K2, V2, lens, 0.2),
                       rtol=1e-12, atol=1e-14)


def test_positions_past_the_length_are_ignored():
    Q, K, V, _ = synthetic.attention_problem(2, 4, 1, 16, 30, [30, 30], 10)
    lens = np.array([12, 29], np.int32)
    K2, V2 = K.copy(), V.copy()
    for b, n in enumerate(lens):
        K2[b, :, n:] = bits(np.full(16, np.nan))
        V2[b, :, n:] = bits(np.full(16, np.inf))
    assert np.array_equal(A.decode_attention(Q, K, V, lens, 0.3), A.decode_attention(Q, K2, V2, lens, 0.3))


def test_constant_added_to_every_key_changes_nothing():
    # integer-valued keys and shift: the shifted keys are exact in bf16
    rng = np.random.default_rng(11)
    Q = bits(rng.standard_normal((1, 2, 16)))
    Kf = rng.integers(-8, 9, (1, 1, 20, 16)).astype(np.float32)
    c = rng.integers(-8, 9, 16).astype(np.float32)
    V = bits(rng.standard_normal((1, 1, 20, 16)))
    lens = np.array([20], np.int32)
    a = A.decode_attention(Q, bits(Kf), V, lens, 0.25)
    b = A.decode_attention(Q, bits(Kf + c), V, lens, 0.25)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_grouping_equals_repeated_kv_heads():
    # g query heads per KV head == one KV head per query head after numpy's repeat along heads
    Q, K, V, lens = synthetic.attention_problem(2, 12, 3, 16, 15, [15, 8], 12)
    grouped = A.decode_attention(Q, K, V, lens, 0.25)
    flat = A.decode_attention(Q, np.repeat(K, 4, axis=1), np.repeat(V, 4, axis=1), lens, 0.25)
    assert np.array_equal(grouped, flat)


# ------------------------------------------------------------------ planted mistakes
def _mutant(kind):
    def attention(Q, K, V, lengths, scale):
        B, Hq, D = Q.shape
        Hkv, L = K.shape[1], K.shape[2]
        g = Hq // Hkv
        O = np.zeros((B, Hq, D))
        for b in range(B):
            n = int(lengths[b])
            if kind == "len_plus_one":
                n = min(n + 1, L)
            elif kind == "whole_cache":
                n = L
            for h in range(Hq):
                kk = h % Hkv if kind == "kv_by_modulo" else h // g
                kv = h % Hkv if kind == "values_by_modulo" else kk
                if n == 0:
                    continue
                s = f64(K[b, kk, :n]) @ f64(Q[b, h]) * (1.0 if kind == "no_scale" else scale)
                w = np.exp(s - s.max())
                den = w.max() if kind == "max_normalised" else w.sum()
                O[b, h] = (w @ f64(V[b, kv, :n])) / den
        return O
    return attention


def _pins_pass(attention):
    cases = [synthetic.attention_problem(2, 4, 2, 16, 9, [9, 4], 1, q_std=2.0),
             synthetic.attention_problem(1, 6, 3, 8, 7, [5], 2)]
    for Q, K, V, lens in cases:
        if not np.allclose(attention(Q, K, V, lens, 0.3), brute_attention(Q, K, V, lens, 0.3),
                           rtol=1e-12, atol=1e-14):
            return False
    return True


def test_pins_accept_the_oracle():
    assert _pins_pass(A.decode_attention)


@pytest.mark.parametrize("kind", ["len_plus_one", "whole_cache", "kv_by_modulo", "values_by_modulo",
                                  "no_scale", "max_normalised"])
def test_pins_catch_planted_mistake(kind):
    assert not _pins_pass(_mutant(kind))
