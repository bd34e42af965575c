"""Pins of the CPU oracle against things other than itself.

Each test targets a plausible mistake in the oracle: a wrong fp16 rounding
(double rounding through fp32, ties away from zero), a swapped nibble order, a
minimum term dropped or counted the wrong number of times, a transposed
operand, a wrong sign, an argmax that prefers the last maximum.  The reference
points are Python's own binary16 packer (``struct`` format 'e'), brute force
written with plain loops and ``math.fsum`` (an exactly rounded sum), closed
forms of the format defined on the rumik-oss-1 page ("Step 3": group-128 codes,
fp16 scale and minimum, w = code*scale + min) and the hand-derived
known-answer fixtures in tests/golden/known_answers.json ("Step 7":
known-answer inputs).
"""
import json
import math
import os
import struct

import numpy as np
import pytest

import oracle
import synthetic

GOLD = os.path.join(os.path.dirname(__file__), "golden", "known_answers.json")


def py_f16_bits(v: float) -> int:
    return struct.unpack("<H", struct.pack("<e", v))[0]


def py_f16_value(bits: int) -> float:
    return struct.unpack("<e", struct.pack("<H", bits))[0]


# ------------------------------------------------------------------ fp16 rounding
def test_f16_rounding_matches_python_packer_random():
    rng = np.random.default_rng(123)
    mags = np.exp2(rng.uniform(-30, 15.9, 20000)) * rng.choice([-1, 1], 20000)
    got = oracle.f16_bits_rne(mags)
    want = np.array([py_f16_bits(float(v)) for v in mags], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_f16_rounding_ties_and_near_ties():
    # every finite fp16 value, the midpoint to its successor, and +-1 ulp(fp64) around it
    vals = []
    for b in list(range(0, 0x7BFF)):
        lo, hi = py_f16_value(b), py_f16_value(b + 1)
        mid = (lo + hi) / 2.0                       # exact in fp64
        vals += [lo, mid, math.nextafter(mid, -math.inf), math.nextafter(mid, math.inf)]
    vals = np.array(vals)
    vals = np.concatenate([vals, -vals])
    got = oracle.f16_bits_rne(vals)
    want = np.array([py_f16_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_f16_no_double_rounding_through_fp32():
    # 1 + 2^-11 + 2^-40 rounds up directly, but to 1.0 via fp32 (tie then even)
    v = 1 + 2.0 ** -11 + 2.0 ** -40
    assert oracle.f16_bits_rne(np.array([v]))[0] == py_f16_bits(v) == 0x3C01


def test_f16_overflow_rejected():
    with pytest.raises(oracle.QuantiseRangeError):
        oracle.f16_bits_rne(np.array([65520.0]))
    assert oracle.f16_bits_rne(np.array([65519.99]))[0] == 0x7BFF


def test_f16_decode_all_finite_patterns():
    bits = np.array([b for b in range(65536) if (b >> 10) & 0x1F != 0x1F], dtype=np.uint16)
    got = oracle.f16_bits_to_f64(bits)
    want = np.array([py_f16_value(int(b)) for b in bits])
    assert np.array_equal(got, want)


def test_bf16_decode():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]
    got = oracle.bf16_bits_to_f64(bits)
    want = np.array([struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in bits])
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ quantiser
def brute_quantise(w):
    """Row by row, group by group, with Python floats, struct and round() (half-even)."""
    N, K = len(w), len(w[0])
    codes = [[0] * K for _ in range(N)]
    sb, mb = [], []
    for n in range(N):
        srow, mrow = [], []
        for g in range(K // 128):
            vals = [float(v) for v in w[n][g * 128:(g + 1) * 128]]
            lo, hi = min(vals), max(vals)
            s_bits = py_f16_bits((hi - lo) / 15.0)
            m_bits = py_f16_bits(lo)
            s, m = py_f16_value(s_bits), py_f16_value(m_bits)
            for j, v in enumerate(vals):
                c = 0 if s == 0 else round((v - m) / s)
                codes[n][g * 128 + j] = min(15, max(0, c))
            srow.append(s_bits)
            mrow.append(m_bits)
        sb.append(srow)
        mb.append(mrow)
    return codes, sb, mb


@pytest.mark.parametrize("N,K,seed", [(1, 128, 0), (3, 256, 1), (4, 128, 2), (4, 256, 3)])
def test_quantiser_matches_brute_force(N, K, seed):
    w, _ = synthetic.weights(N, K, seed, outliers=False)
    w[0, :128] *= 8.0                     # an outlier group
    if N > 1:
        w[1, 0:128] = np.float32(-0.25)   # a constant group
    if N > 2:
        w[2, 128 % K:128 % K + 128] = 0.0  # an all-zero group
    codes, sb, mb = oracle.quantise(w)
    bc, bs, bm = brute_quantise(w.tolist())
    assert codes.tolist() == bc
    assert sb.tolist() == bs
    assert mb.tolist() == bm


def test_known_answer_groups():
    fx = json.load(open(GOLD))
    for grp in fx["groups"]:
        w = np.array([grp["w"]], dtype=np.float32)
        codes, sb, mb = oracle.quantise(w)
        assert int(sb[0, 0]) == grp["scale_bits"], grp["name"]
        assert int(mb[0, 0]) == grp["min_bits"], grp["name"]
        assert codes[0].tolist() == grp["codes"], grp["name"]


def test_known_answer_gemv():
    fx = json.load(open(GOLD))
    groups = {g["name"]: g for g in fx["groups"]}
    for case in fx["gemv"]:
        w = np.array([groups[r]["w"] for r in case["rows"]], dtype=np.float32)
        K = w.shape[1]
        if case["x"] == "ones":
            xf = np.ones(K, np.float32)
        else:
            xf = np.array([1.0 if k % 2 == 0 else -1.0 for k in range(K)], np.float32)
        x = synthetic.f32_to_bf16_bits(xf)[None, :]
        p, sb, mb = oracle.quantise_pack(w)
        y = oracle.gemv_packed(p, sb, mb, x)[0]
        assert y.tolist() == case["y"], case["name"]


def test_roundtrip_bound():
    for name, seed in (("tiny", 0), ("oproj", 5)):
        N, K, outl = synthetic.SHAPES[name]
        w, _ = synthetic.weights(min(N, 512), K, seed, outl)
        codes, sb, mb = oracle.quantise(w)
        w_hat = oracle.dequantise(codes, sb, mb)
        wg = w.astype(np.float64).reshape(w.shape[0], -1, 128)
        mn, mx = wg.min(2), wg.max(2)
        s = oracle.f16_bits_to_f64(sb)
        m = oracle.f16_bits_to_f64(mb)
        bound = s / 2 + 15 * np.abs(s - (mx - mn) / 15) + np.abs(m - mn)
        err = np.abs(w.astype(np.float64) - w_hat).reshape(wg.shape).max(2)
        assert np.all(err <= bound * (1 + 1e-12))
        # and the plain |w - deq(q(w))| <= scale/2 up to fp16 rounding of scale/min
        assert np.all(err <= s / 2 + np.abs(m - mn) + 15 * np.abs(s - (mx - mn) / 15) + 1e-300)


# ------------------------------------------------------------------ pack
def test_pack_exhaustive_bytes():
    allb = np.arange(256, dtype=np.uint8)[None, :]
    assert np.array_equal(oracle.pack(oracle.unpack(allb)), allb)
    c = oracle.unpack(allb)[0]
    for b in range(256):
        assert c[2 * b] == b % 16 and c[2 * b + 1] == b // 16


def test_pack_known_answers():
    fx = json.load(open(GOLD))
    a, b = fx["pack"]
    assert oracle.pack(np.array([a["codes"]], np.uint8))[0].tolist() == [a["byte"]]
    assert oracle.pack(np.array([b["codes"]], np.uint8))[0].tolist() == b["bytes"]


# ------------------------------------------------------------------ matvec
def brute_gemv(packed, sb, mb, x_bits):
    """Plain loops: decode each nibble, dequantise with struct-decoded fp16, fsum."""
    N, H = packed.shape
    K = 2 * H
    out = []
    for xb in x_bits:
        xs = [struct.unpack("<f", struct.pack("<I", int(v) << 16))[0] for v in xb]
        row = []
        for n in range(N):
            terms = []
            for k in range(K):
                byte = int(packed[n, k // 2])
                code = (byte >> 4) if (k % 2) else (byte & 15)
                s = py_f16_value(int(sb[n, k // 128]))
                m = py_f16_value(int(mb[n, k // 128]))
                terms.append((code * s + m) * xs[k])
            row.append(math.fsum(terms))
        out.append(row)
    return np.array(out)


def test_gemv_matches_brute_force():
    w, x = synthetic.random_shape_problem(5, 256, 3, seed=11, outliers=True)
    p, sb, mb = oracle.quantise_pack(w)
    y = oracle.gemv_packed(p, sb, mb, x)
    yb = brute_gemv(p, sb, mb, x)
    assert np.allclose(y, yb, rtol=1e-12, atol=1e-12)
    # row subset path
    ys = oracle.gemv_packed(p, sb, mb, x, rows=np.array([4, 0]), chunk=1)
    assert np.allclose(ys, yb[:, [4, 0]], rtol=1e-12, atol=1e-12)


def _xsum_groups(x_bits, K):
    xf = oracle.bf16_bits_to_f64(x_bits)
    return xf.reshape(xf.shape[0], K // 128, 128).sum(2)


def test_closed_form_zero_codes():
    w, x = synthetic.random_shape_problem(6, 512, 2, seed=3)
    p, sb, mb = oracle.quantise_pack(w)
    p0 = np.zeros_like(p)
    y = oracle.gemv_packed(p0, sb, mb, x)
    S = _xsum_groups(x, 512)                                    # [B, G]
    want = S @ oracle.f16_bits_to_f64(mb).T                     # sum_g min_g * S_g
    assert np.allclose(y, want, rtol=1e-13, atol=1e-13)


def test_closed_form_one_hot():
    w, _ = synthetic.random_shape_problem(7, 384, 1, seed=4)
    p, sb, mb = oracle.quantise_pack(w)
    w_hat = oracle.dequantise(oracle.unpack(p), sb, mb)
    for k in (0, 1, 127, 128, 255, 383):
        x = np.zeros((1, 384), np.uint16)
        x[0, k] = 0x3F80                                        # bf16 1.0
        y = oracle.gemv_packed(p, sb, mb, x)[0]
        assert np.array_equal(y, w_hat[:, k])


def test_closed_form_all_ones_codes():
    w, _ = synthetic.random_shape_problem(4, 256, 1, seed=5)
    _, sb, mb = oracle.quantise_pack(w)
    p1 = np.full((4, 128), 0x11, np.uint8)                      # every code 1
    x = np.full((1, 256), 0x3F80, np.uint16)
    y = oracle.gemv_packed(p1, sb, mb, x)[0]
    want = 128 * (oracle.f16_bits_to_f64(sb) + oracle.f16_bits_to_f64(mb)).sum(1)
    assert np.allclose(y, want, rtol=1e-14)


def test_linearity_per_group():
    w, x = synthetic.random_shape_problem(8, 512, 1, seed=6)
    p, sb, mb = oracle.quantise_pack(w)
    y = oracle.gemv_packed(p, sb, mb, x)[0]
    w_hat = oracle.dequantise(oracle.unpack(p), sb, mb)
    xf = oracle.bf16_bits_to_f64(x)[0]
    for g in range(4):
        xz = x.copy()
        xz[0, g * 128:(g + 1) * 128] = 0
        yz = oracle.gemv_packed(p, sb, mb, xz)[0]
        term = w_hat[:, g * 128:(g + 1) * 128] @ xf[g * 128:(g + 1) * 128]
        assert np.allclose(y - yz, term, rtol=1e-10, atol=1e-12)


def test_batch_rows_independent():
    w, x = synthetic.random_shape_problem(9, 256, 4, seed=7)
    p, sb, mb = oracle.quantise_pack(w)
    y = oracle.gemv_packed(p, sb, mb, x)
    for b in range(4):
        assert np.array_equal(oracle.gemv_packed(p, sb, mb, x[b:b + 1])[0], y[b])


# ------------------------------------------------------------------ argmax + tolerance
def test_argmax_first_on_ties():
    y = np.array([[1.0, 3.0, 3.0, -1.0], [0.0, -0.0, 0.0, -5.0], [-2.0, -1.0, -1.0, -1.0]])
    got = oracle.argmax_first(y)
    want = []
    for row in y:
        best = 0
        for i, v in enumerate(row):
            if v > row[best]:
                best = i
        want.append(best)
    assert got.tolist() == want == [1, 0, 1]


def _top2_gap_by_hand(row):
    """Gap between the largest value and the largest of the others (one occurrence of the maximum
    removed), found with two plain passes -- no sort."""
    best = 0
    for i, v in enumerate(row):
        if v > row[best]:
            best = i
    second = None
    for i, v in enumerate(row):
        if i != best and (second is None or v > second):
            second = v
    return row[best] - second


def test_argmax_ambiguous_decides_by_the_top_two_gap():
    """argmax_ambiguous(y, bound) is True exactly when the two largest logits are at most `bound`
    apart.  Hand cases pin the boundary (the gap equal to the bound counts as ambiguous), a
    repeated maximum (gap 0), a single logit (never ambiguous), negative rows, and rows whose
    closest pair is not the top two (a smallest-gap-anywhere mistake fails there); a reversed
    sort, or an answer that is always True or always False, fails the hand cases."""
    cases = [
        ([1.0, 3.0, 2.75], 0.125, False), ([1.0, 3.0, 2.75], 0.25, True), ([1.0, 3.0, 2.75], 0.5, True),
        ([2.0, 5.0, 5.0, 1.0], 0.0, True), ([7.0], 1e9, False),
        ([-4.0, -1.0, -3.0], 1.5, False), ([-4.0, -1.0, -3.0], 2.0, True),
        ([5.0, 0.0, 4.0, 4.0625], 0.5, False), ([5.0, 0.0, 4.0, 4.0625], 0.9375, True),
        ([0.0, 10.0, 10.001, 3.0], 0.01, True), ([0.0, 10.0, 9.0, 3.0], 0.5, False),
    ]
    for row, bound, want in cases:
        assert bool(oracle.argmax_ambiguous(np.array(row), bound)) == want, (row, bound)
    rng = np.random.default_rng(5)
    for _ in range(200):
        row = rng.standard_normal(int(rng.integers(2, 40)))
        if rng.random() < 0.3:
            row[int(rng.integers(row.size))] = row.max()          # a repeated maximum
        gap = _top2_gap_by_hand(row.tolist())
        for bound in (0.0, gap * 0.5, gap, gap * 1.5):
            assert bool(oracle.argmax_ambiguous(row, bound)) == (gap <= bound), (row, bound)


def test_rel_err_metric():
    r = np.array([[1.0, -2.0, 0.0, 4.0]])
    assert oracle.rel_err(r, r) == 0.0
    t = r.copy()
    t[0, 1] += 2e-3 * 2.0
    assert abs(oracle.rel_err(t, r) - 2e-3) < 1e-12
    t = r.copy()
    t[0, 2] = 1e-4          # near-zero output: floor at 1% of rms
    rms = math.sqrt((1 + 4 + 16) / 4)
    assert abs(oracle.rel_err(t, r) - 1e-4 / (0.01 * rms)) < 1e-12


def test_synthetic_recipe_shapes():
    w, x = synthetic.problem("tiny", B=1, seed=0)
    assert w.shape == (256, 512) and w.dtype == np.float32
    assert x.shape == (1, 512) and x.dtype == np.uint16
    # same stream: the first activation row does not depend on B
    _, x8 = synthetic.problem("tiny", B=8, seed=0)
    assert np.array_equal(x8[0], x[0])
