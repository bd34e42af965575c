"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Every mutant below is a bug one could plausibly write into the oracle: the min
term counted four times (the bug the rumik-oss-1 page reports catching with
known-answer inputs, "Step 7"), a swapped nibble order, a transposed operand, a
dropped minimum, fp16 rounding through fp32, round-half-away instead of
round-half-even, ties in argmax going to the last index.  The pins are the
same references as in test_oracle_pins.py.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import oracle.q4_oracle as Q
import synthetic
from test_oracle_pins import GOLD, brute_gemv, brute_quantise, py_f16_bits, py_f16_value


def _gemv_pins_pass():
    try:
        w, x = synthetic.random_shape_problem(5, 256, 2, seed=21, outliers=True)
        p, sb, mb = Q.quantise_pack(w)
        y = Q.gemv_packed(p, sb, mb, x)
        if not np.allclose(y, brute_gemv(p, sb, mb, x), rtol=1e-12, atol=1e-12):
            return False
        fx = json.load(open(GOLD))
        groups = {g["name"]: g for g in fx["groups"]}
        for case in fx["gemv"]:
            wk = np.array([groups[r]["w"] for r in case["rows"]], dtype=np.float32)
            K = wk.shape[1]
            xf = np.ones(K, np.float32) if case["x"] == "ones" else \
                np.array([1.0 if k % 2 == 0 else -1.0 for k in range(K)], np.float32)
            xb = synthetic.f32_to_bf16_bits(xf)[None, :]
            pk, s2, m2 = Q.quantise_pack(wk)
            if Q.gemv_packed(pk, s2, m2, xb)[0].tolist() != case["y"]:
                return False
        return True
    except Exception:
        return False


def _f16_pins_pass():
    v = 1 + 2.0 ** -11 + 2.0 ** -40
    mids = []
    for b in range(0x3C00, 0x3C40):
        lo, hi = py_f16_value(b), py_f16_value(b + 1)
        mids += [(lo + hi) / 2, math.nextafter((lo + hi) / 2, math.inf)]
    vals = np.array([v] + mids)
    want = np.array([py_f16_bits(float(t)) for t in vals], np.uint16)
    return np.array_equal(np.asarray(Q.f16_bits_rne(vals), np.uint16), want)


def _quant_pins_pass():
    try:
        if not _f16_pins_pass():
            return False
        fx = json.load(open(GOLD))
        for grp in fx["groups"]:
            c, sb, mb = Q.quantise(np.array([grp["w"]], np.float32))
            if int(sb[0, 0]) != grp["scale_bits"] or int(mb[0, 0]) != grp["min_bits"] \
                    or c[0].tolist() != grp["codes"]:
                return False
        w, _ = synthetic.weights(3, 256, 1, outliers=True)
        c, sb, mb = Q.quantise(w)
        bc, bs, bm = brute_quantise(w.tolist())
        return c.tolist() == bc and sb.tolist() == bs and mb.tolist() == bm
    except Exception:
        return False


def test_unmutated_oracle_passes_all_pins():
    assert _gemv_pins_pass() and _quant_pins_pass()


def _min_four_times(codes, sb, mb):
    s = np.repeat(Q.f16_bits_to_f64(sb), 128, axis=1)
    m = np.repeat(Q.f16_bits_to_f64(mb), 128, axis=1)
    return np.asarray(codes, np.float64) * s + 4 * m


def _min_dropped(codes, sb, mb):
    s = np.repeat(Q.f16_bits_to_f64(sb), 128, axis=1)
    return np.asarray(codes, np.float64) * s


def _unpack_swapped(packed):
    p = np.asarray(packed, np.uint8)
    out = np.empty((p.shape[0], 2 * p.shape[1]), np.uint8)
    out[:, 0::2] = p >> 4
    out[:, 1::2] = p & 15
    return out


def _matvec_reversed_x(w_hat, x_bf16):
    x = Q.bf16_bits_to_f64(np.atleast_2d(x_bf16))[:, ::-1]
    return x @ w_hat.T


def _matvec_sign(w_hat, x_bf16):
    return -(Q.bf16_bits_to_f64(np.atleast_2d(x_bf16)) @ w_hat.T)


def _f16_via_fp32(d):
    return np.asarray(d, np.float64).astype(np.float32).astype(np.float16).view(np.uint16)


def _quantise_half_away(w):
    w = np.asarray(w, np.float32)
    N, K = w.shape
    wg = w.astype(np.float64).reshape(N, K // 128, 128)
    mn, mx = wg.min(2), wg.max(2)
    sb = Q.f16_bits_rne((mx - mn) / 15)
    mb = Q.f16_bits_rne(mn)
    s = Q.f16_bits_to_f64(sb)[:, :, None]
    m = Q.f16_bits_to_f64(mb)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.floor((wg - m) / s + 0.5)
    q = np.where(s > 0, q, 0)
    return np.clip(q, 0, 15).astype(np.uint8).reshape(N, K), sb, mb


def _scale_over_16(w):
    w = np.asarray(w, np.float32)
    N, K = w.shape
    wg = w.astype(np.float64).reshape(N, K // 128, 128)
    mn, mx = wg.min(2), wg.max(2)
    sb = Q.f16_bits_rne((mx - mn) / 16)
    mb = Q.f16_bits_rne(mn)
    s = Q.f16_bits_to_f64(sb)[:, :, None]
    m = Q.f16_bits_to_f64(mb)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((wg - m) / s)
    q = np.where(s > 0, q, 0)
    return np.clip(q, 0, 15).astype(np.uint8).reshape(N, K), sb, mb


@pytest.mark.parametrize("name,attr,mutant,pins", [
    ("min counted four times", "dequantise", _min_four_times, "gemv"),
    ("min dropped", "dequantise", _min_dropped, "gemv"),
    ("nibble order swapped", "unpack", _unpack_swapped, "gemv"),
    ("x reversed (transposed index)", "matvec", _matvec_reversed_x, "gemv"),
    ("sign flipped", "matvec", _matvec_sign, "gemv"),
    ("fp16 through fp32", "f16_bits_rne", _f16_via_fp32, "quant"),
    ("round half away from zero", "quantise", _quantise_half_away, "quant"),
    ("scale divisor 16", "quantise", _scale_over_16, "quant"),
])
def test_planted_mistake_is_caught(monkeypatch, name, attr, mutant, pins):
    monkeypatch.setattr(Q, attr, mutant)
    ok = _gemv_pins_pass() if pins == "gemv" else _quant_pins_pass()
    assert not ok, f"pins did not catch: {name}"


def test_argmax_last_tie_is_caught():
    y = np.array([[1.0, 3.0, 3.0]])
    last = lambda v: np.array([len(r) - 1 - int(np.argmax(r[::-1])) for r in np.atleast_2d(v)])
    assert last(y).tolist() != [1]
    assert oracle.argmax_first(y).tolist() == [1]


def _ambiguous_reversed_sort(y_ref_row, abs_bound):
    r = np.sort(np.asarray(y_ref_row, dtype=np.float64))[::-1]
    return r.size > 1 and (r[-1] - r[-2]) <= abs_bound


def _ambiguous_smallest_gap_anywhere(y_ref_row, abs_bound):
    r = np.sort(np.asarray(y_ref_row, dtype=np.float64))
    return r.size > 1 and float(np.min(np.diff(r))) <= abs_bound


def _ambiguous_strict(y_ref_row, abs_bound):
    r = np.sort(np.asarray(y_ref_row, dtype=np.float64))
    return r.size > 1 and (r[-1] - r[-2]) < abs_bound


@pytest.mark.parametrize("mutant", [lambda y, b: True, lambda y, b: False, _ambiguous_reversed_sort,
                                    _ambiguous_smallest_gap_anywhere, _ambiguous_strict],
                         ids=["always_true", "always_false", "reversed_sort", "smallest_gap_anywhere",
                              "strict_bound"])
def test_argmax_ambiguous_mistake_is_caught(monkeypatch, mutant):
    """The pin of argmax_ambiguous (which decides whether the exact-argmax parity check may accept a
    second index) fails for each plausible mistake in it."""
    from test_oracle_pins import test_argmax_ambiguous_decides_by_the_top_two_gap as pin
    monkeypatch.setattr(oracle, "argmax_ambiguous", mutant)
    with pytest.raises(AssertionError):
        pin()
