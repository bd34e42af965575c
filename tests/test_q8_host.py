"""CPU tests of the int8 output head's host side: the packer against the oracle, bit for bit,
and the argument checks of q8_tile / q8_head that run before any launch.  No GPU needed.

The format (rumik-oss-1 write-up, "Steps 9-10: streaming to the speaker": the head in int8;
"Step 2": torchao's int8 weights) is one symmetric fp16 scale per output row.
"""
import ctypes

import numpy as np
import pytest

import oracle.q8_oracle as Q8
import synthetic
import int4_weight_only_q4_gb300 as q4
from int4_weight_only_q4_gb300 import _lib


@pytest.mark.parametrize("N,K,seed,threads", [(1, 128, 0, 1), (37, 384, 1, 3), (300, 3072, 2, 0),
                                              (5, 16384, 3, 2)])
def test_pack_matches_oracle(N, K, seed, threads):
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=seed, outliers=True)
    c, s = q4.pack_int8_host(w, threads)
    oc, osb = Q8.quantise_rows(w)
    assert np.array_equal(s, osb)
    assert np.array_equal(c, oc)


def test_pack_special_rows():
    w = np.zeros((5, 256), np.float32)
    w[0, :6] = [127.0, 2.5, -3.5, 0.5, -0.5, 126.5]          # ties to even at scale 1
    w[1, :3] = [1.25 * 127 * 2.0 ** -24, -127 * 2.0 ** -24, 0]  # subnormal scale: clamp at 127
    w[2] = (np.arange(256) - 128) * 0.0078125                 # ramp
    w[4] = -3.0                                               # constant row
    c, s = q4.pack_int8_host(w)
    oc, osb = Q8.quantise_rows(w)
    assert np.array_equal(s, osb) and np.array_equal(c, oc)
    assert c[0, :6].tolist() == [127, 2, -4, 0, 0, 126]
    assert c[1, 0] == 127 and s[3] == 0 and not c[3].any()


def test_pack_rejects_bad_input():
    L = _lib.lib
    w = np.zeros((2, 128), np.float32)
    codes = np.empty((2, 128), np.int8)
    sc = np.empty(2, np.uint16)
    w[1, 3] = np.inf
    assert L.q8_pack_host(w.ctypes.data, 2, 128, codes.ctypes.data, sc.ctypes.data, 1) == _lib.Q4_ERR_INVALID_ARG
    w[1, 3] = 65504.0 * 127 * 1.01
    assert L.q8_pack_host(w.ctypes.data, 2, 128, codes.ctypes.data, sc.ctypes.data, 1) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_pack_host(w.ctypes.data, 2, 100, codes.ctypes.data, sc.ctypes.data, 1) == \
        _lib.Q4_ERR_UNSUPPORTED_SHAPE
    assert L.q8_pack_host(None, 2, 128, codes.ctypes.data, sc.ctypes.data, 1) == _lib.Q4_ERR_INVALID_ARG


def test_tiled_bytes():
    L = _lib.lib
    assert L.q8_tiled_bytes(65536, 3072) == 4096 * 24 * 2048
    assert L.q8_tiled_bytes(17, 256) == 2 * 2 * 2048
    assert L.q8_tiled_bytes(16, 100) == 0


def test_head_argument_checks_before_any_launch():
    L = _lib.lib
    fake = 1 << 20  # 16-byte aligned dummy addresses: nothing is dereferenced before these checks
    m = _lib.q8_matrix(fake, fake, 1000, 1024, fake)
    ok_y, ok_i = fake, fake
    assert L.q8_head(ctypes.byref(m), fake, 0, ok_y, ok_i, fake, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_head(ctypes.byref(m), fake, 9, ok_y, ok_i, fake, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_head(ctypes.byref(m), fake, 1, None, None, fake, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_head(ctypes.byref(m), None, 1, ok_y, ok_i, fake, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_head(ctypes.byref(m), fake + 2, 1, ok_y, ok_i, fake, 1 << 20, None) == _lib.Q4_ERR_MISALIGNED
    bad = _lib.q8_matrix(fake, fake, 1000, 1000, fake)
    assert L.q8_head(ctypes.byref(bad), fake, 1, ok_y, ok_i, fake, 1 << 20, None) == \
        _lib.Q4_ERR_UNSUPPORTED_SHAPE
    no_tiled = _lib.q8_matrix(fake, fake, 1000, 1024, None)
    assert L.q8_head(ctypes.byref(no_tiled), fake, 1, ok_y, ok_i, fake, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_tile(ctypes.byref(m), None, 0, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q8_tile(ctypes.byref(m), fake, 16, None) == _lib.Q4_ERR_WORKSPACE


def test_sampler_argument_checks_before_any_launch():
    L = _lib.lib
    f = 1 << 20
    assert L.q4_sample_topk(f, 1, 100, 0, 1.0, f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f, 1, 100, 101, 1.0, f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f, 1, 5000, 1025, 1.0, f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f, 1, 100, 5, 0.0, f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f, 1, 100, 5, float("inf"), f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f, 1, 100, 5, float("nan"), f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(None, 1, 100, 5, 1.0, f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f, 0, 100, 5, 1.0, f, f, None, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_sample_topk(f + 2, 1, 100, 5, 1.0, f, f, None, None) == _lib.Q4_ERR_MISALIGNED


def test_flash_decode_argument_checks_before_any_launch():
    L = _lib.lib
    p = 1 << 20                                      # never dereferenced: every call fails its checks
    ws = L.q4_flash_decode_workspace_bytes(2, 24, 6, 128, 16)
    assert ws == 2 * 24 * 16 * 128 * 4 + 2 * 24 * 16 * 2 * 4
    assert L.q4_flash_decode_chunks(6, 16) == 16
    assert L.q4_flash_decode_workspace_bytes(2, 24, 5, 128, 16) == 0       # 24 not a multiple of 5
    assert L.q4_flash_decode_workspace_bytes(1, 34, 2, 128, 1) == 0        # group 17 > 16
    assert L.q4_flash_decode_workspace_bytes(1, 8, 2, 96, 1) == 0          # head_dim 96

    def call(Q=p, K=p, V=p, lens=p, B=2, Hq=24, Hkv=6, D=128, Lmax=2000, scale=0.088, C=16, O=p, w=p, nb=ws):
        return L.q4_flash_decode(Q, K, V, lens, B, Hq, Hkv, D, Lmax, scale, C, O, w, nb, None)

    E = _lib
    assert call(Q=None) == E.Q4_ERR_INVALID_ARG
    assert call(lens=None) == E.Q4_ERR_INVALID_ARG
    assert call(w=None) == E.Q4_ERR_INVALID_ARG
    assert call(B=0) == E.Q4_ERR_INVALID_ARG
    assert call(Hq=25) == E.Q4_ERR_INVALID_ARG
    assert call(Hq=102, Hkv=6) == E.Q4_ERR_INVALID_ARG                     # group 17
    assert call(C=-1) == E.Q4_ERR_INVALID_ARG and call(C=4097) == E.Q4_ERR_INVALID_ARG
    assert call(Lmax=0) == E.Q4_ERR_INVALID_ARG and call(Lmax=(1 << 30) + 1) == E.Q4_ERR_INVALID_ARG
    assert call(scale=float("nan")) == E.Q4_ERR_INVALID_ARG
    assert call(scale=float("inf")) == E.Q4_ERR_INVALID_ARG
    assert call(D=80) == E.Q4_ERR_UNSUPPORTED_SHAPE
    assert call(Q=p + 8) == E.Q4_ERR_MISALIGNED
    assert call(K=p + 4) == E.Q4_ERR_MISALIGNED
    assert call(O=p + 2) == E.Q4_ERR_MISALIGNED
    assert call(lens=p + 1) == E.Q4_ERR_MISALIGNED
    assert call(nb=ws - 1) == E.Q4_ERR_WORKSPACE
