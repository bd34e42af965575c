"""CPU tests of libq4.so: exported symbols, the host packer, host-side argument checks.

No test here launches a kernel or needs a GPU.  The packer must agree bit for
bit with the oracle's quantiser (same written rule, no shared code).
"""
import ctypes

import numpy as np
import pytest

import oracle
import synthetic
import int4_weight_only_q4_gb300 as q4
from int4_weight_only_q4_gb300 import _lib


def test_library_exports_every_declared_function():
    names = _lib.header_functions()
    assert {"q4_pack_host", "q4_gemv", "q4_gemm_skinny", "q4_decode_step", "q4_argmax_f32",
            "q4_workspace_bytes", "q4_decode_step_workspace_bytes", "q4_plan", "q4_device_status",
            "q4_tiled_bytes", "q4_tile", "q4_step_workspace_bytes", "q4_step_prepare", "q4_step_stream",
            "q4_status_string"} <= set(names)
    for n in names:
        assert hasattr(_lib.lib, n), n


def test_status_strings():
    for code in range(7):
        assert _lib.lib.q4_status_string(code)
    assert _lib.lib.q4_status_string(0) == b"ok"


def _pack_equal(w, n_threads=0):
    c, s, m = q4.pack_host(w, n_threads)
    oc, osb, omb = oracle.quantise(w)
    assert np.array_equal(s, osb)
    assert np.array_equal(m, omb)
    assert np.array_equal(c, oracle.pack(oc))


@pytest.mark.parametrize("name", ["tiny"])
def test_pack_matches_oracle_tiny(name):
    w, _ = synthetic.problem(name, 1, seed=0)
    _pack_equal(w)
    _pack_equal(w, n_threads=1)
    _pack_equal(w, n_threads=7)


@pytest.mark.parametrize("N,K,seed,outl", [(1, 128, 1, False), (13, 384, 2, True), (64, 1152, 3, True),
                                          (300, 3072, 4, True)])
def test_pack_matches_oracle_random(N, K, seed, outl):
    w, _ = synthetic.weights(N, K, seed, outl)
    _pack_equal(w)


def test_pack_matches_oracle_full_size_row_sample():
    N, K, outl = synthetic.SHAPES["fused"]
    w, _ = synthetic.weights(N, K, 0, outl)
    rows = np.random.default_rng(9).choice(N, 512, replace=False)
    _pack_equal(np.ascontiguousarray(w[rows]))


def test_pack_degenerate_and_tie_groups():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((8, 256)).astype(np.float32) * 0.02
    w[0, :128] = 0.0                           # all zero
    w[1, :128] = -0.0                          # negative zeros
    w[2, :128] = np.float32(1e-6)              # constant, tiny
    w[3, :128] = np.float32(3e-8)              # subnormal-fp16 minimum
    w[4, :64] = np.float32(1e-7); w[4, 64:128] = np.float32(2e-7)   # scale underflows fp16
    w[5, :128] = np.linspace(0, 15 / 16, 128).astype(np.float32)
    w[5, 5] = np.float32(2.5 / 16); w[5, 6] = np.float32(3.5 / 16)   # exact ties
    w[6, :128] = np.float32(60000.0); w[6, 0] = np.float32(-60000.0)  # large but representable scale
    _pack_equal(w)


def test_known_answer_groups_through_library():
    import json, os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "known_answers.json")))
    for g in fx["groups"]:
        c, s, m = q4.pack_host(np.array([g["w"]], np.float32))
        assert int(s[0, 0]) == g["scale_bits"] and int(m[0, 0]) == g["min_bits"], g["name"]
        assert oracle.unpack(c)[0].tolist() == g["codes"], g["name"]


def test_pack_rejects_bad_input():
    L = _lib.lib
    w = np.zeros((2, 256), np.float32)
    c = np.zeros((2, 128), np.uint8); s = np.zeros((2, 2), np.uint16); m = np.zeros((2, 2), np.uint16)
    args = lambda ww, N, K: (ww.ctypes.data, N, K, c.ctypes.data, s.ctypes.data, m.ctypes.data, 1)
    assert L.q4_pack_host(*args(w, 2, 256)) == _lib.Q4_OK
    assert L.q4_pack_host(*args(w, 2, 200)) == _lib.Q4_ERR_UNSUPPORTED_SHAPE
    assert L.q4_pack_host(*args(w, 0, 256)) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_pack_host(None, 2, 256, c.ctypes.data, s.ctypes.data, m.ctypes.data, 1) == _lib.Q4_ERR_INVALID_ARG
    bad = w.copy(); bad[1, 7] = np.nan
    assert L.q4_pack_host(*args(bad, 2, 256)) == _lib.Q4_ERR_INVALID_ARG
    big = w.copy(); big[0, 0] = 1e6; big[0, 1] = -1e6          # (max-min)/15 overflows fp16
    assert L.q4_pack_host(*args(big, 2, 256)) == _lib.Q4_ERR_INVALID_ARG
    with pytest.raises(q4.Q4Error):
        q4.pack_host(bad)


def test_host_validation_before_any_cuda_call():
    """Invalid arguments are rejected on the host before the library touches CUDA."""
    L = _lib.lib
    m = _lib.q4_matrix(16, 16, 16, 10, 200)   # K not a multiple of 128
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_UNSUPPORTED_SHAPE
    m = _lib.q4_matrix(16, 16, 16, 0, 256)
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_INVALID_ARG
    m = _lib.q4_matrix(None, 16, 16, 10, 256)
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_INVALID_ARG
    m = _lib.q4_matrix(17, 16, 16, 10, 256)   # codes not 16-byte aligned
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_MISALIGNED
    m = _lib.q4_matrix(16, 16, 16, 10, 256)
    assert L.q4_gemm_skinny(ctypes.byref(m), 16, 9, 16, None, 0, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_gemm_skinny(ctypes.byref(m), 16, 0, 16, None, 0, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_gemm_skinny(ctypes.byref(m), 8, 1, 16, None, 0, None) == _lib.Q4_ERR_MISALIGNED
    assert L.q4_gemm_skinny(ctypes.byref(m), 16, 1, 18, None, 0, None) == _lib.Q4_ERR_MISALIGNED
    assert L.q4_gemm_skinny(ctypes.byref(m), None, 1, 16, None, 0, None) == _lib.Q4_ERR_INVALID_ARG
    m = _lib.q4_matrix(16, 16, 16, 10, 65536 + 128)
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_UNSUPPORTED_SHAPE
    m = _lib.q4_matrix(16, 16, 16, 1 << 31, 256)
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_UNSUPPORTED_SHAPE
    assert L.q4_decode_step(None, 1, None, None, 1, None, 0, 1, None) == _lib.Q4_ERR_INVALID_ARG
    arr = (_lib.q4_matrix * 1)(_lib.q4_matrix(16, 16, 16, 10, 256))
    assert L.q4_decode_step(arr, 0, None, None, 1, None, 0, 1, None) == _lib.Q4_ERR_INVALID_ARG
    xp = (_lib.c_vp * 1)(16)
    yp = (_lib.c_vp * 1)(16)
    assert L.q4_decode_step(arr, 1, xp, yp, 9, None, 0, 0, None) == _lib.Q4_ERR_INVALID_ARG
    bad = (_lib.q4_matrix * 1)(_lib.q4_matrix(16, 16, 16, 10, 200))
    assert L.q4_decode_step(bad, 1, xp, yp, 1, None, 0, 1, None) == _lib.Q4_ERR_UNSUPPORTED_SHAPE
    assert L.q4_argmax_f32(16, 9, 10, 16, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_argmax_f32(16, 1, 0, 16, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_argmax_f32(None, 1, 10, 16, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_workspace_bytes(10, 200, 1) == 0
    assert L.q4_tiled_bytes(10, 200) == 0
    Ks = (_lib.c_i64 * 2)(3072, 200)
    assert L.q4_step_workspace_bytes(Ks, 2, 1) == 0
    assert L.q4_step_workspace_bytes(Ks, 1, 1) == (24 * (256 + 32) + 32 + 255) // 256 * 256
    assert L.q4_step_workspace_bytes(Ks, 1, 9) == 0
    assert L.q4_step_prepare(None, 1, None, 1, 16, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    nt = (_lib.q4_matrix * 1)(_lib.q4_matrix(16, 16, 16, 10, 256))          # no tiled copy
    assert L.q4_step_stream(nt, 1, None, 1, 16, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    tt = (_lib.q4_matrix * 1)(_lib.q4_matrix(None, None, None, 10, 256, 16))
    assert L.q4_step_stream(tt, 1, None, 1, 16, 8, None) == _lib.Q4_ERR_WORKSPACE
    assert L.q4_step_stream(tt, 1, None, 1, 8, 1 << 20, None) == _lib.Q4_ERR_MISALIGNED
    assert L.q4_tiled_bytes(17, 384) == 2 * 3 * 1088
    assert L.q4_tile(None, 16, 1 << 20, None) == _lib.Q4_ERR_INVALID_ARG
    m = _lib.q4_matrix(16, 16, 16, 17, 384)
    assert L.q4_tile(ctypes.byref(m), 16, 100, None) == _lib.Q4_ERR_WORKSPACE
    assert L.q4_tile(ctypes.byref(m), 8, 1 << 20, None) == _lib.Q4_ERR_MISALIGNED
    m = _lib.q4_matrix(None, None, None, 17, 384, 16)      # tiled copy only: accepted by the checks
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) != _lib.Q4_ERR_INVALID_ARG
    m = _lib.q4_matrix(None, None, None, 17, 384, 8)       # misaligned tiled copy
    assert L.q4_gemv(ctypes.byref(m), 16, 16, None, 0, None) == _lib.Q4_ERR_MISALIGNED
    info = _lib.q4_plan_info()
    assert L.q4_plan(10, 200, ctypes.byref(info)) == _lib.Q4_ERR_UNSUPPORTED_SHAPE


def test_binding_refuses_host_tensors_before_any_library_call():
    """Every wrapper hands device addresses to kernels; a host tensor would fault the GPU, so the
    binding refuses it (no GPU needed: the check runs before the library is called)."""
    import torch
    import int4_weight_only_q4_gb300 as q4
    w, x = synthetic.random_shape_problem(32, 256, 2, seed=3)
    W = q4.QuantizedMatrix.from_packed(*q4.pack_host(w), device="cpu", tiled=False)
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    Y = torch.empty((2, 32), dtype=torch.float32)
    with pytest.raises(TypeError, match="CUDA tensor"):
        q4.gemm_skinny(W, X, Y, workspace=q4.Workspace(0, "cpu"))
    with pytest.raises(TypeError, match="CUDA tensor"):
        q4.argmax(Y)
    Qb = torch.zeros((1, 8, 64), dtype=torch.bfloat16)
    Kb = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="CUDA tensor"):
        q4.flash_decode(Qb, Kb, Kb, torch.zeros(1, dtype=torch.int32), n_chunks=4,
                        workspace=q4.Workspace(1 << 16, "cpu"))
    with pytest.raises(TypeError, match="CUDA tensor"):
        q4.sample_topk(Y, 4, 1.0, torch.zeros((2, 4)))


def test_binding_refuses_mis_sized_outputs_and_activations():
    """A short or mistyped output buffer would be written past its end by the kernels: the binding
    refuses it, and activations whose width is not the matrix's K, before any library call."""
    import torch
    import int4_weight_only_q4_gb300 as q4
    w, x = synthetic.random_shape_problem(32, 256, 2, seed=3)
    W = q4.QuantizedMatrix.from_packed(*q4.pack_host(w), device="cpu", tiled=False)
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    ws = q4.Workspace(0, "cpu")
    for fn in (lambda Y: q4.gemm_skinny(W, X, Y, workspace=ws), lambda Y: q4.gemm_skinny_noalloc(W, X, Y)):
        with pytest.raises(ValueError, match="smaller than"):
            fn(torch.empty((2, 31), dtype=torch.float32))
        with pytest.raises(TypeError, match="float32"):
            fn(torch.empty((2, 32), dtype=torch.float16))
        with pytest.raises(TypeError, match="contiguous"):
            fn(torch.empty((32, 2), dtype=torch.float32).t())
    with pytest.raises(ValueError, match="K = 256"):
        q4.gemm_skinny(W, X[:, :128].contiguous(), torch.empty((2, 32)), workspace=ws)
    with pytest.raises(ValueError, match="smaller than"):
        q4.gemv(W, X[0], torch.empty((31,), dtype=torch.float32), workspace=ws)
    with pytest.raises(ValueError, match="smaller than"):
        q4.decode_step([W, W], [X, X], [torch.empty((2, 32)), torch.empty((1, 32))], workspace=ws)
    with pytest.raises(ValueError, match="same batch size"):
        q4.decode_step([W, W], [X, X[:1].contiguous()], [torch.empty((2, 32))] * 2, workspace=ws)
    with pytest.raises(ValueError, match="int32"):
        q4.argmax(torch.empty((2, 32)), torch.empty((2,), dtype=torch.int64))


def test_noalloc_host_checks_and_injected_launch_failure(monkeypatch):
    """q4_gemm_skinny_noalloc validates on the host like the other entry points, refuses sizes beyond
    its scratch, and reports an injected launch failure without touching CUDA."""
    L = _lib.lib
    m = _lib.q4_matrix(16, 16, 16, 10, 256)                     # no tiled copy
    assert L.q4_gemm_skinny_noalloc(ctypes.byref(m), 16, 1, 16, None) == _lib.Q4_ERR_INVALID_ARG
    m = _lib.q4_matrix(None, None, None, 10, 256, 16)
    assert L.q4_gemm_skinny_noalloc(ctypes.byref(m), 16, 9, 16, None) == _lib.Q4_ERR_INVALID_ARG
    assert L.q4_gemm_skinny_noalloc(ctypes.byref(m), 8, 1, 16, None) == _lib.Q4_ERR_MISALIGNED
    big = _lib.q4_matrix(None, None, None, 10, 32384, 16)
    assert L.q4_gemm_skinny_noalloc(ctypes.byref(big), 16, 8, 16, None) == _lib.Q4_ERR_WORKSPACE
    monkeypatch.setenv("Q4_FAULT_INJECT", "launch")
    assert L.q4_gemm_skinny_noalloc(ctypes.byref(m), 16, 1, 16, None) == _lib.Q4_ERR_CUDA
