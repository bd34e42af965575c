"""q4_gemm_skinny_noalloc: the skinny GEMM for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: code running while a CUDA graph is
being captured (cudaMalloc is not allowed there), real-time threads that must never wait on the
allocator, and hosts whose device memory is budgeted by someone else.  This entry point keeps its
scratch in a fixed array inside the library instead.  The test calls it through the C ABI twice
in a row, with different activations each time (the array keeps the first call's contents), and
compares each result with q4_gemm_skinny, the entry point that takes a workspace.  This file is
collected last, so a run that stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the tolerance of the parity tests


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as q4
    from int4_weight_only_q4_gb300 import _lib
    N, K, B = 3000, 3072, 4
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=41, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    m = W.c_struct()
    for call, seed in enumerate((101, 202)):
        x = synthetic.activations(B, K, np.random.default_rng(seed))
        X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        Y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        st = _lib.lib.q4_gemm_skinny_noalloc(ctypes.byref(m), X.data_ptr(), B, Y.data_ptr(), stream)
        assert st == _lib.Q4_OK, (call, _lib.STATUS[st])
        Y_ws = q4.gemm_skinny(W, X)  # the entry point that takes a workspace
        torch.cuda.synchronize()
        assert oracle.rel_err(Y.cpu().numpy(), Y_ws.cpu().numpy()) <= TOL, call
    q4.device_status()


def test_noalloc_rejects_requests_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as q4
    from int4_weight_only_q4_gb300 import _lib
    assert _lib.lib.q4_noalloc_scratch_bytes() == 512 * 1024
    N, K = 16, 32768 + 128           # 8 columns need (K/128) * 2080 + 32 bytes > 512 KiB
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=5)
    W = q4.QuantizedMatrix.from_float(w)
    m = W.c_struct()
    X = torch.zeros((8, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((8, N), dtype=torch.float32, device="cuda")
    st = _lib.lib.q4_gemm_skinny_noalloc(ctypes.byref(m), X.data_ptr(), 8, Y.data_ptr(), None)
    assert st == _lib.Q4_ERR_WORKSPACE
    X1 = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")   # one column fits
    Y1 = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    assert _lib.lib.q4_gemm_skinny_noalloc(ctypes.byref(m), X1.data_ptr(), 1, Y1.data_ptr(), None) == _lib.Q4_OK
    torch.cuda.synchronize()
