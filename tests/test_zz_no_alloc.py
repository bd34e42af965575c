"""q4_gemm_skinny_noalloc: the skinny GEMM for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: code running while a CUDA graph is
being captured (cudaMalloc is not allowed there), real-time threads that must never wait on the
allocator, and hosts whose device memory is budgeted by someone else.  This entry point keeps its
scratch in a fixed array inside the library instead.  The tests call it through the C ABI twice in
a row, with different activations each time (the array keeps the first call's contents), and
check each result three ways: bit for bit against the tile kernel run with a caller-owned
workspace (q4_step_prepare + q4_step_stream on the same one-matrix list, which the header says it
computes exactly), against q4_gemm_skinny, and against the fp64 oracle, both within the parity
tolerance.  The size limit is checked at its exact boundaries.  This file is collected last, so a
run that stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the tolerance of the parity tests


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as m
    return m


def _bf16(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc(W, X, B, N):
    """One call through the C ABI into a NaN-filled output; returns the output."""
    from int4_weight_only_q4_gb300 import _lib
    m = W.c_struct()
    Y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = _lib.lib.q4_gemm_skinny_noalloc(ctypes.byref(m), X.data_ptr(), B, Y.data_ptr(), stream)
    assert st == _lib.Q4_OK, _lib.STATUS[st]
    return Y


def _tile_kernel_with_workspace(q4, W, X, B):
    ws = q4.Workspace(q4.step_workspace_bytes([W.K], B))
    Y = torch.empty((B, W.N), dtype=torch.float32, device="cuda")
    q4.step_prepare([W], [X], ws)
    q4.step_stream([W], [Y], B, ws)
    return Y


def _oracle(w, x_bits):
    return oracle.gemv_packed(*oracle.quantise_pack(w), x_bits)


def test_noalloc_matches_workspace_entry_points_on_two_calls(q4):
    N, K, B = 3000, 3072, 4
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=41, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    for call, seed in enumerate((101, 202)):
        x = synthetic.activations(B, K, np.random.default_rng(seed))
        X = _bf16(x)
        Y = _noalloc(W, X, B, N)
        Y_tile = _tile_kernel_with_workspace(q4, W, X, B)
        Y_ws = q4.gemm_skinny(W, X)  # the single-call entry point (another kernel for this shape)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y_tile), call
        y = Y.cpu().numpy()
        assert oracle.rel_err(y, Y_ws.cpu().numpy()) <= TOL, call
        assert oracle.rel_err(y, _oracle(w, x)) <= TOL, call
    q4.device_status()


@pytest.mark.parametrize("K,B", [(32256, 8), (63488, 4), (65536, 2)])
def test_noalloc_accepts_the_largest_sizes_it_documents(q4, K, B):
    """The largest K of each batch tile fits in the scratch: the results match the oracle and the
    tile kernel with a workspace, on two calls in a row."""
    N = 40
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=K + B, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    for seed in (1, 2):
        x = synthetic.activations(B, K, np.random.default_rng(seed + K))
        X = _bf16(x)
        Y = _noalloc(W, X, B, N)
        Y_tile = _tile_kernel_with_workspace(q4, W, X, B)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y_tile), (K, B, seed)
        assert oracle.rel_err(Y.cpu().numpy(), _oracle(w, x)) <= TOL, (K, B, seed)
    q4.device_status()


@pytest.mark.parametrize("K,B", [(32384, 8), (32384, 5), (63616, 4), (63616, 3)])
def test_noalloc_rejects_requests_beyond_its_scratch(q4, K, B):
    from int4_weight_only_q4_gb300 import _lib
    assert _lib.lib.q4_noalloc_scratch_bytes() == 512 * 1024
    N = 16
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=5)
    W = q4.QuantizedMatrix.from_float(w)
    m = W.c_struct()
    X = torch.zeros((B, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((B, N), 7.0, dtype=torch.float32, device="cuda")
    st = _lib.lib.q4_gemm_skinny_noalloc(ctypes.byref(m), X.data_ptr(), B, Y.data_ptr(), None)
    assert st == _lib.Q4_ERR_WORKSPACE
    with pytest.raises(q4.Q4Error):
        q4.gemm_skinny_noalloc(W, X, Y)
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())        # nothing was launched


def test_noalloc_reports_an_injected_launch_failure(q4, monkeypatch):
    """Host-side fault injection covers this entry point too: the call reports Q4_ERR_CUDA, launches
    nothing, and the next call works."""
    from int4_weight_only_q4_gb300 import _lib
    N, K, B = 64, 1024, 2
    w, x = synthetic.random_shape_problem(N, K, B, seed=17)
    W = q4.QuantizedMatrix.from_float(w)
    m = W.c_struct()
    X = _bf16(x)
    Y = torch.full((B, N), 7.0, dtype=torch.float32, device="cuda")
    monkeypatch.setenv("Q4_FAULT_INJECT", "launch")
    assert _lib.lib.q4_gemm_skinny_noalloc(ctypes.byref(m), X.data_ptr(), B, Y.data_ptr(), None) == \
        _lib.Q4_ERR_CUDA
    monkeypatch.delenv("Q4_FAULT_INJECT")
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())
    Y = _noalloc(W, X, B, N)
    torch.cuda.synchronize()
    assert oracle.rel_err(Y.cpu().numpy(), _oracle(w, x)) <= TOL
    q4.device_status()
