"""GPU parity of the int4 prefill GEMM (q4_gemm_prefill) against the fp64 CPU oracle.

Two kernels serve the call: the tensor-memory kernel (tcgen05.mma, TMEM accumulators, TMA) on
compute capability 10.x, and the mma.sync kernel elsewhere or when Q4_PREFILL_TC=0; both are
checked.

The rumik-oss-1 write-up's "Step 8: a prefill that stays int4": the prompt's M tokens multiply
the int4 weights directly (no dequantised copy), on the tensor cores, with each group's scale and
minimum folded into the fp32 result.  The oracle is the
same dequantise-then-matmul (gemv_packed takes any number of activation rows).  Tolerance as for
the GEMV: max relative error <= 2e-3 per output (floor 1% of the output RMS).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as m
    return m


def bf16_tensor(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).cuda()


def oracle_y(w, x, rows):
    p, sb, mb = oracle.quantise_pack(np.ascontiguousarray(w[rows]))
    return oracle.gemv_packed(p, sb, mb, x)


@pytest.mark.parametrize("path", ["tc", "mma"])
@pytest.mark.parametrize("N,K", [(16, 128), (100, 1152), (1000, 640), (3072, 3072), (257, 8192), (64, 8320),
                                 (40, 16384)])
@pytest.mark.parametrize("M", [1, 7, 8, 9, 64, 100, 130, 300])
def test_prefill_matches_oracle(q4, monkeypatch, path, N, K, M):
    if path == "mma":
        monkeypatch.setenv("Q4_PREFILL_TC", "0")
    w, x = synthetic.random_shape_problem(N, K, M, seed=N + M, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    Y = q4.gemm_prefill(W, bf16_tensor(x))
    torch.cuda.synchronize()
    rows = np.arange(N) if N <= 1000 else np.random.default_rng(0).choice(N, 400, replace=False)
    e = oracle.rel_err(Y.cpu().numpy()[:, rows], oracle_y(w, x, rows))
    assert e <= TOL, (path, e)
    q4.device_status()  # no bounded wait gave up


def test_prefill_kernel_choice(q4, monkeypatch):
    """On a compute capability 10.x device the tcgen05 kernel serves every shape; the
    Q4_PREFILL_TC=0 switch selects the mma.sync kernel."""
    if torch.cuda.get_device_capability()[0] == 10:
        for K, M in ((3072, 512), (8192, 1), (65536, 3), (128, 1 << 24)):
            assert q4.prefill_kernel(K, M) == "tcgen05", (K, M)
    with pytest.raises(ValueError):
        q4.prefill_kernel(100, 1)
    monkeypatch.setenv("Q4_PREFILL_TC", "0")
    assert q4.prefill_kernel(3072, 512) == "mma.sync"


def test_prefill_kernels_agree_and_leave_rows_alone(q4, monkeypatch):
    """Both kernels agree to fp32 rounding on a ragged shape (rows and tokens not multiples of the
    128 x 128 tile), and neither writes outside Y (a guard band around it keeps its canaries)."""
    N, K, M = 1000, 3072, 259
    w, x = synthetic.random_shape_problem(N, K, M, seed=91, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    outs = []
    for env in ("1", "0"):
        monkeypatch.setenv("Q4_PREFILL_TC", env)
        buf = torch.full((M * N + 2048,), 7.0, device="cuda")
        Y = buf[1024:1024 + M * N].view(M, N)
        q4.gemm_prefill(W, X, Y)
        torch.cuda.synchronize()
        assert bool((buf[:1024] == 7.0).all()) and bool((buf[1024 + M * N:] == 7.0).all()), env
        outs.append(Y.clone())
    assert torch.allclose(outs[0], outs[1], rtol=1e-4, atol=1e-5)
    q4.device_status()


def test_prefill_long_prompt_full_size(q4):
    """The fused 25,088 x 3072 projection over a 512-token prompt: sampled rows against the oracle,
    and each token's row equal to the single-token GEMV within fp32 rounding."""
    w, x = synthetic.random_shape_problem(25088, 3072, 512, seed=3, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    Y = q4.gemm_prefill(W, X)
    y5 = q4.gemm_skinny(W, X[5:6].contiguous())
    torch.cuda.synchronize()
    rows = np.random.default_rng(1).choice(25088, 256, replace=False)
    toks = np.random.default_rng(2).choice(512, 24, replace=False)
    e = oracle.rel_err(Y.cpu().numpy()[np.ix_(toks, rows)], oracle_y(w, x[toks], rows))
    assert e <= TOL, e
    assert torch.allclose(Y[5], y5[0], rtol=1e-4, atol=1e-5)


def test_prefill_repeatable_and_workspace_checked(q4):
    import ctypes
    from int4_weight_only_q4_gb300 import _lib
    w, x = synthetic.random_shape_problem(640, 1024, 40, seed=8)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    a = q4.gemm_prefill(W, X)
    b = q4.gemm_prefill(W, X)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    m = W.c_struct()
    need = _lib.lib.q4_prefill_workspace_bytes(1024, 40)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    Y = torch.empty((40, 640), device="cuda")
    assert _lib.lib.q4_gemm_prefill(ctypes.byref(m), X.data_ptr(), 40, Y.data_ptr(), ws.data_ptr(), need - 16,
                                    None) == _lib.Q4_ERR_WORKSPACE
    assert _lib.lib.q4_gemm_prefill(ctypes.byref(m), X.data_ptr(), 0, Y.data_ptr(), ws.data_ptr(), need,
                                    None) == _lib.Q4_ERR_INVALID_ARG
