"""GPU parity of the int4 prefill GEMM (q4_gemm_prefill) against the fp64 CPU oracle.

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


@pytest.mark.parametrize("N,K", [(16, 128), (100, 1152), (1000, 640), (3072, 3072), (257, 8192)])
@pytest.mark.parametrize("M", [1, 7, 8, 9, 64, 100, 130])
def test_prefill_matches_oracle(q4, N, K, M):
    w, x = synthetic.random_shape_problem(N, K, M, seed=N + M, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    Y = q4.gemm_prefill(W, bf16_tensor(x))
    torch.cuda.synchronize()
    rows = np.arange(N) if N <= 1000 else np.random.default_rng(0).choice(N, 400, replace=False)
    e = oracle.rel_err(Y.cpu().numpy()[:, rows], oracle_y(w, x, rows))
    assert e <= TOL, e


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
