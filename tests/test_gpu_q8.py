"""GPU parity of the int8 output head (q8_head) against the fp64 CPU oracle (oracle/q8_oracle.py).

The head is the one matrix the rumik-oss-1 write-up keeps in int8 ("Steps 9-10: streaming to the
speaker"); its argmax is the greedy pick of the next token.  Logits: max relative error <= 2e-3
per output (floor 1% of the output RMS), as for the int4 path.  Tiled layout and argmax: exact.
Each batch column is compared bit for bit with the same call at B = 1.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import oracle.q8_oracle as Q8
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


def tiled_reference(codes, N, K):
    """The documented layout, written with numpy (q4.h, q8_tiled_bytes)."""
    T, G = (N + 15) // 16, K // 128
    pad = np.zeros((T * 16, K), np.int8)
    pad[:N] = codes
    out = np.zeros((T, G, 2, 32, 32), np.int8)
    for j in range(T):
        for g in range(G):
            for h in range(2):
                for l in range(32):
                    row = 16 * j + l // 4 + 8 * h
                    k0 = 128 * g + 32 * (l % 4)
                    out[j, g, h, l] = pad[row, k0:k0 + 32]
    return out.reshape(-1).view(np.uint8)


def check_head(q4, w, x, label, rows_sample=None):
    codes, sb = q4.pack_int8_host(w)
    H = q4.Int8Head.from_packed(codes, sb)
    X = bf16_tensor(x)
    Y, idx = H(X)
    torch.cuda.synchronize()
    y = Y.cpu().numpy()
    # the GPU's own argmax of its own logits is exact
    assert idx.cpu().numpy().tolist() == np.argmax(y, axis=1).tolist(), label
    rows = np.arange(w.shape[0]) if rows_sample is None else rows_sample
    y_ref = Q8.matvec(codes, sb, x, rows=rows)
    e = oracle.rel_err(y[:, rows], y_ref)
    _log(label, e)
    assert e <= TOL, (label, e)
    return H, X, y


def _log(label, e):
    import json, os
    log = os.environ.get("Q4_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": label, "rel_err": e}) + "\n")


def test_tiled_copy_matches_documented_layout(q4):
    for N, K in ((1, 128), (37, 384), (300, 1024)):
        w, _ = synthetic.random_shape_problem(N, K, 1, seed=N)
        codes, sb = q4.pack_int8_host(w)
        H = q4.Int8Head.from_packed(codes, sb)
        torch.cuda.synchronize()
        assert np.array_equal(H.tiled.cpu().numpy(), tiled_reference(codes, N, K)), (N, K)


@pytest.mark.parametrize("N,K", [(1, 128), (17, 256), (100, 1152), (1000, 640), (4099, 1024), (257, 8192),
                                 (40, 16384)])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_logits_and_argmax_odd_shapes(q4, N, K, B):
    w, x = synthetic.random_shape_problem(N, K, B, seed=7 + B, outliers=True)
    H, X, y = check_head(q4, w, x, f"q8 N={N} K={K} B={B}")
    # batch invariance: column 1 (or 0) alone gives the same bits
    b = min(1, B - 1)
    y1, i1 = H(X[b:b + 1].contiguous())
    torch.cuda.synchronize()
    assert np.array_equal(y1.cpu().numpy()[0], y[b])
    assert i1.item() == int(np.argmax(y[b]))


def test_logits_only_and_argmax_only_agree(q4):
    w, x = synthetic.random_shape_problem(5000, 3072, 4, seed=11, outliers=True)
    codes, sb = q4.pack_int8_host(w)
    H = q4.Int8Head.from_packed(codes, sb)
    X = bf16_tensor(x)
    ws = H.workspace(4)
    Y, idx = H(X, workspace=ws)
    Y2, none_idx = H(X, argmax=False, workspace=ws)
    none_y, idx2 = H(X, logits=False, workspace=ws)
    torch.cuda.synchronize()
    assert none_idx is None and none_y is None
    assert torch.equal(Y, Y2) and torch.equal(idx, idx2)
    # repeated calls with one workspace: same bits (nothing carries over between calls)
    Y3, idx3 = H(X, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y3) and torch.equal(idx, idx3)


def test_argmax_ties_go_to_lowest_row(q4):
    w, x = synthetic.random_shape_problem(3000, 1024, 2, seed=12)
    codes, sb = q4.pack_int8_host(w)
    # make rows 2999, 1500 and 40 identical and dominant: every batch row must pick 40
    big = np.full(1024, 127, np.int8)
    xs = x.view(np.uint16)
    sign = np.where((xs[0] >> 15) & 1, -1, 1).astype(np.int8)
    for r in (2999, 1500, 40):
        codes[r] = big * sign
        sb[r] = sb.max()
    H = q4.Int8Head.from_packed(codes, sb)
    Y, idx = H(bf16_tensor(x[:1]))
    torch.cuda.synchronize()
    y = Y.cpu().numpy()[0]
    # the fused argmax follows the rule on the GPU's own logits (identical rows in different
    # tiles may be summed in different orders, so their logits need not be bit-equal)
    assert idx.item() == int(np.argmax(y)) and idx.item() in (40, 1500, 2999)
    if y[40] == y[1500] == y[2999]:
        assert idx.item() == 40


def test_full_size_head(q4):
    """The 65,536 x 3072 head, B = 1 and 8: sampled logits against the oracle, argmax against the
    oracle's argmax over all rows (either index accepted only inside the GPU's measured error)."""
    w, x8 = synthetic.problem("head", 8, seed=0)
    codes, sb = q4.pack_int8_host(w)
    H = q4.Int8Head.from_packed(codes, sb)
    y_ref, ref_idx = Q8.head_argmax(codes, sb, x8)
    for B in (1, 8):
        x = x8[:B]
        Y, idx = H(bf16_tensor(x))
        torch.cuda.synchronize()
        y = Y.cpu().numpy()
        e = oracle.rel_err(y, y_ref[:B])
        _log(f"q8 full head 65536x3072 B={B}", e)
        assert e <= TOL
        bound = 2.0 * float(np.abs(y - y_ref[:B]).max())
        for b in range(B):
            if oracle.argmax_ambiguous(y_ref[b], bound):
                assert y_ref[b, idx[b].item()] >= y_ref[b].max() - bound
            else:
                assert idx[b].item() == ref_idx[b]
