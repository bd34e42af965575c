"""GPU parity of libq4.so against the fp64 CPU oracle.

Tolerance: the stated bound, max relative error <= 2e-3 per output with a floor
of 1% of the output RMS for outputs near zero (fp32 accumulation on the GPU,
fp64 on the oracle).  Packing and argmax are compared exactly; each batch
column of the skinny GEMM is compared bit for bit with the batch-1 GEMV (the
pure-C TTS engine page, wpnews.pro: batched output must equal single-stream
output).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 2e-3


def within_tol(name, y, y_ref):
    """rel_err <= TOL; every measured error is appended to $Q4_PARITY_LOG (if set) for the record."""
    import json, os
    e = oracle.rel_err(y, y_ref)
    log = os.environ.get("Q4_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": name, "rel_err": e}) + "\n")
    return e <= TOL


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as m
    return m


def bf16_tensor(x_bits: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).cuda()


def oracle_rows(w, x_bits, rows=None, chunk=8192):
    """Oracle output for the given rows (quantising only those rows, a chunk at a time)."""
    idx = np.arange(w.shape[0]) if rows is None else np.asarray(rows)
    out = []
    for s in range(0, idx.size, chunk):
        p, sb, mb = oracle.quantise_pack(np.ascontiguousarray(w[idx[s:s + chunk]]))
        out.append(oracle.gemv_packed(p, sb, mb, x_bits))
    return np.concatenate(out, axis=1)


def run(q4, W, x_bits, ws=None):
    X = bf16_tensor(x_bits)
    Y = q4.gemm_skinny(W, X, workspace=ws)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


# ----------------------------------------------------------------------------- small configs
def test_tiny_config_b1(q4):
    w, x = synthetic.problem("tiny", 1, seed=0)
    W = q4.QuantizedMatrix.from_float(w)
    y = run(q4, W, x)
    assert within_tol("tiny B=1", y, oracle_rows(w, x))


@pytest.mark.parametrize("N,K", [(1, 128), (7, 128), (16, 256), (17, 384), (33, 512), (100, 1152),
                                 (1000, 640), (4099, 1024), (257, 8192), (40, 16384)])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_odd_shapes(q4, N, K, B):
    w, x = synthetic.random_shape_problem(N, K, B, seed=N * 7 + K + B, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    y = run(q4, W, x)
    assert within_tol(f"odd N={N} K={K} B={B}", y, oracle_rows(w, x))


def test_gemv_entry_point_equals_skinny_b1(q4):
    w, x = synthetic.random_shape_problem(300, 1024, 1, seed=3)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    y1 = q4.gemv(W, X[0])
    y2 = q4.gemm_skinny(W, X)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2[0])


def test_known_answer_gemv_through_gpu(q4):
    import json, os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "known_answers.json")))
    groups = {g["name"]: g for g in fx["groups"]}
    for case in fx["gemv"]:
        w = np.array([groups[r]["w"] for r in case["rows"]], np.float32)
        K = w.shape[1]
        xf = np.ones(K, np.float32) if case["x"] == "ones" else \
            np.array([1.0 if k % 2 == 0 else -1.0 for k in range(K)], np.float32)
        W = q4.QuantizedMatrix.from_float(w)
        y = run(q4, W, synthetic.f32_to_bf16_bits(xf)[None, :])[0]
        assert np.allclose(y, case["y"], rtol=1e-6, atol=1e-6), case["name"]


def test_closed_forms_on_gpu(q4):
    """All-zero codes leave sum_g min_g * S_g; a one-hot x picks one dequantised column."""
    N, K = 64, 512
    w, x = synthetic.random_shape_problem(N, K, 2, seed=8)
    c, s, m = q4.pack_host(w)
    Wz = q4.QuantizedMatrix.from_packed(np.zeros_like(c), s, m)
    y = run(q4, Wz, x)
    S = oracle.bf16_bits_to_f64(x).reshape(2, K // 128, 128).sum(2)
    assert oracle.rel_err(y, S @ oracle.f16_bits_to_f64(m).T) <= TOL
    W = q4.QuantizedMatrix.from_packed(c, s, m)
    w_hat = oracle.dequantise(oracle.unpack(c), s, m)
    for k in (0, 1, 2, 5, 127, 128, 300, 511):
        xh = np.zeros((1, K), np.uint16)
        xh[0, k] = 0x3F80
        yk = run(q4, W, xh)[0]
        assert np.allclose(yk, w_hat[:, k], rtol=1e-6, atol=1e-7), k


def tiled_reference(codes, scales, mins, N, K):
    """The tiled copy's documented record layout, built with numpy from the canonical arrays."""
    G = K // 128
    T = (N + 15) // 16
    c = np.zeros((T * 16, K // 2), np.uint8)
    c[:N] = codes
    sm = np.zeros((T * 16, G), np.uint32)
    sm[:N] = scales.astype(np.uint32) | (mins.astype(np.uint32) << 16)
    out = np.zeros((T, G, 1088), np.uint8)
    for h in range(2):
        for l in range(32):
            rows = np.arange(T) * 16 + l // 4 + 8 * h
            for g in range(G):
                out[:, g, 512 * h + 16 * l: 512 * h + 16 * l + 16] = c[rows, g * 64 + 16 * (l % 4): g * 64 + 16 * (l % 4) + 16]
    words = np.zeros((T, G, 16), np.uint32)
    for q in range(8):
        words[:, :, 2 * q] = sm[np.arange(T) * 16 + q][:, :]
        words[:, :, 2 * q + 1] = sm[np.arange(T) * 16 + q + 8][:, :]
    out[:, :, 1024:] = words.view(np.uint8).reshape(T, G, 64)
    return out.reshape(-1)


@pytest.mark.parametrize("N,K", [(1, 128), (37, 384), (300, 1024)])
def test_tiled_copy_matches_documented_layout(q4, N, K):
    w, _ = synthetic.random_shape_problem(N, K, 1, seed=N + K, outliers=True)
    c, s, m = q4.pack_host(w)
    W = q4.QuantizedMatrix.from_packed(c, s, m)
    torch.cuda.synchronize()
    assert W.tiled.numel() == q4.tiled_bytes(N, K) == ((N + 15) // 16) * (K // 128) * 1088
    assert np.array_equal(W.tiled.cpu().numpy(), tiled_reference(c, s, m, N, K))


def test_tiled_only_matrix(q4, monkeypatch):
    """A matrix that keeps only its tiled copy gives the same result; an L0 kernel choice falls back
    to a kernel that reads the tiled copy (another kernel family: its own, fixed, addition order)."""
    w, x = synthetic.random_shape_problem(1000, 1152, 3, seed=12, outliers=True)
    c, s, m = q4.pack_host(w)
    Wb = q4.QuantizedMatrix.from_packed(c, s, m)
    Wt = q4.QuantizedMatrix.from_packed(c, s, m, keep_canonical=False)
    assert Wt.codes is None and Wt.tiled is not None
    X = bf16_tensor(x)
    y1 = q4.gemm_skinny(Wb, X)
    y2 = q4.gemm_skinny(Wt, X)
    monkeypatch.setenv("Q4_KERNEL", "1")
    y3 = q4.gemm_skinny(Wt, X)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert within_tol("tiled-only fallback", y3.cpu().numpy(), oracle_rows(w, x))


# ----------------------------------------------------------------------------- batch invariance
@pytest.mark.parametrize("N,K", [(256, 512), (3072, 3072), (1000, 8192), (4099, 1024)])
def test_batch_columns_bit_identical_to_b1(q4, N, K):
    w, x = synthetic.random_shape_problem(N, K, 8, seed=N + K, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    singles = [q4.gemm_skinny(W, X[b:b + 1].contiguous()) for b in range(8)]
    for B in (2, 4, 8, 5):
        Y = q4.gemm_skinny(W, X[:B].contiguous())
        for b in range(B):
            assert torch.equal(Y[b], singles[b][0]), (B, b)
    perm = torch.tensor([5, 2, 7, 0, 1, 6, 3, 4], device="cuda")
    Yp = q4.gemm_skinny(W, X[perm].contiguous())
    for i, b in enumerate(perm.tolist()):
        assert torch.equal(Yp[i], singles[b][0])
    torch.cuda.synchronize()


@pytest.mark.parametrize("kernel", ["0", "3"])
def test_k_split_path_parity_and_invariance(q4, monkeypatch, kernel):
    """The kernels that stage activations per CTA split K across CTAs when asked (workspace path)."""
    monkeypatch.setenv("Q4_KERNEL", kernel)
    monkeypatch.setenv("Q4_KSPLIT", "3")
    N, K = 3072, 3072
    assert q4.plan(N, K)["k_splits"] == 3
    w, x = synthetic.random_shape_problem(N, K, 8, seed=77, outliers=True)
    W = q4.QuantizedMatrix.from_float(w)
    ws = q4.Workspace(q4.workspace_bytes(N, K, 8))
    X = bf16_tensor(x)
    Y8 = q4.gemm_skinny(W, X, workspace=ws)
    Y8b = q4.gemm_skinny(W, X, workspace=ws)          # counters were reset by the first call
    for b in range(8):
        y1 = q4.gemm_skinny(W, X[b:b + 1].contiguous(), workspace=ws)
        assert torch.equal(Y8[b], y1[0])
    assert torch.equal(Y8, Y8b)
    torch.cuda.synchronize()
    assert within_tol(f"k-split 3 kernel {kernel} N=3072 K=3072 B=8", Y8.cpu().numpy(), oracle_rows(w, x))
    assert int(ws.buf[:256].view(torch.int32)[: q4.plan(N, K)["row_blocks"]].abs().sum()) == 0


@pytest.mark.parametrize("env", [{"Q4_KERNEL": "0"}, {"Q4_KERNEL": "1"}, {"Q4_KERNEL": "2"}, {"Q4_KERNEL": "3"},
                                 {"Q4_KERNEL": "4"}, {"Q4_KERNEL": "6"}, {"Q4_KERNEL": "6", "Q4_PDL": "0"},
                                 {"Q4_KERNEL": "3", "Q4_SW": "8", "Q4_SD": "1"},
                                 {"Q4_KERNEL": "3", "Q4_SW": "4", "Q4_SD": "4"},
                                 {"Q4_KERNEL": "3", "Q4_SW": "6", "Q4_SD": "2"},
                                 {"Q4_KERNEL": "3", "Q4_KSPLIT": "3"},
                                 {"Q4_KERNEL": "0", "Q4_DEPTH": "2"}, {"Q4_KERNEL": "0", "Q4_DEPTH": "6"},
                                 {"Q4_KERNEL": "0", "Q4_WARPS": "8", "Q4_DEPTH": "4"},
                                 {"Q4_KERNEL": "0", "Q4_WARPS": "8", "Q4_DEPTH": "8"},
                                 {"Q4_KERNEL": "1", "Q4_DEPTH": "6"},
                                 {"Q4_PDL": "0"}, {"Q4_KERNEL": "0", "Q4_KSPLIT": "2"}, {"Q4_ROTATE": "0"}])
def test_kernel_variants(q4, monkeypatch, env):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    for (N, K) in ((1000, 1152), (3072, 3072), (25088, 1024), (6000, 8192)):
        w, x = synthetic.random_shape_problem(N, K, 8, seed=5, outliers=True)
        W = q4.QuantizedMatrix.from_float(w)
        X = bf16_tensor(x)
        Y = q4.gemm_skinny(W, X)
        y1 = q4.gemm_skinny(W, X[3:4].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(Y[3], y1[0])
        rows = _sample_rows(N, n=2048)
        assert within_tol(f"variant {env} N={N} K={K} B=8", Y.cpu().numpy()[:, rows], oracle_rows(w, x, rows))
    q4.device_status()


def test_back_to_back_calls_keep_stream_order(q4):
    """Single calls enqueued back to back (each launch may start while the one before is still
    running, and streams its weights early) give exactly what each call gives alone: the same
    output buffer written by consecutive calls ends with the last call's values, and calls that
    share one workspace do not see each other's prepared activations."""
    cases = [(25088, 3072), (3072, 3072), (3072, 8192), (1000, 1152), (25088, 3072), (3072, 8192)]
    mats, xs = [], []
    for i, (N, K) in enumerate(cases):
        w, x = synthetic.random_shape_problem(N, K, 8, seed=300 + i, outliers=True)
        mats.append((q4.QuantizedMatrix.from_float(w), w))
        xs.append(x)
    for B in (1, 3, 8):
        X = [bf16_tensor(x[:B]) for x in xs]
        ws = q4.Workspace(max(q4.workspace_bytes(W.N, W.K, B) for W, _ in mats))
        alone = []
        for (W, _), x in zip(mats, X):
            alone.append(q4.gemm_skinny(W, x, workspace=ws))
            torch.cuda.synchronize()
        Y = [torch.full((B, W.N), float("nan"), device="cuda") for W, _ in mats]
        shared = torch.full((B * 25088,), float("nan"), device="cuda")
        for _ in range(2):
            for (W, _), x, y in zip(mats, X, Y):
                q4.gemm_skinny(W, x, y, workspace=ws)
            for (W, _), x in zip(mats[:2], X[:2]):  # write after write on one buffer: the last call wins
                q4.gemm_skinny(W, x, shared[:B * W.N].view(B, W.N), workspace=ws)
        torch.cuda.synchronize()
        for i, (a, y) in enumerate(zip(alone, Y)):
            assert torch.equal(a, y), (B, i)
        assert torch.equal(shared[:B * 3072], alone[1].flatten())
        assert torch.equal(shared[B * 3072:], alone[0].flatten()[B * 3072:])
        rows = _sample_rows(25088, n=256)
        assert within_tol(f"back-to-back fused B={B}", Y[0].cpu().numpy()[:, rows],
                          oracle_rows(mats[0][1], xs[0][:B], rows))
    q4.device_status()


# ----------------------------------------------------------------------------- full-size configs
def _sample_rows(N, outl_rows=None, n=1024, seed=1):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, min(n, N), replace=False).tolist()) | {0, N - 1, N // 2}
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["fused", "oproj", "down"])
@pytest.mark.parametrize("B", [1, 8])
def test_full_size_projection_sampled_rows(q4, name, B):
    w, x = synthetic.problem(name, B, seed=0)
    W = q4.QuantizedMatrix.from_float(w)
    y = run(q4, W, x)
    rows = _sample_rows(w.shape[0])
    assert within_tol(f"full {name} B={B} ({rows.size} sampled rows)", y[:, rows], oracle_rows(w, x, rows))
    # packing of the sampled rows is bit-exact
    c, s, m = (t.cpu().numpy() for t in (W.codes, W.scales.view(torch.int16), W.mins.view(torch.int16)))
    oc, osb, omb = oracle.quantise(np.ascontiguousarray(w[rows]))
    assert np.array_equal(c[rows], oracle.pack(oc))
    assert np.array_equal(s[rows].view(np.uint16), osb) and np.array_equal(m[rows].view(np.uint16), omb)


@pytest.mark.parametrize("B", [1, 8])
def test_head_and_argmax_exact(q4, B):
    w, x = synthetic.problem("head", B, seed=0)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    Y = q4.gemm_skinny(W, X)
    idx = q4.argmax(Y)
    torch.cuda.synchronize()
    y = Y.cpu().numpy()
    # argmax kernel == numpy on the same fp32 logits (exact)
    assert idx.cpu().numpy().tolist() == np.argmax(y, axis=1).tolist()
    # oracle logits: full head in row chunks
    y_ref = oracle_rows(w, x)
    assert within_tol(f"full head B={B} (all rows)", y, y_ref)
    ref_idx = oracle.argmax_first(y_ref)
    bound = 2.0 * float(np.abs(y - y_ref).max())     # either index is right inside the GPU's own error
    for b in range(B):
        if oracle.argmax_ambiguous(y_ref[b], bound):
            assert y_ref[b, idx[b].item()] >= y_ref[b].max() - bound
        else:
            assert idx[b].item() == ref_idx[b]


@pytest.mark.parametrize("cluster", ["1", "0"])
def test_argmax_ties_nan_and_layout(q4, monkeypatch, cluster):
    """Both argmax kernels: a cluster of 8 CTAs per row (default) and one CTA per row."""
    monkeypatch.setenv("Q4_ARGMAX_CLUSTER", cluster)
    y = np.random.default_rng(0).standard_normal((8, 70001)).astype(np.float32)
    y[0, 5] = y[0, 9] = 100.0               # tie: lowest index
    y[1, :] = 0.0; y[1, 3] = -0.0           # all equal: index 0
    y[2, 123] = np.nan; y[2, 7] = 1e30       # NaN ranks first (numpy convention)
    y[3, -1] = 50.0                          # last element
    y[4, :] = -np.inf; y[4, 17] = -1e38
    Y = torch.from_numpy(y).cuda()
    got = q4.argmax(Y).cpu().numpy()
    assert got.tolist() == np.argmax(y, axis=1).tolist()
    assert got[0] == 5 and got[1] == 0 and got[2] == 123 and got[3] == 70000 and got[4] == 17
    # short and oddly aligned rows: scalar head, vector body and scalar tail of every size
    rng = np.random.default_rng(1)
    for N in (1, 2, 3, 4, 5, 7, 9, 31, 33, 4097, 4099, 65536, 65539):
        y = rng.standard_normal((8, N)).astype(np.float32)
        got = q4.argmax(torch.from_numpy(y).cuda()).cpu().numpy()
        assert got.tolist() == np.argmax(y, axis=1).tolist(), N
        flat = torch.from_numpy(rng.standard_normal(3 * N + 1).astype(np.float32)).cuda()
        view = flat[1:].view(3, N)                 # rows start 4 bytes past a 16-byte boundary
        got = q4.argmax(view).cpu().numpy()
        assert got.tolist() == np.argmax(view.cpu().numpy(), axis=1).tolist(), N


# ----------------------------------------------------------------------------- decode step
def _decode_mats(q4, layers, B, base=0):
    mats, xs, ws_np = [], [], []
    for l in range(layers):
        for p in range(3):
            w, x = synthetic.decode_step_matrix(l, p, B, base)
            mats.append(q4.QuantizedMatrix.from_float(w))
            xs.append(x)
            ws_np.append(w)
    return mats, xs, ws_np


@pytest.mark.parametrize("B", [1, 8])
def test_decode_step_graph_equals_eager_and_oracle(q4, B):
    layers = 3
    mats, xs, ws_np = _decode_mats(q4, layers, B)
    g = q4.DecodeStepGraph(mats, B)
    for i, x in enumerate(xs):
        g.X[i].copy_(bf16_tensor(x))
    g.replay()
    g.replay()                                  # replays are repeatable
    eager_Y = [torch.empty_like(y) for y in g.Y]
    q4.decode_step(mats, g.X, eager_Y, g.ws)
    torch.cuda.synchronize()
    for i in range(len(mats)):
        assert torch.equal(g.Y[i], eager_Y[i]), i
    # the two phases called separately give the same bits as the one call
    ws2 = q4.Workspace(q4.step_workspace_bytes([m.K for m in mats], B))
    Y2 = [torch.empty_like(y) for y in g.Y]
    q4.step_prepare(mats, g.X, ws2)
    q4.step_stream(mats, Y2, B, ws2)
    torch.cuda.synchronize()
    for i in range(len(mats)):
        assert torch.equal(Y2[i], eager_Y[i]), i
    for i in range(len(mats)):
        rows = _sample_rows(ws_np[i].shape[0], n=256, seed=i)
        y = g.Y[i].cpu().numpy()
        assert within_tol(f"decode step B={B} matrix {i}", y[:, rows], oracle_rows(ws_np[i], xs[i], rows)), i


def test_graph_run_host_one_copy(q4):
    """The activation buffers are views of one contiguous buffer: one pinned host tensor laid out
    like it feeds the whole step, with the same outputs and argmax as filling the views."""
    mats, xs, _ = _decode_mats(q4, 1, 2, base=60)
    g = q4.DecodeStepGraph(mats, 2, with_argmax_of=0)
    assert all(x.data_ptr() % 16 == 0 for x in g.X)
    for i, x in enumerate(xs):
        g.X[i].copy_(bf16_tensor(x))
    g.replay()
    Y_ref = [y.clone() for y in g.Y]
    idx_ref = g.idx.clone()
    host = g.X_flat.cpu().pin_memory()
    g.X_flat.zero_()
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in g.Y]
    hidx = torch.empty(g.idx.shape, dtype=g.idx.dtype).pin_memory()
    g.run_host(host, hy, hidx)
    for a, b in zip(hy, Y_ref):
        assert torch.equal(a, b.cpu())
    assert torch.equal(hidx, idx_ref.cpu())


def test_decode_step_independent_and_chained_agree(q4):
    """Independent lists run the tile kernel, chained ones the direct kernel: both match the oracle,
    agree to fp32 rounding, and each is batch-invariant."""
    mats, xs, ws_np = _decode_mats(q4, 2, 4)
    X = [bf16_tensor(x) for x in xs]
    Y1 = [torch.empty((4, m.N), device="cuda") for m in mats]
    Y2 = [torch.empty((4, m.N), device="cuda") for m in mats]
    shapes = [(m.N, m.K) for m in mats]
    q4.decode_step(mats, X, Y1, q4.Workspace.for_shapes(shapes, 4, independent=True), independent=True)
    q4.decode_step(mats, X, Y2, q4.Workspace.for_shapes(shapes, 4, independent=False), independent=False)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(Y1, Y2)):
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-5), i
        rows = _sample_rows(ws_np[i].shape[0], n=128, seed=i)
        ref = oracle_rows(ws_np[i], xs[i], rows)
        assert within_tol(f"independent list matrix {i}", a.cpu().numpy()[:, rows], ref)
        assert within_tol(f"chained list matrix {i}", b.cpu().numpy()[:, rows], ref)
    # batch invariance of the independent list: column 2 alone equals column 2 of the batch
    Y3 = [torch.empty((1, m.N), device="cuda") for m in mats]
    q4.decode_step(mats, [x[2:3].contiguous() for x in X], Y3, independent=True)
    torch.cuda.synchronize()
    for a, c in zip(Y1, Y3):
        assert torch.equal(a[2], c[0])
    q4.device_status()


@pytest.mark.parametrize("env", [{"Q4_TW": "16"}, {"Q4_TW": "24"}, {"Q4_TW": "32"}, {"Q4_TCONTIG": "1"},
                                 {"Q4_TCONTIG": "0"}, {"Q4_TCONTIG": "1", "Q4_TW": "24"}])
def test_tile_kernel_shapes(q4, monkeypatch, env):
    """Every warp count / ring depth of the tile kernel: oracle parity and batch invariance; the
    shapes share one arithmetic order, so they agree bit for bit with the default."""
    mats, xs, ws_np = _decode_mats(q4, 1, 3, base=40)
    X = [bf16_tensor(x) for x in xs]
    Y0 = [torch.empty((3, m.N), device="cuda") for m in mats]
    q4.decode_step(mats, X, Y0)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    Y = [torch.empty((3, m.N), device="cuda") for m in mats]
    Y1 = [torch.empty((1, m.N), device="cuda") for m in mats]
    q4.decode_step(mats, X, Y)
    q4.decode_step(mats, [x[1:2].contiguous() for x in X], Y1)
    torch.cuda.synchronize()
    for i in range(len(mats)):
        assert torch.equal(Y[i][1], Y1[i][0]), i
        assert torch.equal(Y[i], Y0[i]), i
        rows = _sample_rows(ws_np[i].shape[0], n=128, seed=i)
        assert within_tol(f"tile kernel {env} matrix {i}", Y[i].cpu().numpy()[:, rows],
                          oracle_rows(ws_np[i], xs[i], rows)), i
    q4.device_status()


def test_single_calls_share_one_workspace(q4):
    """Single calls on matrices of different shapes, one workspace reused in both orders: every call
    matches the oracle and repeats bit for bit (nothing a call leaves behind changes the next)."""
    shapes = [(25088, 3072), (3072, 8192), (100, 1152), (3072, 3072), (4099, 1024), (16, 128)]
    B = 3
    probs = [synthetic.random_shape_problem(N, K, B, seed=20 + i) for i, (N, K) in enumerate(shapes)]
    mats = [q4.QuantizedMatrix.from_float(w) for w, _ in probs]
    Xs = [bf16_tensor(x) for _, x in probs]
    ws = q4.Workspace(max(q4.workspace_bytes(N, K, B) for N, K in shapes))
    first = [q4.gemm_skinny(W, X, workspace=ws) for W, X in zip(mats, Xs)]
    again = [q4.gemm_skinny(W, X, workspace=ws) for W, X in reversed(list(zip(mats, Xs)))][::-1]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(first, again)):
        assert torch.equal(a, b), shapes[i]
        rows = _sample_rows(shapes[i][0], n=256, seed=i)
        assert within_tol(f"shared workspace {shapes[i]}", a.cpu().numpy()[:, rows],
                          oracle_rows(probs[i][0], probs[i][1], rows)), shapes[i]
    q4.device_status()


def test_long_list_spans_several_launches(q4):
    """More matrices than one launch's table: the list is cut into launches, results unchanged."""
    n = 140
    w, x = synthetic.random_shape_problem(64, 256, 2, seed=9)
    W = q4.QuantizedMatrix.from_float(w)
    X = [bf16_tensor(x) for _ in range(n)]
    Y = [torch.empty((2, 64), device="cuda") for _ in range(n)]
    q4.decode_step([W] * n, X, Y)
    torch.cuda.synchronize()
    for y in Y:
        assert torch.equal(y, Y[0])
    assert within_tol("140-matrix list", Y[0].cpu().numpy(), oracle_rows(w, x))


def test_decode_step_chained_dependency(q4):
    """Y of one launch feeding X of the next is honoured (the launch waits for its producer)."""
    w1, x1 = synthetic.random_shape_problem(1024, 1024, 1, seed=1)
    w2, _ = synthetic.random_shape_problem(512, 1024, 1, seed=2)
    W1, W2 = q4.QuantizedMatrix.from_float(w1), q4.QuantizedMatrix.from_float(w2)
    X1 = bf16_tensor(x1)
    Y1 = torch.empty((1, 1024), dtype=torch.float32, device="cuda")
    X2 = torch.empty((1, 1024), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty((1, 512), dtype=torch.float32, device="cuda")
    for _ in range(3):
        q4.decode_step([W1], [X1], [Y1], independent=False)
        X2.copy_(Y1)                               # a torch kernel between the two launches
        q4.decode_step([W2], [X2], [Y2], independent=False)
    torch.cuda.synchronize()
    ref = q4.gemm_skinny(W2, Y1.to(torch.bfloat16))
    torch.cuda.synchronize()
    assert torch.equal(ref, Y2)


# ----------------------------------------------------------------------------- guard bands + errors
def test_outputs_stay_inside_their_buffers(q4):
    N, K, B = 1001, 640, 3
    w, x = synthetic.random_shape_problem(N, K, B, seed=4)
    W = q4.QuantizedMatrix.from_float(w)
    pad = 1024
    big = torch.full((B * N + 2 * pad,), 12345.0, dtype=torch.float32, device="cuda")
    Y = big[pad:pad + B * N].view(B, N)
    q4.gemm_skinny(W, bf16_tensor(x), Y=Y)
    torch.cuda.synchronize()
    assert bool((big[:pad] == 12345.0).all()) and bool((big[pad + B * N:] == 12345.0).all())
    assert oracle.rel_err(Y.cpu().numpy(), oracle_rows(w, x)) <= TOL


def test_error_statuses_on_device(q4, monkeypatch):
    import ctypes
    from int4_weight_only_q4_gb300 import _lib
    w, x = synthetic.random_shape_problem(3072, 3072, 1, seed=1)
    W = q4.QuantizedMatrix.from_float(w)
    X = bf16_tensor(x)
    Y = torch.empty((1, 3072), dtype=torch.float32, device="cuda")
    m = W.c_struct()
    L = _lib.lib
    # misaligned x
    assert L.q4_gemv(ctypes.byref(m), X.data_ptr() + 2, Y.data_ptr(), None, 0, None) == _lib.Q4_ERR_MISALIGNED
    # workspace required but missing / too small under a forced k-split of the direct kernel
    monkeypatch.setenv("Q4_KERNEL", "0")
    monkeypatch.setenv("Q4_KSPLIT", "2")
    need = q4.workspace_bytes(3072, 3072, 1)
    assert need > 0
    assert L.q4_gemv(ctypes.byref(m), X.data_ptr(), Y.data_ptr(), None, 0, None) == _lib.Q4_ERR_WORKSPACE
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    assert L.q4_gemv(ctypes.byref(m), X.data_ptr(), Y.data_ptr(), ws.data_ptr(), need - 16, None) == \
        _lib.Q4_ERR_WORKSPACE
    assert L.q4_gemv(ctypes.byref(m), X.data_ptr(), Y.data_ptr(), ws.data_ptr(), need, None) == _lib.Q4_OK
    monkeypatch.delenv("Q4_KSPLIT")
    monkeypatch.delenv("Q4_KERNEL")
    # a simulated launch failure is reported, and nothing is launched
    Y.fill_(7.0)
    wsz = q4.workspace_bytes(3072, 3072, 1)
    ws2 = torch.zeros(max(wsz, 16), dtype=torch.uint8, device="cuda")
    monkeypatch.setenv("Q4_FAULT_INJECT", "launch")
    assert L.q4_gemv(ctypes.byref(m), X.data_ptr(), Y.data_ptr(), ws2.data_ptr(), wsz, None) == _lib.Q4_ERR_CUDA
    with pytest.raises(q4.Q4Error):
        q4.gemv(W, X[0], Y[0])
    monkeypatch.delenv("Q4_FAULT_INJECT")
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())
    # the context is healthy afterwards, and no device-side wait gave up
    y = q4.gemv(W, X[0])
    q4.device_status()
    torch.cuda.synchronize()
    assert oracle.rel_err(y.cpu().numpy()[None], oracle_rows(w, x)) <= TOL


def test_read_only_twin_runs_the_same_launch(q4):
    """The measurement twin of the step kernel takes the same arguments and checks, launches cleanly
    on a decode-step list and leaves no device error; it touches only the outputs it is given."""
    mats, xs, _ = _decode_mats(q4, 1, 2, base=70)
    X = [bf16_tensor(x) for x in xs]
    ws = q4.Workspace(q4.step_workspace_bytes([m.K for m in mats], 2))
    pad = 256
    bufs = [torch.full((2 * m.N + 2 * pad,), 12345.0, device="cuda") for m in mats]
    Y = [b[pad:pad + 2 * m.N].view(2, m.N) for b, m in zip(bufs, mats)]
    q4.step_prepare(mats, X, ws)
    q4.step_stream_readonly(mats, Y, 2, ws)
    torch.cuda.synchronize()
    q4.device_status()
    for b, m in zip(bufs, mats):
        assert bool((b[:pad] == 12345.0).all()) and bool((b[pad + 2 * m.N:] == 12345.0).all())
    Y2 = [torch.empty((2, m.N), device="cuda") for m in mats]
    q4.step_stream(mats, Y2, 2, ws)            # the real kernel on the same prepared activations
    torch.cuda.synchronize()
    ref = [torch.empty_like(y) for y in Y2]
    q4.decode_step(mats, X, ref)
    torch.cuda.synchronize()
    for a, b in zip(Y2, ref):
        assert torch.equal(a, b)
