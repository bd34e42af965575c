"""GPU parity of flash-decoding attention (q4_flash_decode) against the fp64 CPU oracle
(oracle/attn_oracle.py).

One decode step of grouped-query attention over a KV cache, split over chunks of the cache and
merged by a second kernel (rumik-oss-1 write-up, "Step 6: flash-decoding for long clips").

Tolerance.  An output is a softmax-weighted mean of value rows, so an error in the weights shows
up relative to the weighted mean of |V|, A = sum_p w_p |v_p| (the oracle run on |V|, i.e. with
the value sign bits cleared).  The bound is |O - O_ref| <= 1e-4 * A per element.  The weights
carry the fp32 rounding of the scores (products of bf16 values are exact on the tensor cores;
sums of 128 terms of size <= 45 round to ~1e-5 absolute, times scale), of u = s * scale * log2 e
(|u| <= ~40: ~3e-6), of exp2 (2 ulp) and of the bf16 hi + lo split (2^-18 ~ 4e-6): below 1e-5
relative, and the fp32 accumulation of P V adds less than that at these lengths -- a factor of
ten under the bound.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle.attn_oracle as A
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as m
    return m


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run(q4, Q, K, V, lens, scale=None, n_chunks=0):
    O = q4.flash_decode(dev_bf16(Q), dev_bf16(K), dev_bf16(V), torch.from_numpy(lens).cuda(),
                        scale=scale, n_chunks=n_chunks)
    torch.cuda.synchronize()
    return O.cpu().numpy().astype(np.float64)


def attn_err(O, Q, K, V, lens, scale, heads=None):
    """max |O - O_ref| / (weighted mean of |V|) over the compared outputs."""
    ref = A.decode_attention(Q, K, V, lens, scale, heads=heads)
    mag = A.decode_attention(Q, K, V & np.uint16(0x7FFF), lens, scale, heads=heads)
    if heads is not None:
        sel = tuple(np.array(heads).T)
        O, ref, mag = O[sel], ref[sel], mag[sel]
    den = np.where(mag > 0, mag, 1.0)
    return float(np.max(np.abs(O - ref) / den)) if O.size else 0.0


def _log(label, e):
    import json, os
    log = os.environ.get("Q4_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": label, "attn_err": e}) + "\n")


def check(q4, B, Hq, Hkv, D, Lmax, lens, seed, q_std=1.0, n_chunks=0, label=""):
    Q, K, V, lens = synthetic.attention_problem(B, Hq, Hkv, D, Lmax, lens, seed, q_std=q_std)
    scale = 1 / math.sqrt(D)
    O = run(q4, Q, K, V, lens, n_chunks=n_chunks)
    e = attn_err(O, Q, K, V, lens, scale)
    _log(label or f"attn B={B} Hq={Hq} Hkv={Hkv} D={D} L={list(lens)} C={n_chunks} qs={q_std}", e)
    assert e <= TOL, (label, e)
    for b in range(B):
        if lens[b] == 0:
            assert not O[b].any()
    return Q, K, V, lens, O


@pytest.mark.parametrize("n_chunks", [0, 16])
def test_page_case_2000_positions(q4, n_chunks):
    # 24 query heads sharing 6 KV heads, head_dim 128, a 2,000-position cache, batch 1
    check(q4, 1, 24, 6, 128, 2000, [2000], 0, n_chunks=n_chunks)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_group_sizes_and_head_dims(q4, D, g):
    check(q4, 2, 2 * g, 2, D, 300, [300, 129], 10 + g)


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_lengths(q4, D):
    check(q4, 6, 8, 2, D, 400, [0, 1, 15, 17, 333, 400], 20)


@pytest.mark.parametrize("n_chunks", [1, 3, 7, 64, 1000, 4096])
def test_chunk_counts(q4, n_chunks):
    check(q4, 2, 8, 2, 128, 1500, [1500, 37], 30, n_chunks=n_chunks)


@pytest.mark.parametrize("q_std", [0.1, 4.0, 8.0])
def test_flat_and_peaked_softmax(q4, q_std):
    check(q4, 2, 24, 6, 128, 1024, [1024, 700], 40, q_std=q_std)


def test_one_position_returns_its_value(q4):
    Q, K, V, lens, O = check(q4, 2, 8, 2, 64, 1, [1, 1], 50)
    f = synthetic.bf16_bits_to_f32(V).astype(np.float64)
    for h in range(8):
        assert np.array_equal(O[:, h], f[:, h // 4, 0])      # a single weight of exactly 1


def test_lengths_past_the_cache_are_clamped(q4):
    Q, K, V, lens = synthetic.attention_problem(2, 8, 2, 128, 64, [64, 64], 60)
    a = run(q4, Q, K, V, lens)
    b = run(q4, Q, K, V, np.array([1000, 2 ** 31 - 1], np.int32))
    c = run(q4, Q, K, V, np.array([-5, 0], np.int32))
    assert np.array_equal(a, b)
    assert not c.any()


def test_cache_past_the_length_is_never_read(q4):
    Q, K, V, lens = synthetic.attention_problem(3, 12, 3, 128, 256, [256, 100, 17], 70)
    K2, V2 = K.copy(), V.copy()
    for b, n in enumerate(lens):
        K2[b, :, n:] = 0x7FC0        # NaN
        V2[b, :, n:] = 0x7F80        # +inf
    assert np.array_equal(run(q4, Q, K, V, lens), run(q4, Q, K2, V2, lens))


def test_batch_invariance_and_determinism(q4):
    Q, K, V, lens = synthetic.attention_problem(8, 24, 6, 128, 1200, [1200, 5, 777, 1199, 64, 0, 1000, 33], 80)
    full = run(q4, Q, K, V, lens)
    again = run(q4, Q, K, V, lens)
    assert np.array_equal(full, again)
    for b in (0, 2, 5, 7):
        one = run(q4, Q[b:b + 1], K[b:b + 1], V[b:b + 1], lens[b:b + 1])
        assert np.array_equal(one[0], full[b]), b


def test_graph_replay_with_new_lengths(q4):
    # one captured step serves every length up to the cache size: the lengths are read on the device
    Q, K, V, lens = synthetic.attention_problem(2, 24, 6, 128, 512, [512, 300], 90)
    dq, dk, dv = dev_bf16(Q), dev_bf16(K), dev_bf16(V)
    dl = torch.from_numpy(lens).cuda()
    O = torch.empty((2, 24, 128), dtype=torch.float32, device="cuda")
    ws = q4.flash_decode_workspace(2, 24, 6, 128)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        q4.flash_decode(dq, dk, dv, dl, O, workspace=ws, stream=side)
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            q4.flash_decode(dq, dk, dv, dl, O, workspace=ws, stream=side)
    for new in ([1, 512], [511, 2], [0, 250]):
        nl = np.array(new, np.int32)
        dl.copy_(torch.from_numpy(nl))
        g.replay()
        torch.cuda.synchronize()
        got = O.cpu().numpy().astype(np.float64)
        assert attn_err(got, Q, K, V, nl, 1 / math.sqrt(128)) <= TOL, new
        assert np.array_equal(got, run(q4, Q, K, V, nl)), new


@pytest.mark.parametrize("fill", ["0", "1"])
def test_both_ring_fills_give_the_same_bits(q4, fill, monkeypatch):
    # bulk row copies (default) and per-lane cp.async fill the ring with the same data
    Q, K, V, lens = synthetic.attention_problem(3, 24, 6, 128, 700, [700, 333, 17], 110)
    ref = run(q4, Q, K, V, lens)
    monkeypatch.setenv("Q4_FD_BULK", fill)
    for stages in ("2", "3"):
        monkeypatch.setenv("Q4_FD_STAGES", stages)
        assert np.array_equal(run(q4, Q, K, V, lens), ref), (fill, stages)


def test_combine_thread_counts_give_the_same_bits(q4, monkeypatch):
    # the combine sums chunk classes in a fixed order whatever its CTA size (512 or 256 threads)
    Q, K, V, lens = synthetic.attention_problem(2, 24, 6, 128, 3000, [3000, 1111], 130)
    Q64, K64, V64, lens64 = synthetic.attention_problem(2, 8, 2, 64, 3000, [2999, 400], 131)
    for nc in (0, 16, 4096):
        monkeypatch.setenv("Q4_FD_COMBINE", "512")
        a = run(q4, Q, K, V, lens, n_chunks=nc)
        a64 = run(q4, Q64, K64, V64, lens64, n_chunks=nc)
        monkeypatch.setenv("Q4_FD_COMBINE", "256")
        assert np.array_equal(run(q4, Q, K, V, lens, n_chunks=nc), a), nc
        assert np.array_equal(run(q4, Q64, K64, V64, lens64, n_chunks=nc), a64), nc


def test_device_status_clean_after_calls(q4):
    check(q4, 2, 8, 2, 64, 300, [300, 2], 120)
    q4.device_status()


def test_long_cache_batch_8(q4):
    """Batch 8 over an 8,192-position cache (the bench's long case), ragged, all 192 heads."""
    lens = [8192, 8000, 4096, 1, 2000, 8191, 7777, 16]
    check(q4, 8, 24, 6, 128, 8192, lens, 100, label="attn long B=8 L=8192 ragged")
