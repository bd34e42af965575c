"""Row-sharded step on one GPU, with the ranks emulated one after another (no collective).

One GPU runs every rank's share in turn -- each a separate ShardedStep with its own rows and its own
CUDA graph, none waiting on another -- and the test stands in for the two collectives: the
all-gather is the concatenation of the ranks' exchange buffers, the MAX all-reduce an elementwise
maximum of their keys.  Checked: every assembled output is bit-identical to the unsharded step
(the tile kernel's arithmetic for a row does not depend on the other rows), the merged argmax
equals q4_argmax_f32 on the full logits, including equal maxima on two ranks and NaN, and the
keys q4_argmax_key_f32 writes are exactly the format q4.h documents.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synthetic
from test_shard_host import doc_key

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as m
    return m


def doc_keys(y: np.ndarray, base: int) -> np.ndarray:
    """doc_key over a row, vectorised: uint64 keys before the sign flip, as int64 after it."""
    b = y.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = np.where(b & 0x7FFFFFFF == 0, np.uint64(0), b)
    r = np.where(b & 0x80000000 != 0, ~b & np.uint64(0xFFFFFFFF), b | np.uint64(0x80000000))
    r = np.where(np.isnan(y), np.uint64(0xFFFFFFFF), r)
    g = (np.arange(y.size, dtype=np.uint64) + np.uint64(base)) & np.uint64(0xFFFFFFFF)
    u = (r << np.uint64(32)) | (~g & np.uint64(0xFFFFFFFF))
    return (u ^ np.uint64(1 << 63)).view(np.int64)


def test_argmax_key_kernel_writes_the_documented_keys(q4):
    rng = np.random.default_rng(3)
    B, N = 5, 70001
    y = rng.standard_normal((B, N)).astype(np.float32)
    y[0, 5] = y[0, 9] = 50.0
    y[1, 77] = np.nan
    y[2, :] = -0.0
    y[2, 10] = 0.0
    y[3, :] = -np.inf
    for base in (0, 12345, (1 << 32) - 1 - N):
        for lo, hi in ((0, N), (1, N), (3, 4099)):          # rows starting off a 16-byte boundary too
            Y = torch.from_numpy(np.ascontiguousarray(y[:, lo:hi])).cuda()
            keys = q4.argmax_keys(Y, base).cpu().numpy().tolist()
            for b in range(B):
                row = y[b, lo:hi]
                k = doc_keys(row, base)
                j = int(np.argmax(k))
                assert int(k[j]) == doc_key(float(row[j]), base + j)   # the vectorised form agrees
                assert keys[b] == int(k.max()), (base, lo, b)
            idx = q4.argmax_key_index(q4.argmax_keys(Y, base)).cpu().numpy()
            assert (idx.astype(np.int64) & 0xFFFFFFFF).tolist() == \
                [(base + int(np.argmax(y[b, lo:hi]))) & 0xFFFFFFFF for b in range(B)]


def _packed_list(q4, shapes, seed):
    out = []
    for i, (N, K) in enumerate(shapes):
        w, _ = synthetic.weights(N, K, seed + i, True)
        out.append(q4.pack_host(w))
    return out


@pytest.mark.parametrize("P", [2, 3])
@pytest.mark.parametrize("B", [1, 4])
def test_emulated_ranks_match_the_unsharded_step(q4, P, B):
    from int4_weight_only_q4_gb300 import shard
    shapes = [(25088, 3072), (3072, 3072), (3072, 8192), (1000, 1024), (6000, 3072)]
    head = len(shapes) - 1
    packed = _packed_list(q4, shapes, 90)
    rng = np.random.default_rng(B)
    xs = [synthetic.activations(B, K, rng) for _, K in shapes]
    full = [q4.QuantizedMatrix.from_packed(*p) for p in packed]
    g = q4.DecodeStepGraph(full, B, with_argmax_of=head)
    ranks = [shard.ShardedStep(packed, B, rank=r, world=P, head=head) for r in range(P)]
    for i, x in enumerate(xs):
        xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        g.X[i].copy_(xt)
        for st in ranks:
            st.graph.X[i].copy_(xt)
    g.replay()
    for st in ranks:
        st.graph.replay()
    torch.cuda.synchronize()
    L = ranks[0].layout
    gathered = torch.cat([st.send for st in ranks])               # stands in for the all-gather
    for i in range(len(shapes)):
        assert torch.equal(L.assemble(gathered, i), g.Y[i]), i
    keys = torch.stack([st.keys for st in ranks]).max(dim=0).values   # stands in for the all-reduce
    assert torch.equal(q4.argmax_key_index(keys), g.idx)
    # the key merge on edited copies of the head's logits: equal maxima on the first and the last
    # rank, and a NaN on the last rank
    Yh = g.Y[head].clone()
    sh = L.shards[head]
    Yh[0, sh[0][0] + 7] = Yh[0, sh[-1][0] + 2] = 1e6
    if B > 1:
        Yh[1, sh[-1][0] + 11] = float("nan")
    parts = [q4.argmax_keys(Yh[:, s:e].contiguous(), s) for s, e in sh]
    merged = torch.stack(parts).max(dim=0).values
    assert torch.equal(q4.argmax_key_index(merged), q4.argmax(Yh))
    assert int(q4.argmax_key_index(merged)[0]) == sh[0][0] + 7
    q4.device_status()
