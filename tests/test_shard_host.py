"""Host logic of the row-sharded step (int4_weight_only_q4_gb300.shard), on the CPU with gloo ranks.

What needs no GPU is checked here: the shard bounds (whole 16-row tiles covering every row once,
tile counts within one of each other), the exchange buffer's layout, the one all-gather that
moves every matrix's rows (gather order: rank-major, each matrix at its fixed offset), and the one
MAX all-reduce of 64-bit argmax keys that merges the per-rank maxima (equal maxima on two ranks
go to the lower global index, NaN ranks first, -0 equals +0).  The keys are built here from the
format q4.h documents; a GPU test checks that q4_argmax_key_f32 writes exactly that format.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

from int4_weight_only_q4_gb300 import shard

SHAPES = [25088, 3072, 1000, 33, 65536, 48]


def doc_key(v: float, gidx: int) -> int:
    """The documented key of logit v at global row gidx, as the signed int64 the all-reduce sees."""
    f = np.float32(v)
    if np.isnan(f):
        r = 0xFFFFFFFF
    else:
        b = int(np.array([f]).view(np.uint32)[0])
        if b & 0x7FFFFFFF == 0:
            b = 0
        r = (~b & 0xFFFFFFFF) if b & 0x80000000 else (b | 0x80000000)
    u = (r << 32) | (~gidx & 0xFFFFFFFF)
    u ^= 1 << 63
    return u - (1 << 64) if u >= 1 << 63 else u


def key_index(k: int) -> int:
    return ~k & 0xFFFFFFFF


@pytest.mark.parametrize("N", [1, 15, 16, 17, 1000, 3072, 25088, 65536])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_row_shards_cover_every_row_in_whole_tiles(N, P):
    T = (N + 15) // 16
    if T < P:
        with pytest.raises(ValueError):
            shard.row_shards(N, P)
        return
    sh = shard.row_shards(N, P)
    assert len(sh) == P and sh[0][0] == 0 and sh[-1][1] == N
    for (s0, e0), (s1, _) in zip(sh, sh[1:]):
        assert e0 == s1                                  # contiguous, no overlap
    tiles = []
    for s, e in sh:
        assert s % 16 == 0 and e > s
        assert e % 16 == 0 or e == N
        tiles.append((e - s + 15) // 16)
    assert max(tiles) - min(tiles) <= 1 and sum(tiles) == T


def test_layout_slots_are_disjoint_and_aligned():
    for P in (1, 2, 3):
        for B in (1, 3, 8):
            L = shard.ShardLayout.build(SHAPES, P, B)
            ends = 0
            for i, N in enumerate(SHAPES):
                assert L.off[i] % 4 == 0 and L.off[i] >= ends
                ends = L.off[i] + B * L.rmax[i]
                assert L.rmax[i] == max(e - s for s, e in L.shards[i])
            assert L.per_rank >= ends and L.per_rank % 4 == 0


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from int4_weight_only_q4_gb300 import shard as S
    B = 3
    L = S.ShardLayout.build(SHAPES, world, B)
    rng = np.random.default_rng(7)
    full = [rng.standard_normal((B, N)).astype(np.float32) for N in SHAPES]   # the same on every rank
    send = torch.full((L.per_rank,), float("nan"))
    for i, y in enumerate(full):
        s, e = L.shards[i][rank]
        L.local_view(send, i, rank).copy_(torch.from_numpy(y[:, s:e]))
    recv = torch.empty((world * L.per_rank,))
    S.all_gather_outputs(send, recv)
    gathered_ok = all(np.array_equal(L.assemble(recv, i).numpy(), y) for i, y in enumerate(full))
    # argmax keys of the head-like matrix 4: this rank's best per batch row, merged by MAX
    head = full[4].copy()
    s4 = L.shards[4]
    head[0, s4[0][0] + 5] = head[0, s4[-1][0] + 3] = 100.0      # equal maxima on the first and last rank
    head[1, s4[-1][0] + 9] = np.nan                              # NaN on the last rank only
    head[1, s4[0][0] + 2] = 1e30
    head[2, :] = -0.0
    head[2, s4[-1][0] + 1] = 0.0                                 # -0 == +0: index 0 wins
    s, e = s4[rank]
    keys = []
    for b in range(B):
        keys.append(max(doc_key(head[b, n], n) for n in range(s, e)))
    kt = torch.tensor(keys, dtype=torch.int64)
    S.all_reduce_keys(kt)
    got = [key_index(int(k)) for k in kt.tolist()]
    dist.barrier()
    out[rank] = (gathered_ok, got, np.argmax(head, axis=1).tolist())
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gather_order_and_argmax_merge_over_gloo_ranks(world):
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        gathered_ok, got, want = res[r]
        assert gathered_ok, r
        assert got == want, (r, got, want)
    L = shard.ShardLayout.build(SHAPES, world, 3)
    assert res[0][1][0] == L.shards[4][0][0] + 5                 # the lower of the two equal maxima
    assert res[0][1][1] == L.shards[4][-1][0] + 9                # NaN first
    assert res[0][1][2] == 0


def test_documented_key_orders_like_the_argmax_rule():
    """Larger key <=> ranks above in the argmax order (NaN first, larger value, then lower index)."""
    vals = [np.nan, np.inf, 3.0, 1.0, 0.0, -0.0, -1.0, -np.inf]
    idxs = [0, 1, 7, 1 << 20, 4_000_000_000]
    pairs = [(v, i) for v in vals for i in idxs]

    def above(a, b):
        (va, ia), (vb, ib) = a, b
        na, nb = np.isnan(va), np.isnan(vb)
        if na or nb:
            return na and (not nb or ia < ib)
        return va > vb or (va == vb and ia < ib)

    for a in pairs:
        for b in pairs:
            if a is b:
                continue
            ka, kb = doc_key(*a), doc_key(*b)
            if above(a, b):
                assert ka > kb, (a, b)
            elif above(b, a):
                assert ka < kb, (a, b)
        assert key_index(doc_key(*a)) == a[1]
