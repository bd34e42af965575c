"""A model of the flash-decoding split kernel's integer bookkeeping, checked over random shapes
(CPU, no GPU).

The model restates csrc/q4_attn.cu's chunking (fd_chunking), the warp -> chunk assignment, the
ring's issue cursor (issue_next: chunk ic, tile it, slot islot, one call per computed tile plus
S - 1 ahead) and the compute cursor (slot rs, mbarrier phase), and checks the invariants the
kernel relies on:
  * every position 0..len-1 lies in exactly one tile of exactly one chunk, and chunk indices
    stay below the number used, which never exceeds the chunk capacity C;
  * each warp computes exactly the tiles it issued, in issue order, from the slot they were
    copied into, and waits on the mbarrier phase of that slot's current use (so no wait can be
    for a copy that was never issued, and no slot is refilled before its tile was computed);
  * the clamped copy positions stay inside [chunk start, chunk end) and inside the cache.
"""
import random

import pytest


def fd_chunking(n, Lmax, C, min_chunk):
    n = 0 if n < 0 else min(n, Lmax)
    per = (n + C - 1) // C
    cs = max((per + 15) // 16 * 16, min_chunk)
    used = (n + cs - 1) // cs
    return n, cs, used


def run_warp(w0, nw, length, cs, used, S):
    """Issue and compute sequences of one warp, as the kernel steps through them."""
    issued, computed = [], []
    state = {"ic": w0, "it": 0, "islot": 0}
    slot_uses = [0] * S          # completed uses of each slot (mbarrier phases passed)
    slot_tile = [None] * S       # tile currently held by each slot

    def issue_next():
        ic, it, islot = state["ic"], state["it"], state["islot"]
        if ic < used:
            s0 = ic * cs
            e0 = min(length, s0 + cs)
            base = s0 + 16 * it
            assert base < e0
            assert slot_tile[islot] is None, "slot refilled before its tile was computed"
            rows = [min(base + r, e0 - 1) for r in range(16)]
            assert all(s0 <= r < e0 for r in rows)
            slot_tile[islot] = (ic, base)
            issued.append((ic, base, islot))
            if base + 16 >= e0:
                state["ic"], state["it"] = ic + nw, 0
            else:
                state["it"] = it + 1
        state["islot"] = 0 if islot == S - 1 else islot + 1

    for _ in range(S - 1):
        issue_next()
    rs, phase = 0, 0
    cc = w0
    while cc < used:
        s0 = cc * cs
        e0 = min(length, s0 + cs)
        base = s0
        while base < e0:
            # the wait: the slot's current use must be this tile, with the expected parity
            assert slot_tile[rs] == (cc, base), "waiting on a slot that holds another tile"
            assert slot_uses[rs] & 1 == phase
            tile = slot_tile[rs]
            issue_next()                     # after the reads (bulk) or before (cp.async): same slots
            computed.append((cc, base, rs))
            slot_tile[rs] = None             # consumed
            slot_uses[rs] += 1
            if rs == S - 1:
                rs, phase = 0, phase ^ 1
            else:
                rs += 1
            base += 16
            assert tile[0] == cc
        cc += nw
    assert all(t is None for t in slot_tile), "a copy is still in flight at the end"
    return issued, computed


@pytest.mark.parametrize("seed", range(6))
def test_schedule_invariants_random_shapes(seed):
    rng = random.Random(seed)
    for _ in range(400):
        Lmax = rng.choice([1, 15, 16, 17, 31, 33, 100, 2000, 4096, 8192, 32768])
        n = rng.choice([0, 1, 2, 15, 16, 17, Lmax // 2, Lmax - 1, Lmax, Lmax + 5, -3])
        C = rng.choice([1, 2, 3, 7, 16, 50, 202, 1000, 4096])
        S = rng.choice([2, 3])
        warps_per_head = rng.choice([1, 4, 8, 24, 64])
        length, cs, used = fd_chunking(n, Lmax, C, 32)
        assert used <= C
        assert cs % 16 == 0 and cs >= 32
        covered = []
        for w0 in range(warps_per_head):
            if w0 >= used:
                continue                      # the kernel's early exit
            issued, computed = run_warp(w0, warps_per_head, length, cs, used, S)
            assert [(c, b) for c, b, _ in issued] == [(c, b) for c, b, _ in computed]
            assert [s for _, _, s in issued] == [s for _, _, s in computed]
            assert all(c < used for c, _, _ in computed)
            for c, b, _ in computed:
                e0 = min(length, c * cs + cs)
                covered.extend(range(b, min(b + 16, e0)))
        assert sorted(covered) == list(range(length))
