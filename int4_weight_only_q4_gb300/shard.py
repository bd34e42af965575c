"""Row-sharded decode step across GPUs, one process per GPU (torch.distributed).

A GEMV's output rows are independent: rank r of P holds rows [start_r, stop_r) of every matrix (and
their scale/min), the activations are replicated, and each rank computes its rows with the same
kernels as a single GPU -- the tile kernel's arithmetic for a row depends only on that row's
records and the activations, so every row is bit-identical to the unsharded step.  Two exchanges
follow, only where the full result is needed on every rank:

  * the outputs: one all-gather of one flat buffer that holds every matrix's local rows, each at a
    fixed offset and padded to the largest rank's row count, so one collective moves the step;
  * the head's argmax: each rank's best logit per batch row as one 64-bit key (q4_argmax_key_f32),
    one MAX all-reduce of B int64 values, then the key's index (q4_argmax_key_index).

The pages run their engine on one GPU (the rumik-oss-1 write-up, "A detour: the laptop engine on
an H100"); splitting the rows is the plain reading of spreading that GEMV over several GPUs.
Shards are whole 16-row tiles (the tiled layout's unit), their tile counts differing by at most one.
Collectives go through torch.distributed (NCCL on GPUs, gloo for the host-side tests); no peer
memory is read by any kernel.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import DecodeStepGraph, QuantizedMatrix

TILE = 16


def row_shards(N: int, P: int) -> list[tuple[int, int]]:
    """Rows [start, stop) of each of P ranks: whole 16-row tiles, rank r taking tiles
    [r T / P, (r + 1) T / P) of the T = ceil(N / 16); every rank gets at least one tile."""
    if N < 1 or P < 1:
        raise ValueError("N and P must be positive")
    T = (N + TILE - 1) // TILE
    if T < P:
        raise ValueError(f"{N} rows are {T} tiles of {TILE}: too few for {P} ranks")
    out = []
    for r in range(P):
        t0, t1 = r * T // P, (r + 1) * T // P
        out.append((TILE * t0, min(N, TILE * t1)))
    return out


@dataclass
class ShardLayout:
    """Where each matrix's local rows sit in the flat exchange buffer of every rank.

    For matrix i: shards[i] = the P row ranges, rmax[i] = the largest of them, and its local
    output [B, rows_r] occupies elements off[i] .. off[i] + B * rows_r of the buffer (the slot is
    B * rmax[i] long on every rank, so rank r's rows of matrix i sit at r * per_rank + off[i] after
    the all-gather)."""
    P: int
    B: int
    shards: list
    rmax: list
    off: list
    per_rank: int

    @classmethod
    def build(cls, Ns, P: int, B: int) -> "ShardLayout":
        shards = [row_shards(int(N), P) for N in Ns]
        rmax = [max(e - s for s, e in sh) for sh in shards]
        off, o = [], 0
        for r in rmax:
            off.append(o)
            o += -(-B * r // 4) * 4          # every slot starts 16-byte aligned (fp32)
        return cls(P, B, shards, rmax, off, o)

    def local_view(self, buf: torch.Tensor, i: int, rank: int) -> torch.Tensor:
        """Rank `rank`'s output of matrix i ([B, rows]) inside its own exchange buffer."""
        s, e = self.shards[i][rank]
        return buf[self.off[i]:self.off[i] + self.B * (e - s)].view(self.B, e - s)

    def assemble(self, gathered: torch.Tensor, i: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """Full output [B, N_i] of matrix i from the all-gathered buffer [P * per_rank]."""
        N = self.shards[i][-1][1]
        if out is None:
            out = torch.empty((self.B, N), dtype=gathered.dtype, device=gathered.device)
        g = gathered.view(self.P, self.per_rank)
        for r, (s, e) in enumerate(self.shards[i]):
            out[:, s:e].copy_(g[r, self.off[i]:self.off[i] + self.B * (e - s)].view(self.B, e - s))
        return out


def all_gather_outputs(send: torch.Tensor, recv: torch.Tensor, group=None) -> None:
    """One all-gather of every rank's flat exchange buffer (recv = P * send, rank-major)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_gather_into_tensor(recv, send, group=group)
    else:
        recv.copy_(send)


def all_reduce_keys(keys: torch.Tensor, group=None) -> None:
    """Largest argmax key per batch row over every rank, in place (one MAX all-reduce of int64)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(keys, op=dist.ReduceOp.MAX, group=group)


class ShardedStep:
    """Rank `rank` of `world`: its rows of every matrix of an independent decode-step list (two or
    more matrices, so that the tile kernel runs and every row is bit-identical to one GPU), run as
    one CUDA graph (activation prep, one tile-kernel launch over the local rows, and -- when `head`
    names the output head -- the head slice's argmax key), followed by the exchange.

    ``packed`` holds each matrix's canonical host arrays (codes, scales, mins) as q4_pack_host
    writes them; only this rank's rows are copied to its GPU.  Write the (replicated) activations
    into ``self.graph.X[i]`` and call ``step()``; then ``output(i)`` is the full [B, N_i] output
    (when ``gather``) and ``self.idx`` the head's argmax per batch row."""

    def __init__(self, packed, B: int, rank: int | None = None, world: int | None = None, group=None,
                 head: int | None = None, gather: bool = True, device="cuda"):
        import torch.distributed as dist
        dist_on = dist.is_available() and dist.is_initialized()
        self.rank = rank if rank is not None else (dist.get_rank(group) if dist_on else 0)
        self.world = world if world is not None else (dist.get_world_size(group) if dist_on else 1)
        self.group, self.head, self.gather, self.B = group, head, gather, B
        self.layout = ShardLayout.build([c.shape[0] for c, _, _ in packed], self.world, B)
        self.mats = []
        for i, (c, s, m) in enumerate(packed):
            a, e = self.layout.shards[i][self.rank]
            self.mats.append(QuantizedMatrix.from_packed(c[a:e], s[a:e], m[a:e], device=device,
                                                         keep_canonical=False))
        self.send = torch.zeros((self.layout.per_rank,), dtype=torch.float32, device=device)
        self.recv = torch.zeros((self.world * self.layout.per_rank,), dtype=torch.float32, device=device) \
            if gather else None
        Y = [self.layout.local_view(self.send, i, self.rank) for i in range(len(self.mats))]
        self.keys = torch.zeros((B,), dtype=torch.int64, device=device)
        self.idx = torch.zeros((B,), dtype=torch.int32, device=device)
        after = None
        if head is not None:
            from . import argmax_keys
            base = self.layout.shards[head][self.rank][0]
            after = lambda st: argmax_keys(Y[head], base, self.keys, stream=st)
        self.graph = DecodeStepGraph(self.mats, B, Y=Y, device=device, after=after)

    def step(self) -> None:
        """One decode step: the local graph, then the output all-gather and the argmax all-reduce."""
        from . import argmax_key_index
        self.graph.replay()
        if self.gather:
            all_gather_outputs(self.send, self.recv, self.group)
        if self.head is not None:
            all_reduce_keys(self.keys, self.group)
            argmax_key_index(self.keys, self.idx)

    def output(self, i: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """The full output [B, N_i] of matrix i after step() (needs gather=True)."""
        if self.recv is None:
            raise RuntimeError("built with gather=False: only the local rows exist")
        return self.layout.assemble(self.recv, i, out)
