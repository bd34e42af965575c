"""Host logic of `bench.py --gpus N` (N independent replicas, one per rank): the job's time is the
max over ranks.  Two gloo ranks on the CPU; no GPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, _ = bench.dist_setup()
    m = bench.dist_max(1.5 + rank)
    dist.barrier()
    out[rank] = (ws, r, m)
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == (2, 0, 2.5) and res[1] == (2, 1, 2.5)


def test_dist_max_is_identity_without_process_group():
    import bench
    assert bench.dist_max(3.25) == 3.25
