"""World-size-2 `gloo` run of the benchmark's multi-rank timing logic on CPU:
every rank sees the max of the per-rank event times, and the whole-job value
counts every rank's tokens over that max (weak scaling, no data-path
collective)."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.5][rank]
    m = bench.reduce_max_ms(ms, world, "cpu")
    v = bench.whole_job_value(131072, world, m)
    dist.barrier()
    out[rank] = (m, v)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0][0] == out[1][0] == 3.5
    assert out[0][1] == pytest.approx(2 * 131072 / 3.5e-3)
