"""Host-side logic of bench.py's multi-GPU path, run as two gloo ranks on CPU.

Each rank is an independent replica of the layer (no data-path exchange);
the job's value is all ranks' work over the slowest rank's time.  These
ranks time nothing on a GPU: they feed fixed per-rank times through the same
aggregation bench.py uses.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [400.0, 500.0][rank]          # rank 1 is the slow one
    value, per = bench.job_throughput(local_ms, 100, 5.0e11, world)
    bench.barrier(world)
    out[rank] = (value, per)
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_slowest_rank():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        value, per = out[r]
        assert per == pytest.approx(5.0)                      # 500 ms / 100 steps
        assert value == pytest.approx(2 * 5.0e11 / 5e-3 / 1e12)  # both ranks' work


def test_single_rank_needs_no_process_group():
    import bench
    value, per = bench.job_throughput(200.0, 100, 5.0e11, 1)
    assert per == pytest.approx(2.0)
    assert value == pytest.approx(5.0e11 / 2e-3 / 1e12)
