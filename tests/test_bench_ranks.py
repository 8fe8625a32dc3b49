"""bench.py's multi-GPU arithmetic, on the CPU with two gloo ranks: the run is replicas of the
same step (no data-path collective); the timed figure is the slowest rank's, and the value is the
bytes of every rank over that time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 1.0 + rank                       # rank 1 is the slower replica
    out[rank] = bench.max_over_ranks(ms, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 2.0 and out[1] == 2.0
    import bench
    # 870,872,832 bytes per replica, two replicas, 0.5 ms per step -> 3483.49 GB/s
    assert abs(bench.job_gbs(870872832, 2, 0.5) - 2 * 870872832 / 0.5e-3 / 1e9) < 1e-9
    assert bench.max_over_ranks(3.5, 1) == 3.5
