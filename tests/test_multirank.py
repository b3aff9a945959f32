"""The multi-rank harness of bench.py on CPU: two gloo ranks (no GPU).

Every rank runs the whole per-token workload on its own GPU (tokens shard with
no exchange); the job's step time is the slowest rank's and the job value is
all ranks' bytes over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.0 + rank, 10.0 - rank]          # rank 0: (1, 10); rank 1: (2, 9)
    out = bench.reduce_max(ms, world)
    val = bench.job_value(world, 1_000_000_000, out[0])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out, val))


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out, val in res:
        assert out == [2.0, 10.0]
        assert val == pytest.approx(2 * 1e9 / 2e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max([3.5, 1.0], 1) == [3.5, 1.0]
    assert bench.job_value(1, 1_677_721_600, 0.25) == pytest.approx(6.7108864)
