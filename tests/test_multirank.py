"""The multi-rank harness of bench.py on CPU: two gloo ranks (no GPU).

The job's batch is split into contiguous token shards, one per rank, with no
exchange between them (every token's seam is independent); the job's step time
is the slowest rank's and the job value is all ranks' bytes over that time."""
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


def _shard_main(rank, world, port, q):
    # Each rank draws its shard of one 11-token batch through bench.py's own
    # workload code and runs the oracle on it; the shards are gathered over gloo.
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle as O
    T_total, H = 11, 64
    t0, t1 = bench.token_shard(T_total, rank, world)
    w = dict(T=t1 - t0, H=H, post=True, out="bf16", seed=1234)
    wl = bench.make_workload(w, "cpu", token_offset=t0, unique=4)
    h = wl["host"]
    o = O.seam(h["R"], h["Y"], h["post_prev"], h["comb_prev"], h["pre_prev"], h["fn"], h["bias"], h["alpha"],
               h["gamma"], wl["eps"])
    parts = [None] * world
    dist.all_gather_object(parts, (t0, t1, {k: o[k] for k in ("residual_out", "norm", "pre", "post", "comb")}))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, parts))


def test_two_rank_token_shards_reassemble_the_batch():
    import numpy as np

    import bench
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    parts = res[0][1]
    assert [(a, b) for a, b, _ in parts] == [(0, 6), (6, 11)]     # contiguous, uneven split
    # the whole batch on one rank: the same outputs, token for token
    w = dict(T=11, H=64, post=True, out="bf16", seed=1234)
    wl = bench.make_workload(w, "cpu", token_offset=0, unique=4)
    h = wl["host"]
    whole = O.seam(h["R"], h["Y"], h["post_prev"], h["comb_prev"], h["pre_prev"], h["fn"], h["bias"], h["alpha"],
                   h["gamma"], wl["eps"])
    for k in ("residual_out", "norm", "pre", "post", "comb"):
        got = np.concatenate([p[2][k] for p in parts], axis=0)
        assert np.array_equal(got, whole[k]), k
    # the shards differ from each other (the batch is not one replicated shard)
    assert not np.array_equal(parts[0][2]["norm"][:5], parts[1][2]["norm"][:5])


def test_token_shard_partitions_the_batch():
    import bench
    for T in (0, 1, 7, 16384, 16385):
        for world in (1, 2, 3, 8):
            spans = [bench.token_shard(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
