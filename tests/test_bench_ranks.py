"""The benchmark's multi-rank host logic on CPU with two gloo ranks: times
are the slowest rank's, the status the worst rank's, the whole-job rate
counts every rank's units, and only rank 0 runs the reference arm."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
    status = -5 if rank == 1 else 0
    out = bench.reduce_over_ranks(times, status, "cpu")
    env = bench.dist_env()
    ref = bench.reference_arm(type("A", (), {"steps": 1, "warmup": 0})()) if rank == 1 else None
    q.put((rank, out, env, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_job():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (times, status), env, ref in results:
        assert times == [2.0, 5.0, 0.5]          # max over ranks, element by element
        assert status == -5                      # the worst status wins
        assert env == (2, rank, rank)
    assert results[1][3] is None                 # rank 1 does no reference-arm work


def test_weak_scaling_rate_counts_all_ranks():
    # 2 ranks x 1e12 FLOP each in 2 ms (the slowest rank) = 1000 TFLOP/s
    assert bench.weak_scaling_rate(1e12, 2, 2.0, 1e12) == pytest.approx(1000.0)
    assert bench.weak_scaling_rate(1e9, 1, 1.0, 1e9) == pytest.approx(1000.0)
