"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks (spawned processes,
rendezvous on 127.0.0.1) reduce their timed regions to the slowest one, and the whole-job
throughput counts every rank's copy of the workload."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t = bench.max_over_ranks(1.0 + 0.5 * rank)
        dist.barrier()
        out.put((rank, t, bench.job_tokens_per_s(world, 16384, 10, t)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, t, v in res:
        assert t == pytest.approx(1.5)
        assert v == pytest.approx(2 * 16384 * 10 / 1.5)


def test_single_process_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.job_tokens_per_s(1, 16384, 50, 0.01) == pytest.approx(16384 * 50 / 0.01)
