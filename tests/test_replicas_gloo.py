"""The multi-GPU mode of bench.py on CPU: independent replicas (no collective on the data path),
timed together with a barrier, the job's time being the slowest rank's.  Two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    bench._PG = True
    try:
        assert bench.dist_env() == (world, rank, rank)
        bench.barrier()
        ms = bench.max_over_ranks(1.5 + rank)   # rank 1 is the slower replica
        value = bench.job_tokens_per_s(8192, world, ms)
        q.put((rank, ms, value))
    finally:
        torch.distributed.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == pytest.approx(2.5)                      # max over ranks
        assert value == pytest.approx(8192 * 2 / 2.5e-3)     # whole-job tokens over that time


def test_single_process_needs_no_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_tokens_per_s(100, 1, 1.0) == pytest.approx(1e5)
