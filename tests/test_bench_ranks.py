"""The multi-GPU contract of bench.py on the host: independent replicas, one per rank,
with the step time taken as the slowest rank's and the whole-job throughput as all
ranks' tokens over it.  Run as two gloo processes on the CPU (the data path has no
collective; this max over ranks is the bench's only exchange)."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.5, 2.25][rank]  # each rank's own step time
    ms_max = bench.max_over_ranks(ms, world, "cpu")
    out[rank] = (ms_max, bench.job_throughput(8192, world, ms_max))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_tokens_add_up():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as man:
        out = man.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms_max, value = res[r]
        assert ms_max == 3.5
        assert value == pytest.approx(8192 * 2 / 3.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.job_throughput(1000, 1, 2.0) == pytest.approx(5e5)
