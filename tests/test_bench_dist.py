"""The benchmark's multi-rank logic on the CPU with two gloo ranks: the timed
region is the slowest rank's, the reported rate counts every rank's units, and
under the reference arm only rank 0 works."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        rate = bench.whole_job_rate(1000.0, world, ms)
        # the reference arm: ranks other than 0 leave at once, without work
        rc = bench.main(["--impl", "reference"]) if rank != 0 else 0
        out.put((rank, ms, rate, rc))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_units():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=5) for _ in procs)
    for rank, ms, rate, rc in res:
        assert ms == 15.0                      # max over ranks
        assert abs(rate - 2 * 1000.0 / 15e-3) < 1e-6
        assert rc == 0


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(500.0, 1, 2.0) == 250000.0
