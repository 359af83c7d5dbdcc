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


def test_roofline_accounting():
    """The algorithmic bytes bench.py divides by: per-stage formulas from the workload's
    shapes and budgets; the fused launch (the whole path) on the each-byte-once basis
    of the headline HBM fraction, with the sum of its four steps kept as phase_bytes."""
    import numpy as np
    import bench
    import synth
    wl = synth.BY_NAME["long_32L_8kv_32q_d128_n131072_pyramid10"]
    L, H, d, n = wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.seq_lengths()[0]
    budgets = np.full((1, L, H), 13107, dtype=np.int32)
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0}
    kv_bytes = L * H * n * d * 2 * 2
    q_bytes = L * wl.num_q_heads * wl.window * d * 2
    att = bench.stage_roofline("attention", 1.0, wl, budgets, peaks)
    assert att["algorithmic_bytes"] == kv_bytes + q_bytes
    res = bench.stage_roofline("rescore", 1.0, wl, budgets, peaks)
    assert res["algorithmic_bytes"] == kv_bytes + q_bytes + L * H * n * 4
    # achieved GB/s = bytes / time; frac against the given peak
    assert abs(att["achieved"] - att["algorithmic_bytes"] / 1e-3 / 1e9) < 1e-6 * att["achieved"]
    assert abs(att["frac"] - att["achieved"] / 6000.0) < 1e-12
    fused = bench.stage_roofline("fused", 1.0, wl, budgets, peaks)
    parts = [bench.stage_roofline(s, 1.0, wl, budgets, peaks)
             for s in ("attention", "rescore", "select", "compact")]
    rows = int(budgets.sum())
    once = kv_bytes + q_bytes + rows * (2 * d * 2 + 4) + 8 * (L * H + 1)
    assert fused["algorithmic_bytes"] == once == bench.algorithmic_bytes(wl, budgets)
    assert fused["phase_bytes"] == sum(p["algorithmic_bytes"] for p in parts)
    assert fused["tensor"]["algorithmic_flops"] == \
        att["tensor"]["algorithmic_flops"] + res["tensor"]["algorithmic_flops"]
    # the attention sum reads K only
    att2 = bench.stage_roofline("attention", 1.0, wl, budgets, peaks, rule=2)
    assert att2["algorithmic_bytes"] == kv_bytes // 2 + q_bytes
