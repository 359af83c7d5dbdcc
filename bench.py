#!/usr/bin/env python
"""Throughput of the KV-cache eviction hot path on one GB300 (or N, weak scaling).

One step = kv_score (window attention + rescoring) + kv_select_topk +
kv_compact over the whole workload, inputs resident in HBM.  The default
workload is the long-context configuration at n = 131072 (32 layers, 8 KV
heads, 32 query heads, d = 128, w = 64, pyramid budgets averaging 10%).

Prints one JSON line.  `value` counts unit-tokens (tokens x layers x KV heads,
each scored, selected and compacted) per second over all ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--score-rule dropkv|squared|attn_sum] [--pool KERNEL] [--head-budgets]
                  [--block-layers N]

--score-rule picks what kv_score sums (the DropKV removal score by default;
its squared form; the SnapKV/PyramidKV attention sum) and --pool adds the
max pooling of the scores before selection (kernel 11 on the DropKV page, 13
on the BellowsKV blog); --head-budgets redistributes each layer's budget over
its heads from the scores (AdaDropKV) before selection.  All default to the
DropKV step without pooling and with the policy's per-layer budgets.
--block-layers N runs block eviction (BellowsKV): one selection per block of N
layers from the scores summed over the block, pooled with --pool, keeping the
sinks, the window and the workload's budget ratio of the rest, then every
layer and head compacted with its block's tokens.

--impl reference times the fp64 CPU oracle (the only reference arm: the
pages ship no code) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV tokens scored+selected+compacted/s at n=128K; achieved HBM GB/s vs GB300 peak"
UNIT = "unit-tokens/s"
DEFAULT_WORKLOAD = "long_32L_8kv_32q_d128_n131072_pyramid10"
SCORE_RULES = {"dropkv": 0, "squared": 1, "attn_sum": 2}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (0: enough for about 2 s of timed work, at least 20)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=21)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-units", type=int, default=0, help="oracle sample size (0: one per core)")
    ap.add_argument("--score-rule", choices=sorted(SCORE_RULES), default="dropkv")
    ap.add_argument("--pool", type=int, default=1, help="max-pool kernel before selection (1: none)")
    ap.add_argument("--head-budgets", action="store_true",
                    help="per-head budgets from the scores before selection")
    ap.add_argument("--fused", action="store_true",
                    help="score, select and compaction as one cooperative launch "
                         "(kv_evict_fused); no pooling, per-head budgets or blocks")
    ap.add_argument("--block-layers", type=int, default=0,
                    help="block eviction over blocks of this many layers (0: off)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step (every call of the path) in a CUDA graph after the "
                         "warm-up and time its replays; stage times come from eager steps")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------
def kv_cache_bytes(layers, kv_heads, head_dim, tokens, bytes_per_elem=2):
    """K and V bytes of a cache: 2 (K,V) x bytes x L x H x D x N (PyramidKV guide,
    "The Long-Context Memory Wall")."""
    return 2 * bytes_per_elem * layers * kv_heads * head_dim * tokens


def algorithmic_bytes(wl, budgets):
    """Bytes the path must move at least once: K+V read, the window queries read,
    the compacted K/V and int32 indices written, the offsets table."""
    L, H, d = wl.num_layers, wl.num_kv_heads, wl.head_dim
    n_tot = sum(wl.seq_lengths())
    kv_read = kv_cache_bytes(L, H, d, n_tot)
    q_read = wl.num_requests * L * wl.num_q_heads * wl.window * d * 2
    rows = int(np.asarray(budgets).sum())
    out = rows * (2 * d * 2 + 4)
    offsets = 8 * (wl.num_units + 1)
    return kv_read + q_read + out + offsets


def pass_pairs(wl):
    """(row, key) pairs one scoring pass visits: each window row sees keys 0..pos."""
    G, w = wl.group, wl.window
    tot = 0
    for n in wl.seq_lengths():
        per_unit = G * sum(n - w + t + 1 for t in range(w))
        tot += per_unit * wl.num_layers * wl.num_kv_heads
    return tot


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle on host cores
# ---------------------------------------------------------------------------
def oracle_inputs(wl, budgets, units, rows_per_unit=None):
    """Host-regenerated inputs of `units` for the oracle (not timed)."""
    import synth
    outl = synth.outlier_channels(wl)
    hp = synth.heavy_positions(wl)
    qh = synth.q_window(wl)
    hv = synth.heavy_rows(wl, qh) if wl.num_heavy else None
    G, R = wl.group, wl.rows
    rows = rows_per_unit or R
    inputs = []
    for u in units:
        r, l, h = wl.unit_coords(u)
        q = qh[r, l, h * G:(h + 1) * G].reshape(R, wl.head_dim)[:rows]
        k, v = synth.kv_unit(wl, r, l, h, outl=outl, heavy_pos=hp, heavy_vec=hv)
        inputs.append((q, k, v, int(budgets.reshape(-1)[u])))
    return inputs


def oracle_time(wl, inputs, threads, rule=0, pool=1):
    """Times the oracle (score under `rule`, pooling if pool > 1, select, gather) over
    prepared inputs, one unit per thread; returns (seconds, unit-token equivalents).
    An input with fewer than G*w query rows counts as that fraction of a unit."""
    import oracle
    w = wl.window

    def one(args):
        q, k, v, b = args
        S = oracle.unit_scores_rule(q, k, v, max(1, q.shape[0] // w), w, rule)
        if pool > 1:
            S = oracle.pool_unit(S, w, pool)
        idx = oracle.select(S, w, wl.num_sinks, b)
        oracle.compact(k, v, idx)
        return k.shape[0] * q.shape[0] / wl.rows

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        work = sum(ex.map(one, inputs))
    return time.perf_counter() - t0, work


def run_reference(args, wl, budgets):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import synth
    cores = os.cpu_count() or 1
    units = list(range(min(cores, wl.num_units)))
    rows = wl.window   # one query head's window rows per unit per step
    inputs = oracle_inputs(wl, budgets, units, rows_per_unit=rows)
    times = []
    work = 0.0
    rule = SCORE_RULES[args.score_rule]
    for s in range(args.warmup + args.steps):
        dt, work = oracle_time(wl, inputs, cores, rule, args.pool)
        if s >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    value = work / t
    sample = ("%d units x %d of %d window rows (one query head), full n=%d, per step; "
              "work counted as %.4f units" % (len(units), rows, wl.rows, wl.seq_lengths()[0],
                                              work / wl.seq_lengths()[0]))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config_tag(wl, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
# Kernels of one step and how many launches each makes (the timed region
# launches only these).
STAGES = ["attention", "rescore", "blocks", "pool", "heads", "select", "compact"]
# attention: plan_kernel, attn_tc_kernel, attn_merge_kernel; rescore: plan_kernel,
# rescore_tc_kernel and, when the window rows span more than one 128-row chunk,
# chunk_sum_kernel.  The two plan_kernel launches happen only when the requests
# form more than 32 runs of equal length (otherwise the work items decode from
# tables passed as kernel parameters).
# pool: pool_kernel, only with --pool > 1; heads: head_budget_kernel, only with
# --head-budgets.
# heads launches a memset and six kernels; blocks (block_sum_kernel) only with
# --block-layers.
LAUNCHES_PER_STEP = {"attention": 3, "rescore": 2, "blocks": 1, "pool": 1, "heads": 6,
                     "select": 1, "compact": 1}
STAGE_KERNELS = {"attention": "attn_tc_kernel", "rescore": "rescore_tc_kernel",
                 "blocks": "block_sum_kernel", "pool": "pool_kernel", "heads": "hb_hist_kernel",
                 "select": "select_kernel", "compact": "compact_range_kernel"}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a stage's
# kernel at full size, keyed by (workload, score rule, pool kernel, fused): one ncu
# launch of a reduced copy of the workload (the same per-unit shapes, fewer units)
# scaled by the ratio of units.  Each entry records the kernel sources it was
# measured on ("src": kernel_source_hash() at capture time), the reduced case and
# the scale factor; bench reports traffic as null once the sources differ.
TRAFFIC = {
    ("long_32L_8kv_32q_d128_n131072_pyramid10", "dropkv", 1, False): {
        "src": "42267627bf73f97c", "case": "long_2L_2kv_8q_d128_n131072_pyramid10", "scale": 64,
        "bytes": {"attn_tc_kernel": 17546493952, "rescore_tc_kernel": 17584996352}},
    ("llama8b_32L_8kv_32q_d128_n32768", "dropkv", 1, False): {
        "src": "42267627bf73f97c", "case": "llama8b_2L_8kv_32q_d128_n32768", "scale": 16,
        "bytes": {"attn_tc_kernel": 4389621760, "rescore_tc_kernel": 4383350784}},
    ("qwen7b_28L_4kv_28q_d128_n131072_ripple5", "dropkv", 1, False): {
        "src": "42267627bf73f97c", "case": "qwen7b_2L_2kv_14q_d128_n131072_ripple5", "scale": 28,
        "bytes": {"attn_tc_kernel": 8184501248, "rescore_tc_kernel": 7831118848}},
    ("ragged8_mistral7b_32L_8kv_32q_d128_n16k-128k", "dropkv", 1, False): {
        "src": "42267627bf73f97c", "case": "ragged8_mistral7b_2L_2kv_8q_d128_n16k-128k",
        "scale": 64,
        "bytes": {"attn_tc_kernel": 91530002432, "rescore_tc_kernel": 88923734016}},
}


def kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) of the CUDA sources of the library."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_eviction_split_gb300", "csrc")
    for path in sorted(glob.glob(os.path.join(csrc, "*.cu")) +
                       glob.glob(os.path.join(csrc, "*.cuh"))):
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(key, kernel):
    """(bytes per launch, provenance) of `kernel`, or (None, reason)."""
    entry = TRAFFIC.get(key)
    if entry is None or kernel not in entry["bytes"]:
        return None, "no ncu capture for this workload and kernel"
    if entry["src"] != kernel_source_hash():
        return None, "kernel sources changed since the ncu capture (%s)" % entry["src"]
    return entry["bytes"][kernel], "ncu, %s, x%g" % (entry["case"], entry["scale"])


def stage_kernel(stage, rule, blk=0):
    if stage == "attention" and rule == SCORE_RULES["attn_sum"]:
        return "attn_stats_kernel"
    if stage == "compact" and blk:
        return "compact_kernel"      # the block-eviction form
    return STAGE_KERNELS[stage]


def product_budgets(kv, wl):
    import synth
    L, H = wl.num_layers, wl.num_kv_heads
    prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
    rows = []
    for B in wl.mean_budgets():
        if wl.budget_policy == "uniform":
            bl = kv.kv_budgets_uniform(L, B)
        elif wl.budget_policy == "pyramid":
            bl = kv.kv_budgets_pyramid(L, B, wl.pyramid_max, wl.pyramid_min)
        else:
            bl = kv.kv_budgets_ripple(L, B, prof, wl.ripple_beta)
        rows.append(np.repeat(np.asarray(bl, np.int32)[:, None], H, axis=1))
    return np.asarray(rows, dtype=np.int32)


def bench_config_tag(wl, args):
    tag = {"workload": wl.name}
    if getattr(args, "fused", False):
        tag["launch"] = "fused: one cooperative kernel per step"
    if getattr(args, "graph", False):
        tag["graph"] = "one step captured in a CUDA graph, replayed per timed step"
    if args.score_rule != "dropkv" or args.pool > 1 or args.head_budgets or args.block_layers:
        tag.update(score_rule=args.score_rule, pool_kernel=args.pool,
                   head_budgets=bool(args.head_budgets))
    if args.block_layers:
        tag.update(block_layers=args.block_layers, keep_fraction=wl.budget_ratio)
    return tag


def stage_roofline(stage, ms, wl, budgets, peaks, rule=0, blk=1):
    """Roofline of one stage's kernel from its algorithmic bytes (and, for the two
    scoring passes, their algorithmic tensor flops: two d-long dot products per
    (window row, visible key) pair each, one for the attention sum, which needs
    only q.k).  The attention sum needs no V: its passes read K only."""
    if stage == "fused":
        # the fused kernel is the whole path: its roofline counts every byte once
        # (K+V, the window queries, the kept rows and indices, the offsets), the
        # headline basis; the sum of its phases' own bytes (K+V twice, the scores
        # written and read) is kept beside it as phase_bytes
        parts = [stage_roofline(s, ms, wl, budgets, peaks, rule, blk)
                 for s in ("attention", "rescore", "select", "compact")]
        nbytes = algorithmic_bytes(wl, budgets)
        flops = sum(p["tensor"]["algorithmic_flops"] for p in parts if "tensor" in p)
        achieved = nbytes / (ms * 1e-3) / 1e9
        tpeak = peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"]
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "algorithmic_bytes": nbytes,
                "phase_bytes": sum(p["algorithmic_bytes"] for p in parts),
                "tensor": {"algorithmic_flops": flops,
                           "achieved_tflops": flops / (ms * 1e-3) / 1e12, "peak_tflops": tpeak,
                           "frac": flops / (ms * 1e-3) / 1e12 / tpeak}}
    d = wl.head_dim
    units = wl.num_units
    n_tot = sum(wl.seq_lengths())
    L, H = wl.num_layers, wl.num_kv_heads
    rows = int(np.asarray(budgets).sum())
    if stage in ("pool", "select") and blk > 1:
        keys_div = H * blk                     # block problem: one score row per block
    else:
        keys_div = 1
    kv = kv_cache_bytes(L, H, d, n_tot)
    q = wl.num_requests * L * wl.num_q_heads * wl.window * d * 2
    keys = n_tot * L * H
    kv_pass = kv // 2 if rule == SCORE_RULES["attn_sum"] else kv
    if stage == "attention":
        nbytes = kv_pass + q                   # K, V and the window queries, once
    elif stage == "rescore":
        nbytes = kv_pass + q + keys * 4        # ... plus one fp32 score per key
    elif stage == "pool":
        nbytes = keys // keys_div * 4 * 2      # every score read and written once
    elif stage == "heads":
        nbytes = keys * 4 + units * (4 + 8) * 2   # scores read once; budgets, offsets
    elif stage == "blocks":
        nbytes = keys * 4 + keys * 4 // (H * blk)  # scores read once, block scores written
    elif stage == "select":
        nbytes = keys // keys_div * 4 + rows // (H * blk if blk > 1 else 1) * 4 + \
            8 * (units // (H * blk if blk > 1 else 1) + 1) * 2
    else:
        nbytes = rows * (2 * d * 2) * 2 + rows * 4 + 8 * (units + 1)
    achieved = nbytes / (ms * 1e-3) / 1e9
    out = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": achieved / peaks["hbm_gbs"], "algorithmic_bytes": nbytes}
    if stage in ("attention", "rescore"):
        flops = pass_pairs(wl) * (2 if rule == SCORE_RULES["attn_sum"] else 4) * d
        tpeak = peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"]
        out["tensor"] = {"algorithmic_flops": flops, "achieved_tflops": flops / (ms * 1e-3) / 1e12,
                         "peak_tflops": tpeak, "frac": flops / (ms * 1e-3) / 1e12 / tpeak}
    return out


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (the timed region of the slowest rank);
    `value` itself when there is no process group."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second: every rank scores its own copy of the
    workload (weak scaling), timed by the slowest rank."""
    return units_per_rank * world / (ms_per_step * 1e-3)


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def main(argv=None):
    args = parse_args(argv)
    import synth
    wl = synth.BY_NAME[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
        return run_reference(args, wl, oracle.segment_budgets(wl, prof))

    import torch
    import kv_cache_eviction_split_gb300 as kv
    from synth.device import DeviceWorkload
    kv.load()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()

    budgets = product_budgets(kv, wl)
    dw = DeviceWorkload(wl, device=dev)
    rule = SCORE_RULES[args.score_rule]
    pool = args.pool
    heads = args.head_budgets
    blk = args.block_layers
    if blk and heads:
        raise SystemExit("--block-layers and --head-budgets do not combine")
    fused = args.fused
    if fused and (blk or heads or pool > 1):
        raise SystemExit("--fused takes neither --pool, --head-budgets nor --block-layers")
    stage_names = ["fused"] if fused else STAGES
    prob = kv.Problem.for_workload(wl, device=dev, score_rule=rule, pool_kernel=pool,
                                   head_budgets=heads)
    bufs = kv.Buffers(prob, budgets)
    # a graph is captured on a side stream; everything else then runs there too
    stream = torch.cuda.Stream(dev) if args.graph else torch.cuda.current_stream(dev)
    if args.graph:
        stream.wait_stream(torch.cuda.current_stream(dev))
    ranked = bufs.pooled if pool > 1 else bufs.scores
    bb = None
    if blk:
        bb = kv.BlockBuffers(prob, blk, wl.budget_ratio, pool_kernel=pool)
        ranked = bb.pooled if pool > 1 else bb.block_scores
        # rows kept per unit: every unit keeps its block's budget
        budgets = np.repeat(np.repeat(bb.block_budgets_host.reshape(wl.num_requests, -1), blk,
                                      axis=1)[:, :, None], wl.num_kv_heads, axis=2)
    sel_b, sel_o = (bufs.head_budgets, bufs.head_offsets) if heads else (bufs.budgets,
                                                                         bufs.offsets)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if fused:
            kv.kv_evict_fused(prob, dw.q, dw.k, dw.v, bufs.budgets, bufs.offsets,
                              bufs.total_rows, bufs.scores, bufs.sel, bufs.k_out, bufs.v_out,
                              bufs.score_ws, stream)
            if ev is not None:
                ev[1].record(stream)
            return
        kv.kv_score_attention(prob, dw.q, dw.k, dw.v, bufs.score_ws, stream)
        if ev is not None:
            ev[1].record(stream)
        kv.kv_score_rescore(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws, stream)
        if ev is not None:
            ev[2].record(stream)
        if blk:
            kv.kv_block_scores(prob, blk, bufs.scores, bb.block_scores, stream)
        if ev is not None:
            ev[3].record(stream)
        if pool > 1 and blk:
            kv.kv_pool_scores(bb.bprob, pool, bb.block_scores, bb.pooled, stream)
        elif pool > 1:
            kv.kv_pool_scores(prob, pool, bufs.scores, bufs.pooled, stream)
        if ev is not None:
            ev[4].record(stream)
        if heads:
            kv.kv_head_budgets(prob, ranked, bufs.budgets, bufs.offsets, bufs.head_budgets,
                               bufs.head_offsets, bufs.select_ws, stream)
        if ev is not None:
            ev[5].record(stream)
        if blk:
            kv.kv_select_topk(bb.bprob, ranked, bb.block_budgets, bb.block_offsets, bb.sel,
                              bb.select_ws, stream)
        else:
            kv.kv_select_topk(prob, ranked, sel_b, sel_o, bufs.sel, bufs.select_ws, stream)
        if ev is not None:
            ev[6].record(stream)
        if blk:
            kv.kv_compact_blocks(prob, blk, dw.k, dw.v, bb.sel, bb.block_offsets,
                                 bb.unit_offsets, bb.total_rows, bb.k_out, bb.v_out, stream)
        else:
            kv.kv_compact(prob, dw.k, dw.v, bufs.sel, sel_o, bufs.total_rows, bufs.k_out,
                          bufs.v_out, stream)
        if ev is not None:
            ev[7].record(stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    # Inputs smaller than a few L2s (the tiny configuration) would stay in L2 from one
    # step to the next: then L2 is flushed (a 512 MB buffer written) before every
    # step, outside its events, and each step is timed alone.
    n_tot = sum(wl.seq_lengths())
    kv_in = kv_cache_bytes(wl.num_layers, wl.num_kv_heads, wl.head_dim, n_tot)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if kv_in < 4 * l2_bytes \
        else None
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    t_w0 = time.perf_counter()
    for _ in range(max(args.warmup, 0)):
        if flush is not None:
            flush.zero_()
        step()
    barrier()
    if args.steps <= 0:
        per = (time.perf_counter() - t_w0) / max(args.warmup, 1)
        args.steps = int(min(20000 if flush is not None else 2000,
                             max(20, math.ceil(2.0 / max(per, 1e-4)))))
    # per-stage events on every step when each step is timed alone, else on the
    # first 200 timed steps (the step time itself spans all of them)
    staged = args.steps if flush is not None else min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stage_names) + 1)]
           for _ in range(staged)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    graph = None
    if args.graph:
        # stage times from eager steps (a replay records no per-stage events), then
        # one step captured and its replays timed
        staged = min(args.steps, 50)
        evs = evs[:staged]
        for i in range(staged):
            if flush is not None:
                flush.zero_()
            step(evs[i])
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        step_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                    for _ in range(args.steps)] if flush is not None else None
        barrier()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                if flush is not None:
                    flush.zero_()
                    step_evs[i][0].record(stream)
                graph.replay()
                if flush is not None:
                    step_evs[i][1].record(stream)
            t_end.record(stream)
    else:
        t_start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            step(evs[i] if i < staged else None)
        t_end.record(stream)
    barrier()
    clocks = sampler.stop()
    if flush is not None:
        total_ms = sum((step_evs[i][0].elapsed_time(step_evs[i][1]) for i in range(args.steps))
                       if graph is not None else
                       (evs[i][0].elapsed_time(evs[i][-1]) for i in range(args.steps)))
    else:
        total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, dist, dev)
    st = (kv.kv_check_status(bufs.score_ws, stream),
          kv.kv_check_status(bb.select_ws if blk else bufs.select_ws, stream))
    if st != (0, 0):
        raise SystemExit("device status after the timed region: %s" % (st,))
    stage_ms = {s: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1])
                                   for i in range(staged)) for j, s in enumerate(stage_names)}
    ms_per_step = total_ms / args.steps
    unit_tokens = n_tot * wl.num_layers * wl.num_kv_heads
    value = whole_job_rate(unit_tokens, world, ms_per_step)
    alg_bytes = algorithmic_bytes(wl, budgets)
    hbm_gbs = alg_bytes / (ms_per_step * 1e-3) / 1e9

    stages = ["fused"] if fused else \
        [s for s in STAGES if (s != "pool" or pool > 1) and (s != "heads" or heads)
         and (s != "blocks" or blk)]
    for s in list(stage_ms):
        if s not in stages:
            stage_ms.pop(s)
    dominant = max(stages, key=lambda s: stage_ms[s])
    roof = stage_roofline(dominant, stage_ms[dominant], wl, budgets, peaks, rule, blk)
    kernel = "fused_kernel" if fused else stage_kernel(dominant, rule, blk)
    if heads or blk:
        traffic, traffic_src = None, "no ncu capture for per-head budgets or block eviction"
    else:
        traffic, traffic_src = measured_traffic((wl.name, args.score_rule, pool, fused), kernel)
    roof.update({"kernel": kernel, "peak_source": peak_src,
                 "traffic": traffic, "traffic_source": traffic_src,
                 "kernel_source_hash": kernel_source_hash(), "stage_ms": stage_ms[dominant],
                 "all_stages": {s: stage_roofline(s, stage_ms[s], wl, budgets, peaks,
                                                  rule, blk)["frac"] for s in stages}})

    lens = wl.seq_lengths()
    runs = 1 + sum(1 for a, b in zip(lens, lens[1:]) if a != b)
    launches = (1 if fused else sum(LAUNCHES_PER_STEP[s] for s in stages)
                + (1 if wl.rows > 128 else 0) - (2 if runs <= 32 else 0))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {**bench_config_tag(wl, args), "layers": wl.num_layers,
                       "kv_heads": wl.num_kv_heads, "q_heads": wl.num_q_heads,
                       "head_dim": wl.head_dim, "n": wl.seq_lengths(), "window": wl.window,
                       "budget": "%s, mean %s tokens/head" % (wl.budget_policy,
                                                              wl.mean_budgets()),
                       "units": wl.num_units, "parallelism": "replicas x%d" % world,
                       "l2": ("flushed before every step (512 MB written outside the step's "
                              "events; each step timed alone): the K+V inputs (%.2f MB) fit "
                              "in L2" % (kv_in / 1e6)) if flush is not None else
                             "no flush: the K+V inputs (%.1f GB) exceed L2 every step"
                             % (kv_in / 1e9)},
            "seq_tokens_per_s": n_tot * world / (ms_per_step * 1e-3),
            "hbm": {"alg_bytes_per_step": alg_bytes, "achieved_gbs": hbm_gbs,
                    "peak_gbs": peaks["hbm_gbs"], "frac": hbm_gbs / peaks["hbm_gbs"],
                    "peak_source": peak_src},
            "stages_ms": stage_ms,
            "roofline": roof,
            "gpu_launches": args.steps * launches,
            "us_per_launch": ms_per_step * 1e3 / launches,
            "clocks": clocks}

    if not args.no_e2e:
        line["e2e"] = e2e_measure(args, kv, torch, wl, dw, prob, bufs, stream, unit_tokens * world,
                                  bb, budgets)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
        ob = oracle.segment_budgets(wl, prof)
        cores = os.cpu_count() or 1
        n_units = args.cpu_units or min(cores, 16, wl.num_units)
        thr = min(cores, n_units)
        dt, work = oracle_time(wl, oracle_inputs(wl, ob, list(range(n_units))), thr, rule, pool)
        line["cpu_baseline"] = {"value": work / dt, "unit": UNIT,
                                "cores": thr, "kind": "oracle",
                                "sample": "%d full units (of %d) of the same workload, one "
                                          "thread each, fp64 score (%s)%s + select + gather%s"
                                          % (n_units, wl.num_units, args.score_rule,
                                             " + pool %d" % pool if pool > 1 else "",
                                             " (per-head budgets and block selection are not "
                                             "in the sample: they need whole layers)"
                                             if heads or blk else "")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def e2e_measure(args, kv, torch, wl, dw, prob, bufs, stream, unit_tokens, bb=None, budgets=None):
    """Same metric through the public API with host buffers: pinned host Q/K/V
    copied in, scored, selected and compacted, the kept indices and packed K/V
    copied out.  The C entry point kv_evict_host (through kv.HostPipeline, which
    only allocates its buffers) overlaps the copies of one layer group with the
    work on another; block eviction copies everything in, then runs."""
    if bb is None:
        # inputs page-locked at their exact size, unless that would lock more than
        # 60% of the host's memory (then pageable: the copies no longer overlap)
        in_bytes = sum(t.numel() * t.element_size() for t in (dw.q, dw.k, dw.v))
        out_bytes = bufs.total_rows * (4 + 2 * wl.head_dim * 2)
        host_ram = host_memory_bytes()
        pin_inputs = in_bytes + out_bytes <= 0.6 * host_ram
        try:
            if pin_inputs:
                qh, kh, vh = (kv.PinnedTensor(tuple(t.shape), t.dtype) for t in (dw.q, dw.k, dw.v))
            else:
                qh, kh, vh = (torch.empty(t.shape, dtype=t.dtype) for t in (dw.q, dw.k, dw.v))
            qh.copy_(dw.q)
            kh.copy_(dw.k)
            vh.copy_(dw.v)
            pipe = kv.HostPipeline(prob, budgets, group_layers=4,
                                   fused=bool(getattr(args, "fused", False)))
        except RuntimeError as e:
            return {"value": None, "unit": UNIT, "error": "host allocation failed: %s" % e}
        pipe.run(qh, kh, vh)
        dt, spread = _timed_steps(args.e2e_steps, lambda: pipe.run(qh, kh, vh), torch)
        out = {"value": unit_tokens / dt, "unit": UNIT, "ms_per_step": dt * 1e3,
               "ms_per_step_min_max": spread,
               "h2d_bytes_per_step": pipe.h2d_bytes, "d2h_bytes_per_step": pipe.d2h_bytes,
               "steps": args.e2e_steps, "statistic": "median of per-step host wall times",
               "api": "kv_evict_host (C ABI), groups of 4 layers%s"
                      % (", fused launch per group" if pipe.fused else ""),
               "host_inputs": "pinned (cudaHostAlloc, exact size)" if pin_inputs else
                              "pageable: pinning %.0f GB would lock over 60%% of the %.0f GB "
                              "of host memory available" % ((in_bytes + out_bytes) / 1e9,
                                                            host_ram / 1e9)}
        del qh, kh, vh, pipe
        return out
    try:
        qh = torch.empty(dw.q.shape, dtype=dw.q.dtype, pin_memory=True)
        kh = torch.empty(dw.k.shape, dtype=dw.k.dtype, pin_memory=True)
        vh = torch.empty(dw.v.shape, dtype=dw.v.dtype, pin_memory=True)
        qh.copy_(dw.q)
        kh.copy_(dw.k)
        vh.copy_(dw.v)
        rows = bb.total_rows if bb is not None else bufs.total_rows
        selh = torch.empty(int(bb.block_offsets_host[-1]) if bb is not None else rows,
                           dtype=torch.int32, pin_memory=True)
        koh = torch.empty((rows, wl.head_dim), dtype=torch.bfloat16, pin_memory=True)
        voh = torch.empty_like(koh, pin_memory=True)
    except RuntimeError as e:
        return {"value": None, "unit": UNIT, "error": "pinned host allocation failed: %s" % e}

    def one():
        dw.q.copy_(qh, non_blocking=True)
        dw.k.copy_(kh, non_blocking=True)
        dw.v.copy_(vh, non_blocking=True)
        if bb is None:
            sel, ko, vo, _ = kv.evict(prob, dw.q, dw.k, dw.v, bufs, stream)
        else:
            kv.kv_score(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws, stream)
            sel, ko, vo, _ = kv.evict_blocks(prob, bufs.scores, dw.k, dw.v, bb, stream)
        selh.copy_(sel, non_blocking=True)
        koh.copy_(ko, non_blocking=True)
        voh.copy_(vo, non_blocking=True)

    one()
    torch.cuda.synchronize()
    dt, spread = _timed_steps(args.e2e_steps, one, torch)
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = selh.numel() * 4 + (koh.numel() + voh.numel()) * 2
    return {"value": unit_tokens / dt, "unit": UNIT, "ms_per_step": dt * 1e3,
            "ms_per_step_min_max": spread, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "statistic": "median of per-step host wall times"}


def host_memory_bytes() -> int:
    """Host memory this process may use: the smallest of MemAvailable, the cgroup
    limit (a container's can be far below the machine's RAM) and physical RAM."""
    cands = [os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")]
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    cands.append(int(ln.split()[1]) * 1024)
    except OSError:
        pass
    for path in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(path) as f:
                v = f.read().strip()
            if v.isdigit():
                cands.append(int(v))
        except OSError:
            pass
    return min(cands)


def _timed_steps(steps, fn, torch):
    """Host wall time of each of `steps` calls of fn (each ending in a device
    synchronisation): the median in seconds and [min, max] in ms.  The host link
    is shared with other work on the machine, so single steps can stall; the
    median keeps one stall from setting the number."""
    times = []
    for _ in range(max(1, steps)):
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    times.sort()
    n = len(times)
    med = times[n // 2] if n % 2 else 0.5 * (times[n // 2 - 1] + times[n // 2])
    return med, [round(times[0] * 1e3, 2), round(times[-1] * 1e3, 2)]


if __name__ == "__main__":
    sys.exit(main())
