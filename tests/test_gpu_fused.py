"""The fused path (kv_evict_fused: score, select and compaction in one cooperative
launch) against the three separate calls and against the fp64 oracle.

The fused kernel runs the same device code as kv_score, kv_select_topk and kv_compact,
so every output -- scores, kept indices, packed K and V -- must match theirs bit for
bit; parity.check_units then holds the fused outputs to the oracle directly.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu

SMALL = [
    synth.TINY,
    synth.small_variant(synth.LONG_128K, 5003),                       # G w = 256: two chunks
    synth.small_variant(synth.QWEN7B_128K, 10500, kv_heads=1),        # G w = 448: four chunks
    synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 4097, 2222]),
]
RULES = [0, oracle.RULE_DROPKV_SQUARED, oracle.RULE_ATTN_SUM]


def _same(a, b, what):
    """Bit-for-bit equality (floats compared as their integer bit patterns)."""
    import torch
    bits = {torch.float32: torch.int32, torch.bfloat16: torch.int16}
    assert a.shape == b.shape and a.dtype == b.dtype, what
    if a.dtype in bits:
        a, b = a.view(bits[a.dtype]), b.view(bits[b.dtype])
    assert torch.equal(a, b), what


def _compare(sep, fus):
    n = sep.bufs.total_rows
    _same(sep.bufs.scores, fus.bufs.scores, "scores")
    _same(sep.bufs.sel[:n], fus.bufs.sel[:n], "kept indices")
    _same(sep.bufs.k_out[:n].view(-1), fus.bufs.k_out[:n].view(-1), "packed K")
    _same(sep.bufs.v_out[:n].view(-1), fus.bufs.v_out[:n].view(-1), "packed V")


@pytest.mark.parametrize("rule", RULES, ids=["dropkv", "squared", "attn_sum"])
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_fused_matches_separate_calls_bitwise(cuda_lib, wl, rule):
    sep = parity.DeviceRun(cuda_lib, wl, score_rule=rule)
    fus = parity.DeviceRun(cuda_lib, wl, dw=sep.dw, score_rule=rule, fused=True)
    assert sep.status_score == 0 and sep.status_select == 0
    assert fus.status_score == 0
    _compare(sep, fus)


@pytest.mark.parametrize("wl", [w for w in __import__("tests.test_gpu_parity",
                                                      fromlist=["ROW_EDGES"]).ROW_EDGES],
                         ids=lambda w: w.name)
def test_fused_matches_separate_calls_row_edges(cuda_lib, wl):
    sep = parity.DeviceRun(cuda_lib, wl)
    fus = parity.DeviceRun(cuda_lib, wl, dw=sep.dw, fused=True)
    assert sep.status_score == 0 and fus.status_score == 0
    _compare(sep, fus)


@pytest.mark.parametrize("wl", SMALL[1:], ids=lambda w: w.name)
def test_fused_against_oracle_all_units(cuda_lib, wl):
    run = parity.DeviceRun(cuda_lib, wl, fused=True)
    assert run.status_score == 0
    res = parity.check_units(run, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL


@pytest.mark.parametrize("wl,count", [(synth.LLAMA8B_32K, 1), (synth.LONG_128K, 2),
                                      (synth.QWEN7B_128K, 1), (synth.RAGGED_MISTRAL, 1)],
                         ids=lambda x: getattr(x, "name", str(x)))
def test_fused_full_size(cuda_lib, wl, count):
    """Every full-size configuration: the fused launch equals the separate calls on every
    output (scores, indices, packed K and V), and sampled units match the oracle."""
    import torch
    sep = parity.DeviceRun(cuda_lib, wl)
    fus = parity.DeviceRun(cuda_lib, wl, dw=sep.dw, fused=True)
    assert fus.status_score == 0
    _compare(sep, fus)
    del sep
    parity.check_units(fus, parity.sample_units(wl, count, seed=91))
    del fus
    torch.cuda.empty_cache()


def test_fused_repeated_launches_agree(cuda_lib):
    """The barrier words are re-armed by every launch: back-to-back launches on one
    workspace give identical results."""
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[3000, 5000])
    run = parity.DeviceRun(kv, wl, fused=True)
    b = run.bufs
    first = (b.scores.clone(), b.sel.clone(), b.k_out.clone())
    for _ in range(3):
        kv.evict(run.prob, run.dw.q, run.dw.k, run.dw.v, b, fused=True)
    torch.cuda.synchronize()
    assert kv.kv_check_status(b.score_ws) == 0
    assert torch.equal(first[0], b.scores) and torch.equal(first[1], b.sel)
    assert torch.equal(first[2], b.k_out)


def test_fused_bad_budget_posts_status(cuda_lib):
    """A unit whose budget is below sinks + window: KV_ERR_BUDGET in the score
    workspace, every other unit selected and compacted as by the separate calls."""
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 4999)
    sep = parity.DeviceRun(kv, wl)
    b = sep.bufs
    bad = b.budgets.clone()
    bad[1] = wl.num_sinks + wl.window - 1
    sel = torch.full_like(b.sel, -7)
    scores = torch.empty_like(b.scores)
    kout, vout = torch.zeros_like(b.k_out), torch.zeros_like(b.v_out)
    kv.kv_evict_fused(sep.prob, sep.dw.q, sep.dw.k, sep.dw.v, bad, b.offsets, b.total_rows,
                      scores, sel, kout, vout, b.score_ws)
    torch.cuda.synchronize()
    assert kv.kv_check_status(b.score_ws) == kv.KV_ERR_BUDGET
    off = b.offsets_host
    assert bool((sel[int(off[1]):int(off[2])] == -7).all())      # unit 1 untouched
    keep = torch.ones(b.total_rows, dtype=torch.bool, device=sel.device)
    keep[int(off[1]):int(off[2])] = False
    assert torch.equal(sel[:b.total_rows][keep], b.sel[:b.total_rows][keep])
    assert torch.equal(kout[:b.total_rows][keep], b.k_out[:b.total_rows][keep])


def test_fused_wait_limit_zero_times_out_and_recovers(cuda_lib):
    """With a zero wait limit the first grid barrier gives up: KV_ERR_TIMEOUT, the
    kernel returns, and the next launch with the default limit gives the right result."""
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.LONG_128K, 5003)
    sep = parity.DeviceRun(kv, wl)
    b = sep.bufs
    old = kv.load().kv_get_wait_limit_ns()
    try:
        kv.load().kv_set_wait_limit_ns(0)
        kv.evict(sep.prob, sep.dw.q, sep.dw.k, sep.dw.v, b, fused=True)
        torch.cuda.synchronize()
        assert kv.kv_check_status(b.score_ws) == kv.KV_ERR_TIMEOUT
    finally:
        kv.load().kv_set_wait_limit_ns(old)
    fus = parity.DeviceRun(kv, wl, dw=sep.dw, fused=True)
    sep2 = parity.DeviceRun(kv, wl, dw=sep.dw)
    assert fus.status_score == 0
    _compare(sep2, fus)


def test_fused_rejects_pooling_and_head_budgets(cuda_lib):
    kv = cuda_lib
    wl = synth.TINY
    prob = kv.Problem.for_workload(wl, pool_kernel=11)
    with pytest.raises(ValueError):
        kv.evict(prob, None, None, None, None, fused=True)
