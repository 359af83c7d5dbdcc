"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small workloads are checked on every unit; the full-size configurations on a
seeded sample of units, in the same launch configuration the benchmark times.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu


def _run(cuda_lib, wl, **kw):
    run = parity.DeviceRun(cuda_lib, wl, **kw)
    assert run.status_score == 0 and run.status_select == 0
    return run


def test_device_generator_matches_host(cuda_lib):
    import torch
    from synth.device import DeviceWorkload
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[3000, 4100])
    dw = DeviceWorkload(wl)
    for (r, l, h) in [(0, 0, 0), (1, 1, 1), (1, 0, 1)]:
        _, k, v = dw.unit_host(r, l, h)
        c0, c1 = int(dw.cu_host[r]), int(dw.cu_host[r + 1])
        kd = dw.k[l, h, c0:c1].cpu().view(torch.int16).numpy().view(np.uint16)
        vd = dw.v[l, h, c0:c1].cpu().view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(kd, k)
        np.testing.assert_array_equal(vd, v)


def test_product_budgets_equal_oracle_budgets(cuda_lib):
    for wl in synth.CONFIGS:
        prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
        np.testing.assert_array_equal(parity.product_budgets(cuda_lib, wl, prof),
                                      oracle.segment_budgets(wl, prof))


@pytest.mark.parametrize("wl", [
    synth.TINY,
    synth.small_variant(synth.LLAMA8B_32K, 4999),
    synth.small_variant(synth.LONG_128K, 5003),
    synth.small_variant(synth.QWEN7B_128K, 10500, kv_heads=1),
    # G w = 224 (G = 7, w = 32): a full 128-row chunk and a 96-row one
    synth.small_variant(synth.QWEN7B_128K, 7001).scaled(name="qwen7b_rows224_w32_small", window=32),
    synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 4097, 2222]),
], ids=lambda w: w.name)
def test_small_workloads_all_units(cuda_lib, wl):
    run = _run(cuda_lib, wl)
    res = parity.check_units(run, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL


def test_head_dim_64_many_splits(cuda_lib):
    wl = synth.TINY.scaled(name="d64_n40000", lengths=(40000,), num_kv_heads=2, num_q_heads=6,
                           window=8, budget_tokens=1000)
    run = _run(cuda_lib, wl)
    parity.check_units(run, list(range(wl.num_units)))


# window-row counts at the edges of the 128-row chunking: the largest G*w the kernels
# take (512 = four full chunks) at both head dims, and 129 rows (the second chunk holds
# one row, padded to the 32-row MMA width)
ROW_EDGES = [
    synth.LLAMA8B_32K.scaled(name="rows512_d128_g8_w64", num_layers=1, num_kv_heads=2,
                             num_q_heads=16, window=64, lengths=(3000,), ragged_range=None,
                             num_heavy=8, budget_ratio=0.1),
    synth.TINY.scaled(name="rows512_d64_g16_w32", num_kv_heads=1, num_q_heads=16, window=32,
                      lengths=(2600,), budget_tokens=400),
    synth.LLAMA8B_32K.scaled(name="rows129_d128_g3_w43", num_layers=1, num_kv_heads=2,
                             num_q_heads=6, window=43, lengths=(2500, 1700), ragged_range=None,
                             num_heavy=8, budget_ratio=0.1),
]


@pytest.mark.parametrize("wl", ROW_EDGES, ids=lambda w: w.name)
def test_window_row_edges_all_units(cuda_lib, wl):
    assert wl.rows in (512, 129)
    run = _run(cuda_lib, wl)
    res = parity.check_units(run, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL


def test_short_last_chunk_over_several_grid_rounds(cuda_lib):
    """448 window rows (chunks of 128, 128, 128, 64) with about two rounds of pass-2
    work items on the grid, where the row chunk rotates by round: every unit
    against the oracle."""
    wl = synth.QWEN7B_128K.scaled(name="qwen7b_rows448_4L_4kv_n40000", num_layers=4,
                                  num_kv_heads=4, num_q_heads=28, lengths=(40000,),
                                  ragged_range=None, num_heavy=8)
    assert wl.rows == 448 and wl.num_units == 16
    run = _run(cuda_lib, wl)
    res = parity.check_units(run, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL


def test_more_length_runs_than_the_order_tables(cuda_lib):
    """34 requests of distinct lengths: more runs of equal length than the work-item
    order tables hold, so both passes decode their items from the plan tables that
    a kernel computes in the workspace; every unit against the oracle, and the
    fused launch bit for bit against the separate calls."""
    lengths = tuple(300 + 97 * i for i in range(34))
    wl = synth.TINY.scaled(name="runs34_d64_g4_w8", num_kv_heads=1, num_q_heads=4, window=8,
                           lengths=lengths, ragged_range=None, num_heavy=0,
                           budget_tokens=None, budget_ratio=0.3)
    assert len(set(lengths)) == 34
    run = _run(cuda_lib, wl)
    res = parity.check_units(run, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL
    import torch
    fused = _run(cuda_lib, wl, dw=run.dw, fused=True)
    for name in ("scores", "sel", "k_out", "v_out"):
        a, b = getattr(run.bufs, name), getattr(fused.bufs, name)
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), name


@pytest.mark.parametrize("b_kind", ["minimum", "everything"])
def test_budget_extremes(cuda_lib, b_kind):
    wl = synth.small_variant(synth.LLAMA8B_32K, 700, layers=1)
    n = 700
    b = wl.num_sinks + wl.window if b_kind == "minimum" else n
    budgets = np.full((1, wl.num_layers, wl.num_kv_heads), b, dtype=np.int32)
    run = _run(cuda_lib, wl, budgets=budgets)
    parity.check_units(run, list(range(wl.num_units)))


def test_shortest_request_window_plus_sinks(cuda_lib):
    """n = sinks + w: no middle candidates; every token kept."""
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[36, 1200], layers=1)
    budgets = np.zeros((2, 1, wl.num_kv_heads), dtype=np.int32)
    budgets[0] = 36
    budgets[1] = 300
    wl = wl.scaled(num_heavy=0)
    run = _run(cuda_lib, wl, budgets=budgets)
    parity.check_units(run, list(range(wl.num_units)))


def test_equal_scores_break_ties_to_lower_index(cuda_lib):
    """Identical K/V rows give bit-identical GPU scores; the lower index must win."""
    import torch
    from synth.device import DeviceWorkload
    wl = synth.small_variant(synth.LLAMA8B_32K, 900, layers=1, kv_heads=1).scaled(num_heavy=0)
    dw = DeviceWorkload(wl)
    dw.k[0, 0, 100:900 - wl.window] = dw.k[0, 0, 100]
    dw.v[0, 0, 100:900 - wl.window] = dw.v[0, 0, 100]
    budgets = np.full((1, 1, 1), 200, dtype=np.int32)
    run = parity.DeviceRun(cuda_lib, wl, budgets=budgets, dw=dw)
    n, scores, sel, _, _, b = run.unit_results(0, 0, 0)
    mine = oracle.select(scores.astype(np.float64), wl.window, wl.num_sinks, b)
    np.testing.assert_array_equal(sel, mine)
    tied = scores[100:n - wl.window]
    assert np.all(tied == tied[0])


def test_bad_device_budget_posts_status(cuda_lib):
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 600, layers=1, kv_heads=1)
    from synth.device import DeviceWorkload
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    good = np.full((1, 1, 1), 100, dtype=np.int32)
    bufs = kv.Buffers(prob, good)
    kv.kv_score(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws)
    bufs.budgets.fill_(7)   # below sinks + window, and disagrees with offsets
    kv.kv_select_topk(prob, bufs.scores, bufs.budgets, bufs.offsets, bufs.sel, bufs.select_ws)
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_ERR_BUDGET
    assert kv.kv_check_status(bufs.select_ws) == 0   # cleared


@pytest.mark.parametrize("wl", [synth.LLAMA8B_32K, synth.LONG_128K, synth.QWEN7B_128K,
                                synth.RAGGED_MISTRAL], ids=lambda w: w.name)
def test_full_size_every_unit(cuda_lib, wl):
    """The full-size configurations in the launch configuration the benchmark times:
    selection and compaction of every unit (all 2048 segments of the ragged batch)
    against the oracle's rule and the generator, oracle scores on 16 seeded units
    (computed in parallel on the host cores), and properties of every score."""
    import torch
    run = _run(cuda_lib, wl)
    assert parity.check_every_unit_select_compact(run) == wl.num_units
    res = parity.check_units(run, parity.sample_units(wl, 16))
    assert len(res) == 16
    b = run.bufs
    seg_len = torch.diff(b.offsets)
    assert int(seg_len.min()) >= wl.num_sinks + wl.window
    assert bool(torch.isfinite(b.scores).all()) and float(b.scores.min()) >= 0.0
    del run
    torch.cuda.empty_cache()
