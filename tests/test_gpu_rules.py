"""GPU parity of the other score rules and of max pooling against the fp64 oracle.

The squared DropKV aggregation and the observation-window attention sum run
through the same C-ABI calls as the DropKV score (kv_problem.score_rule), and
kv_pool_scores pools the scores before selection; parity.check_unit compares
the raw scores, the pooled scores (bit-exact against the oracle's pooling of
the GPU's own raw scores), the selection and the compaction unit by unit.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu

SQUARED, ATTN_SUM = oracle.RULE_DROPKV_SQUARED, oracle.RULE_ATTN_SUM

SMALL = [
    synth.TINY,
    synth.small_variant(synth.LONG_128K, 5003),                       # G w = 256: two chunks
    synth.small_variant(synth.QWEN7B_128K, 10500, kv_heads=1),        # G w = 448: four chunks
    synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 4097, 2222]),
]


def _run(kv, wl, **kw):
    run = parity.DeviceRun(kv, wl, **kw)
    assert run.status_score == 0 and run.status_select == 0
    return run


@pytest.mark.parametrize("rule", [SQUARED, ATTN_SUM], ids=["squared", "attn_sum"])
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_rule_small_workloads_all_units(cuda_lib, wl, rule):
    run = _run(cuda_lib, wl, score_rule=rule)
    res = parity.check_units(run, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL


def test_attention_sum_totals_rows_on_gpu(cuda_lib):
    """Every window row's weights sum to one: each unit's scores sum to G * w."""
    import torch
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[3000, 5000])
    run = _run(cuda_lib, wl, score_rule=ATTN_SUM)
    cu = run.dw.cu_host
    s = run.bufs.scores.double()
    for r in range(len(cu) - 1):
        tot = s[:, :, int(cu[r]):int(cu[r + 1])].sum(dim=2)
        torch.testing.assert_close(tot, torch.full_like(tot, wl.group * wl.window), rtol=1e-4,
                                   atol=0)


@pytest.mark.parametrize("rule,kernel", [(0, 11), (0, 13), (ATTN_SUM, 11), (SQUARED, 13)],
                         ids=["dropkv_k11", "dropkv_k13", "attn_sum_k11", "squared_k13"])
@pytest.mark.parametrize("wl", SMALL[1:], ids=lambda w: w.name)
def test_pooled_small_workloads_all_units(cuda_lib, wl, rule, kernel):
    run = _run(cuda_lib, wl, score_rule=rule, pool_kernel=kernel)
    parity.check_units(run, list(range(wl.num_units)))


@pytest.mark.parametrize("kernel", [1, 3, 17, 21, 255],
                         ids=lambda k: "k%d" % k)
def test_pool_kernel_widths_and_request_edges(cuda_lib, kernel):
    """Register path (radius <= 8) and shared-memory path (larger), across several
    requests packed in one row, one of them with no candidates beyond the sinks."""
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[36, 2049, 37, 4500, 300])
    prob = kv.Problem.for_workload(wl)
    L, H = wl.num_layers, wl.num_kv_heads
    N = prob.total_tokens
    g = torch.Generator(device="cuda").manual_seed(kernel)
    s_in = torch.rand((L, H, N), generator=g, device="cuda", dtype=torch.float32)
    s_in[0, 0, 100:200] = 0.5          # plateaus and exact ties
    s_out = torch.full_like(s_in, -1.0)
    kv.kv_pool_scores(prob, kernel, s_in, s_out)
    torch.cuda.synchronize()
    a, b = s_in.cpu().numpy().astype(np.float64), s_out.cpu().numpy()
    cu = prob.cu_host
    for l in range(L):
        for h in range(H):
            for r in range(len(cu) - 1):
                c0, c1 = int(cu[r]), int(cu[r + 1])
                np.testing.assert_array_equal(b[l, h, c0:c1],
                                              oracle.pool_unit(a[l, h, c0:c1], wl.window, kernel))


@pytest.mark.parametrize("rule,kernel,wl,count", [
    (ATTN_SUM, 11, synth.LONG_128K, 2),
    (SQUARED, 1, synth.LLAMA8B_32K, 2),
    (0, 13, synth.RAGGED_MISTRAL, 2),
], ids=["attn_sum_k11_long128k", "squared_llama32k", "dropkv_k13_ragged"])
def test_full_size_rules_sampled_units(cuda_lib, rule, kernel, wl, count):
    import torch
    run = _run(cuda_lib, wl, score_rule=rule, pool_kernel=kernel)
    parity.check_units(run, parity.sample_units(wl, count, seed=77))
    b = run.bufs
    assert bool(torch.isfinite(b.scores).all()) and float(b.scores.min()) >= 0.0
    if rule == ATTN_SUM:
        assert float(b.scores.max()) <= wl.group * wl.window * (1 + 1e-4)
    del run
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# per-head budgets (AdaDropKV)
# --------------------------------------------------------------------------
def _layer_heads(run, r, l, ranked):
    cu = run.dw.cu_host
    return ranked[l, :, int(cu[r]):int(cu[r + 1])].astype(np.float64)


@pytest.mark.parametrize("rule,kernel", [(0, 1), (ATTN_SUM, 11)], ids=["dropkv", "attn_sum_k11"])
@pytest.mark.parametrize("wl", SMALL[1:] + [synth.TINY.scaled(name="tiny_1L_4kv_d64_n2048",
                                                              num_kv_heads=4, num_q_heads=16)],
                         ids=lambda w: w.name)
def test_head_budgets_small_workloads(cuda_lib, wl, rule, kernel):
    run = _run(cuda_lib, wl, score_rule=rule, pool_kernel=kernel, head_budgets=True)
    ranked = run.ranked_scores()
    H, w, s = wl.num_kv_heads, wl.window, wl.num_sinks
    inb = np.asarray(run.budgets).reshape(-1)
    for r in range(wl.num_requests):
        for l in range(wl.num_layers):
            u0 = wl.unit_index(r, l, 0)
            want = oracle.head_budgets(_layer_heads(run, r, l, ranked), w, s, inb[u0:u0 + H])
            np.testing.assert_array_equal(run.eff_budgets[u0:u0 + H], want,
                                          err_msg="head budgets (%d, %d)" % (r, l))
            assert run.eff_budgets[u0:u0 + H].sum() == inb[u0:u0 + H].sum()
    np.testing.assert_array_equal(run.eff_offsets, oracle.offsets(run.eff_budgets))
    parity.check_units(run, list(range(wl.num_units)))


def test_head_budgets_against_oracle_scores(cuda_lib):
    """Layer-wide winners from the GPU scores and from the oracle's scores differ only in
    tokens within the score tolerance of the oracle's layer threshold."""
    wl = synth.small_variant(synth.LONG_128K, 5003)
    run = _run(cuda_lib, wl, head_budgets=True)
    H, w, s = wl.num_kv_heads, wl.window, wl.num_sinks
    inb = np.asarray(run.budgets).reshape(-1)
    ranked = run.ranked_scores()
    for l in range(wl.num_layers):
        u0 = wl.unit_index(0, l, 0)
        So = np.stack([parity.oracle_unit(wl, run.dw, 0, l, h)[3] for h in range(H)])
        Sg = _layer_heads(run, 0, l, ranked)
        n = So.shape[1]
        k = int(inb[u0:u0 + H].sum()) - H * (s + w)

        def winners(S):
            vals = S[:, s:n - w].reshape(-1)
            hh = np.repeat(np.arange(H), n - w - s)
            jj = np.tile(np.arange(s, n - w), H)
            order = np.lexsort((jj, hh, -vals))[:k]
            return set(zip(hh[order].tolist(), jj[order].tolist())), vals[order[-1]]

        wo, theta = winners(So)
        wg, _ = winners(Sg)
        for (h, j) in wo ^ wg:
            assert abs(So[h, j] - theta) <= parity.SCORE_RTOL * theta, (l, h, j)


def test_head_budgets_bad_input_posts_status(cuda_lib):
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 4999)
    run = _run(kv, wl)
    b = run.bufs
    bad = b.budgets.clone()
    bad[0] = wl.num_sinks + wl.window - 1
    out_b, out_o = torch.empty_like(b.budgets), torch.empty_like(b.offsets)
    kv.kv_head_budgets(run.prob, b.scores, bad, b.offsets, out_b, out_o, b.select_ws)
    assert kv.kv_check_status(b.select_ws) == kv.KV_ERR_BUDGET
    # the offending layer is copied through; the others are computed
    H = wl.num_kv_heads
    np.testing.assert_array_equal(out_b[:H].cpu().numpy(), bad[:H].cpu().numpy())
    assert int(out_o[-1]) == int(b.offsets[-1])
