"""The bounds-checked build (libkvevict_debug.so, compiled with -DKV_DEBUG_BOUNDS).

Every TMA tile coordinate, workspace offset and gather index of the kernels is
tested against its tensor's extent before use; a failed check posts
KV_ERR_INVALID_ARG to the workspace status word and skips the access (it never
traps).  It stands in for a memory checker on this hardware.  The tests run the
tiny and a ragged small workload through every call of the debug library --
the two scoring passes under all three score rules, pooling, per-head budgets,
selection, compaction and the fused launch -- and require status KV_OK and
results bit-identical to the release library.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

WORKLOADS = [synth.TINY,
             synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 4097, 2222]),
             synth.small_variant(synth.QWEN7B_128K, 10500, kv_heads=1)]


def _path(kv, lib, prob, dw, rule, pool, heads, fused, budgets):
    """The whole path through the C functions of `lib`; returns the outputs (host)
    and the two status words."""
    import torch
    s = torch.cuda.current_stream().cuda_stream
    N, d = prob.total_tokens, prob.head_dim
    L, H = prob.num_layers, prob.num_kv_heads
    b = np.ascontiguousarray(budgets, dtype=np.int32).reshape(-1)
    offs = kv.kv_make_offsets(prob, b)
    total = int(offs[-1])
    dev = "cuda"
    bd, od = torch.from_numpy(b).to(dev), torch.from_numpy(offs).to(dev)
    scores = torch.full((L, H, N), float("nan"), dtype=torch.float32, device=dev)
    pooled = torch.full_like(scores, float("nan"))
    n_ws = ctypes.c_size_t()
    assert lib.kv_score_workspace_size(prob.c, ctypes.byref(n_ws)) == 0
    ws = torch.full((max(n_ws.value, 256),), 0xFF, dtype=torch.uint8, device=dev)
    assert lib.kv_select_workspace_size(prob.c, ctypes.byref(n_ws)) == 0
    sws = torch.full((max(n_ws.value, 256),), 0xFF, dtype=torch.uint8, device=dev)
    sel = torch.full((max(total, 1),), -1, dtype=torch.int32, device=dev)
    ko = torch.zeros((max(total, 1), d), dtype=torch.bfloat16, device=dev)
    vo = torch.zeros_like(ko)
    hb, ho = torch.empty_like(bd), torch.empty_like(od)
    p = lambda t: t.data_ptr()
    if fused:
        rc = lib.kv_evict_fused(prob.c, p(dw.q), p(dw.k), p(dw.v), p(bd), p(od), total,
                                p(scores), p(sel), p(ko), p(vo), p(ws), ws.numel(), s)
        assert rc == 0, kv.status_string(rc)
    else:
        assert lib.kv_score_attention(prob.c, p(dw.q), p(dw.k), p(dw.v), p(ws), ws.numel(),
                                      s) == 0
        assert lib.kv_score_rescore(prob.c, p(dw.q), p(dw.k), p(dw.v), p(scores), p(ws),
                                    ws.numel(), s) == 0
        ranked = scores
        if pool > 1:
            assert lib.kv_pool_scores(prob.c, pool, p(scores), p(pooled), s) == 0
            ranked = pooled
        sb, so = bd, od
        if heads:
            assert lib.kv_head_budgets(prob.c, p(ranked), p(bd), p(od), p(hb), p(ho), p(sws),
                                       sws.numel(), s) == 0
            sb, so = hb, ho
        assert lib.kv_select_topk(prob.c, p(ranked), p(sb), p(so), p(sel), p(sws), sws.numel(),
                                  s) == 0
        assert lib.kv_compact(prob.c, p(dw.k), p(dw.v), p(sel), p(so), total, p(ko), p(vo),
                              s) == 0
    st_score, st_sel = ctypes.c_int32(), ctypes.c_int32()
    assert lib.kv_check_status(p(ws), s, ctypes.byref(st_score)) == 0
    assert lib.kv_check_status(p(sws), s, ctypes.byref(st_sel)) == 0
    as_bits = lambda t: t.cpu().view(torch.int32 if t.element_size() == 4 else torch.int16).numpy()
    out = [as_bits(scores), as_bits(sel), as_bits(ko), as_bits(vo)]
    if pool > 1:
        out.append(as_bits(pooled))
    return out, (st_score.value, 0 if fused else st_sel.value)


@pytest.mark.parametrize("wl", WORKLOADS, ids=lambda w: w.name)
@pytest.mark.parametrize("rule,pool,heads,fused", [
    (0, 1, False, False), (1, 1, False, False), (2, 11, True, False), (0, 1, False, True),
    (2, 1, False, True)], ids=["dropkv", "squared", "attnsum_pool_heads", "fused",
                               "fused_attnsum"])
def test_debug_build_in_bounds_and_identical(cuda_lib, wl, rule, pool, heads, fused):
    from synth.device import DeviceWorkload
    kv = cuda_lib
    dbg = kv.load_debug()
    rel = kv.load()
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl, score_rule=rule)
    prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
    from tests import parity
    budgets = parity.product_budgets(kv, wl, prof)
    got, st = _path(kv, dbg, prob, dw, rule, pool, heads, fused, budgets)
    assert st == (kv.KV_OK, kv.KV_OK), "debug build posted %s" % (st,)
    ref, st_ref = _path(kv, rel, prob, dw, rule, pool, heads, fused, budgets)
    assert st_ref == (kv.KV_OK, kv.KV_OK)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)
