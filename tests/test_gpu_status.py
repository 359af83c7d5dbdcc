"""The workspace status contract on the GPU.

Workspaces need no initialisation: each call that starts a sequence on a
workspace (kv_score_attention, so kv_score; kv_evict_fused; kv_select_topk;
kv_head_budgets) zeroes its status word before its first kernel, and
kv_score_rescore adds to the word of the attention pass it follows.  These
tests fill every workspace with 0xFF bytes -- what an uninitialised
allocation can hold -- and check that good input gives KV_OK and the same
results as zeroed workspaces, and that device-side errors are still reported.
No test here faults a GPU: the errors are bad budgets in device memory and V
values the fp16 product of pass 1 cannot carry.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _ff(n):
    import torch
    return torch.full((max(n, 256),), 0xFF, dtype=torch.uint8, device="cuda")


def _bits(t):
    import torch
    return t.contiguous().view(torch.int32 if t.element_size() == 4 else torch.int16).cpu().numpy()


@pytest.mark.parametrize("rule", [0, 2], ids=["dropkv", "attn_sum"])
def test_uninitialised_workspaces_give_ok_and_identical_results(cuda_lib, rule):
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 2300])
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl, score_rule=rule, head_budgets=True)
    budgets = np.full((wl.num_requests, wl.num_layers, wl.num_kv_heads), 300, dtype=np.int32)
    ref = kv.Buffers(prob, budgets)       # zeroed workspaces
    kv.evict(prob, dw.q, dw.k, dw.v, ref)
    torch.cuda.synchronize()
    assert kv.kv_check_status(ref.score_ws) == 0 and kv.kv_check_status(ref.select_ws) == 0

    bufs = kv.Buffers(prob, budgets)
    bufs.score_ws = _ff(kv.kv_score_workspace_size(prob))
    bufs.select_ws = _ff(kv.kv_select_workspace_size(prob))
    # the separate passes, then the whole-score call, then selection with per-head budgets
    kv.kv_score_attention(prob, dw.q, dw.k, dw.v, bufs.score_ws)
    kv.kv_score_rescore(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws)
    assert kv.kv_check_status(bufs.score_ws) == kv.KV_OK
    np.testing.assert_array_equal(_bits(bufs.scores), _bits(ref.scores))
    bufs.score_ws.fill_(0xFF)
    bufs.select_ws.fill_(0xFF)
    sel, k_out, v_out, _ = kv.evict(prob, dw.q, dw.k, dw.v, bufs)
    assert kv.kv_check_status(bufs.score_ws) == kv.KV_OK
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_OK
    np.testing.assert_array_equal(_bits(bufs.scores), _bits(ref.scores))
    np.testing.assert_array_equal(bufs.head_budgets.cpu().numpy(), ref.head_budgets.cpu().numpy())
    n = ref.total_rows
    np.testing.assert_array_equal(sel.cpu().numpy(), ref.sel[:n].cpu().numpy())
    np.testing.assert_array_equal(_bits(k_out), _bits(ref.k_out[:n]))
    np.testing.assert_array_equal(_bits(v_out), _bits(ref.v_out[:n]))


def test_uninitialised_workspace_fused_launch(cuda_lib):
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.LONG_128K, 3001)
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    budgets = np.full((1, wl.num_layers, wl.num_kv_heads), 400, dtype=np.int32)
    ref = kv.Buffers(prob, budgets)
    kv.evict(prob, dw.q, dw.k, dw.v, ref)
    bufs = kv.Buffers(prob, budgets)
    bufs.score_ws = _ff(kv.kv_score_workspace_size(prob))
    sel, k_out, _, _ = kv.evict(prob, dw.q, dw.k, dw.v, bufs, fused=True)
    assert kv.kv_check_status(bufs.score_ws) == kv.KV_OK
    np.testing.assert_array_equal(_bits(bufs.scores), _bits(ref.scores))
    np.testing.assert_array_equal(sel.cpu().numpy(), ref.sel[:ref.total_rows].cpu().numpy())
    np.testing.assert_array_equal(_bits(k_out), _bits(ref.k_out[:ref.total_rows]))
    # a bad device budget is still reported from an uninitialised workspace
    bufs.score_ws.fill_(0xFF)
    bufs.budgets.fill_(7)
    kv.evict(prob, dw.q, dw.k, dw.v, bufs, fused=True)
    assert kv.kv_check_status(bufs.score_ws) == kv.KV_ERR_BUDGET


def test_bad_budget_reported_from_uninitialised_select_workspace(cuda_lib):
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 600, layers=1, kv_heads=2)
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    bufs = kv.Buffers(prob, np.full((1, 1, 2), 100, dtype=np.int32))
    bufs.score_ws = _ff(kv.kv_score_workspace_size(prob))
    bufs.select_ws = _ff(kv.kv_select_workspace_size(prob))
    kv.kv_score(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws)
    kv.kv_select_topk(prob, bufs.scores, bufs.budgets, bufs.offsets, bufs.sel, bufs.select_ws)
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_OK
    bufs.select_ws.fill_(0xFF)
    bufs.budgets.fill_(7)   # below sinks + window, and disagrees with offsets
    kv.kv_select_topk(prob, bufs.scores, bufs.budgets, bufs.offsets, bufs.sel, bufs.select_ws)
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_ERR_BUDGET
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_OK   # cleared


def test_head_budget_error_is_seen_after_the_selection(cuda_lib):
    """kv_head_budgets copies a bad layer's budgets through; the kv_select_topk that
    takes its outputs zeroes the status word, fails the same check on the same
    units and posts KV_ERR_BUDGET again."""
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 600, layers=1, kv_heads=2)
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl, head_budgets=True)
    bufs = kv.Buffers(prob, np.full((1, 1, 2), 100, dtype=np.int32))
    bufs.select_ws = _ff(kv.kv_select_workspace_size(prob))
    kv.kv_score(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws)
    bad = bufs.budgets.clone()
    bad.fill_(7)
    kv.kv_head_budgets(prob, bufs.scores, bad, bufs.offsets, bufs.head_budgets,
                       bufs.head_offsets, bufs.select_ws)
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_ERR_BUDGET
    np.testing.assert_array_equal(bufs.head_budgets.cpu().numpy(), bad.cpu().numpy())
    bufs.select_ws.fill_(0xFF)
    kv.kv_head_budgets(prob, bufs.scores, bad, bufs.offsets, bufs.head_budgets,
                       bufs.head_offsets, bufs.select_ws)
    kv.kv_select_topk(prob, bufs.scores, bufs.head_budgets, bufs.head_offsets, bufs.sel,
                      bufs.select_ws)
    torch.cuda.synchronize()
    assert kv.kv_check_status(bufs.select_ws) == kv.KV_ERR_BUDGET


def test_each_scoring_call_starts_a_new_status(cuda_lib):
    """An error posted by one kv_score stays until kv_check_status or the next
    kv_score on the workspace, which starts from zero."""
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 1200, layers=1, kv_heads=1)
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    bufs = kv.Buffers(prob, np.full((1, 1, 1), 100, dtype=np.int32))
    good_v = dw.v.clone()
    dw.v[0, 0, 300, 3] = 1.0e5
    kv.kv_score(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws)
    dw.v.copy_(good_v)
    kv.kv_score(prob, dw.q, dw.k, dw.v, bufs.scores, bufs.score_ws)
    assert kv.kv_check_status(bufs.score_ws) == kv.KV_OK


def test_tiny_value_block_reports_unsupported_and_zero_v_does_not(cuda_lib):
    """fp16 keeps few bits of values below 2^-14: when P V runs in fp16 (window rows
    over one 128-row chunk), a block of 64 V rows whose values are all that small
    (but not all zero) is refused; V that is exactly zero is carried exactly and
    accepted."""
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.LONG_128K, 1200, layers=1, kv_heads=2).scaled(
        budget_policy="uniform")
    assert wl.rows > 128
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    ws = torch.zeros(kv.kv_score_workspace_size(prob), dtype=torch.uint8, device="cuda")
    scores = torch.zeros((1, 2, dw.N_tot), dtype=torch.float32, device="cuda")
    good_v = dw.v.clone()
    dw.v[0, 0, 128:192] *= 1.0e-6       # one 64-row block of the first unit, ~1e-6
    kv.kv_score(prob, dw.q, dw.k, dw.v, scores, ws)
    assert kv.kv_check_status(ws) == kv.KV_ERR_UNSUPPORTED
    dw.v.copy_(good_v)
    dw.v[0, 1].zero_()                  # a whole unit of exact zeros
    kv.kv_score(prob, dw.q, dw.k, dw.v, scores, ws)
    assert kv.kv_check_status(ws) == kv.KV_OK
    assert float(scores[0, 1].abs().max()) == 0.0


@pytest.mark.parametrize("scale", [1.0e5, 1.0e-6], ids=["huge", "tiny"])
def test_single_chunk_form_takes_the_whole_bf16_range(cuda_lib, scale):
    """With the window rows in one 128-row chunk, P V multiplies bf16 V by P as a
    bf16 hi/lo pair: V values fp16 cannot hold (|v| >= 65504, or all below 2^-14)
    are accepted and scored to the oracle's tolerance."""
    from synth.device import DeviceWorkload
    from tests import parity
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 1500, layers=1, kv_heads=2)
    assert wl.rows <= 128
    dw = DeviceWorkload(wl)
    dw.v[0, 1, 100:400] *= scale          # a stretch of unit (0, 0, 1)
    budgets = np.full((1, 1, 2), 200, dtype=np.int32)
    run = parity.DeviceRun(kv, wl, budgets=budgets, dw=dw)
    assert run.status_score == kv.KV_OK and run.status_select == kv.KV_OK
    # the oracle's input: the host regeneration with the same scaling (an fp32
    # product rounded to bf16, as torch's bf16 multiply does), checked against the
    # device's bits
    import torch
    import oracle
    q, k, v = dw.unit_host(0, 0, 1)
    v = v.copy()
    v[100:400] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(v[100:400]) * np.float32(scale))
    dev = dw.v[0, 1].cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(dev, v)
    S = oracle.unit_scores_rule(q, k, v, wl.group, wl.window, 0)
    parity.check_unit(run, 0, 0, 1, oracle_out=(q, k, v, S))
