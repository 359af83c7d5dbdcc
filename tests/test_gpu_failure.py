"""Failure detection on the GPU, without a GPU fault.

Every device wait in the tensor-core kernels is bounded.  With the limit set
to 0 (kv_set_wait_limit_ns), any wait that is not already satisfied gives up
at once: the kernels post KV_ERR_TIMEOUT to the workspace status word, wait
for their own copies and MMAs still in flight, free TMEM and return.  The
tests check that status, then that the context is still usable: with the
default limit the same call gives the oracle's scores again.
"""
import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu

DEFAULT_NS = 2_000_000_000


@pytest.mark.parametrize("rule", [0, 2], ids=["dropkv", "attn_sum"])
@pytest.mark.parametrize("wl", [
    synth.small_variant(synth.LONG_128K, 5003),      # two row chunks per unit
    synth.small_variant(synth.LLAMA8B_32K, 4999),    # one row chunk, alternate tiles
], ids=lambda w: w.name)
def test_expired_waits_report_timeout_and_context_recovers(cuda_lib, wl, rule):
    """Both pass-1 kernels (attention, and row statistics for the attention sum) and
    both rescoring variants."""
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl, score_rule=rule)
    ws = torch.zeros(kv.kv_score_workspace_size(prob), dtype=torch.uint8, device="cuda")
    scores = torch.zeros((wl.num_layers, wl.num_kv_heads, dw.N_tot), dtype=torch.float32,
                         device="cuda")
    assert kv.kv_get_wait_limit_ns() == DEFAULT_NS
    try:
        kv.kv_set_wait_limit_ns(0)
        kv.kv_score(prob, dw.q, dw.k, dw.v, scores, ws)
        assert kv.kv_check_status(ws) == kv.KV_ERR_TIMEOUT
    finally:
        kv.kv_set_wait_limit_ns(DEFAULT_NS)
    # kv_check_status cleared the word; the same call now completes normally
    kv.kv_score(prob, dw.q, dw.k, dw.v, scores, ws)
    assert kv.kv_check_status(ws) == kv.KV_OK
    cu = dw.cu_host
    for (r, l, h) in [(0, 0, 0), (0, wl.num_layers - 1, wl.num_kv_heads - 1)]:
        _, _, _, S = parity.oracle_unit(wl, dw, r, l, h, rule)
        g = scores[l, h, int(cu[r]):int(cu[r + 1])].cpu().numpy().astype(np.float64)
        big = S >= parity.SCORE_ATOL
        rel = np.abs(g[big] - S[big]) / S[big]
        assert rel.max() <= parity.SCORE_RTOL


def test_value_outside_fp16_range_reports_unsupported(cuda_lib):
    """The attention pass multiplies p by v in fp16; a V value of magnitude
    65504 or more cannot be represented and is reported, not silently used."""
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    wl = synth.small_variant(synth.LONG_128K, 5003)
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    ws = torch.zeros(kv.kv_score_workspace_size(prob), dtype=torch.uint8, device="cuda")
    scores = torch.zeros((wl.num_layers, wl.num_kv_heads, dw.N_tot), dtype=torch.float32,
                         device="cuda")
    kv.kv_score(prob, dw.q, dw.k, dw.v, scores, ws)
    assert kv.kv_check_status(ws) == kv.KV_OK
    dw.v[1, 0, 777, 5] = 1.0e5
    kv.kv_score(prob, dw.q, dw.k, dw.v, scores, ws)
    assert kv.kv_check_status(ws) == kv.KV_ERR_UNSUPPORTED
