"""The host-memory pipeline (HostPipeline) against the device path.

HostPipeline copies layer groups of pinned host Q/K/V in while earlier groups are
scored, selected and compacted (by the separate calls, or by the fused launch), and
copies the kept rows out; it runs the same kernels on sub-problems of a few layers.
These problems are small enough that the sub-problems and the whole problem choose the
same pass-1 split size, so every unit's kept indices and rows must equal those of the
whole-problem device path bit for bit (that path is checked against the oracle in
test_gpu_parity.py and test_gpu_rules.py).
"""
import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl,group,rule,pool,heads,fused", [
    (synth.small_variant(synth.LONG_128K, 5003, layers=4), 2, 0, 1, False, False),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=5, requests=[1500, 4097, 2222]), 2, 0, 1,
     False, False),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=4, requests=[3000, 2100]), 3, 2, 11, True,
     False),
    (synth.small_variant(synth.LONG_128K, 5003, layers=4), 2, 0, 1, False, True),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=5, requests=[1500, 4097, 2222]), 2, 1, 1,
     False, True),
], ids=["long_g2", "ragged_l5_g2", "ragged_g3_attnsum_pool_heads", "long_g2_fused",
        "ragged_l5_g2_squared_fused"])
def test_host_pipeline_equals_device_path(cuda_lib, wl, group, rule, pool, heads, fused):
    import torch
    kv = cuda_lib
    run = parity.DeviceRun(kv, wl, score_rule=rule, pool_kernel=pool, head_budgets=heads)
    assert run.status_score == 0 and run.status_select == 0
    dw = run.dw
    qh = torch.empty(dw.q.shape, dtype=dw.q.dtype, pin_memory=True)
    kh = torch.empty(dw.k.shape, dtype=dw.k.dtype, pin_memory=True)
    vh = torch.empty(dw.v.shape, dtype=dw.v.dtype, pin_memory=True)
    qh.copy_(dw.q)
    kh.copy_(dw.k)
    vh.copy_(dw.v)
    pipe = kv.HostPipeline(run.prob, run.budgets, group_layers=group, fused=fused)
    for _ in range(2):                    # the second run reuses every buffer
        sel, ko, vo, offs = pipe.run(qh, kh, vh)
    assert pipe.total_rows == run.bufs.total_rows
    sel = sel.numpy()
    ko = ko.view(torch.int16).numpy()
    vo = vo.view(torch.int16).numpy()
    ref_sel = run.bufs.sel.cpu().numpy()
    ref_k = run.bufs.k_out.cpu().view(torch.int16).numpy()
    ref_v = run.bufs.v_out.cpu().view(torch.int16).numpy()
    H = wl.num_kv_heads
    # group-major order: groups of layers, then request, layer, head
    i = 0
    for (l0, l1) in pipe.groups:
        for r in range(wl.num_requests):
            for l in range(l0, l1):
                for h in range(H):
                    u = wl.unit_index(r, l, h)
                    a, b = int(run.eff_offsets[u]), int(run.eff_offsets[u + 1])
                    assert int(offs[i + 1] - offs[i]) == b - a
                    c = int(offs[i])
                    np.testing.assert_array_equal(sel[c:c + b - a], ref_sel[a:b])
                    np.testing.assert_array_equal(ko[c:c + b - a], ref_k[a:b])
                    np.testing.assert_array_equal(vo[c:c + b - a], ref_v[a:b])
                    i += 1
