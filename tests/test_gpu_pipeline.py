"""kv_evict_host (the host-memory pipeline, through the C ABI) against the device path.

kv_evict_host copies layer groups of host Q/K/V in while earlier groups are scored,
selected and compacted (by the separate calls, or by the fused launch), and copies
the kept indices and rows back, each group's rows straight into their place in the
standard unit order.  It runs the same kernels on sub-problems of a few layers.
These problems are small enough that the sub-problems and the whole problem choose
the same pass-1 split size, so the offsets, kept indices and rows must equal those
of the whole-problem device path bit for bit (that path is checked against the
oracle in test_gpu_parity.py and test_gpu_rules.py).
"""
import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu


def _host_copies(dw, pinned=True):
    import torch
    out = []
    for t in (dw.q, dw.k, dw.v):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=pinned)
        h.copy_(t)
        out.append(h)
    return out


@pytest.mark.parametrize("wl,group,rule,pool,heads,fused", [
    (synth.small_variant(synth.LONG_128K, 5003, layers=4), 2, 0, 1, False, False),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=5, requests=[1500, 4097, 2222]), 2, 0, 1,
     False, False),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=4, requests=[3000, 2100]), 3, 2, 11, True,
     False),
    (synth.small_variant(synth.LONG_128K, 5003, layers=4), 2, 0, 1, False, True),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=5, requests=[1500, 4097, 2222]), 2, 1, 1,
     False, True),
    (synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=3, requests=[1200, 900]), 3, 0, 1, False,
     False),
], ids=["long_g2", "ragged_l5_g2", "ragged_g3_attnsum_pool_heads", "long_g2_fused",
        "ragged_l5_g2_squared_fused", "ragged_one_group"])
def test_host_pipeline_equals_device_path(cuda_lib, wl, group, rule, pool, heads, fused):
    import torch
    kv = cuda_lib
    run = parity.DeviceRun(kv, wl, score_rule=rule, pool_kernel=pool, head_budgets=heads)
    assert run.status_score == 0 and run.status_select == 0
    qh, kh, vh = _host_copies(run.dw)
    pipe = kv.HostPipeline(run.prob, run.budgets, group_layers=group, fused=fused)
    for _ in range(2):                    # the second run reuses every buffer
        sel, ko, vo, offs = pipe.run(qh, kh, vh)
    assert pipe.total_rows == run.bufs.total_rows
    np.testing.assert_array_equal(offs, run.eff_offsets)
    n = pipe.total_rows
    np.testing.assert_array_equal(sel.numpy(), run.bufs.sel[:n].cpu().numpy())
    np.testing.assert_array_equal(ko.view(torch.int16).numpy(),
                                  run.bufs.k_out[:n].cpu().view(torch.int16).numpy())
    np.testing.assert_array_equal(vo.view(torch.int16).numpy(),
                                  run.bufs.v_out[:n].cpu().view(torch.int16).numpy())


def test_host_pipeline_pageable_buffers(cuda_lib):
    """Pageable host inputs work (their copies do not overlap the kernels)."""
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=4, requests=[1300, 2000])
    run = parity.DeviceRun(kv, wl)
    qh, kh, vh = _host_copies(run.dw, pinned=False)
    pipe = kv.HostPipeline(run.prob, run.budgets, group_layers=3)
    sel, ko, _, offs = pipe.run(qh, kh, vh)
    np.testing.assert_array_equal(offs, run.eff_offsets)
    np.testing.assert_array_equal(sel.numpy(), run.bufs.sel[:pipe.total_rows].cpu().numpy())
    np.testing.assert_array_equal(
        ko.view(torch.int16).numpy(),
        run.bufs.k_out[:pipe.total_rows].cpu().view(torch.int16).numpy())


def test_host_pipeline_reports_device_status_of_an_early_group(cuda_lib):
    """A V value fp16 cannot carry in the first group is reported although later
    groups (which zero their own status words) run clean."""
    kv = cuda_lib
    wl = synth.small_variant(synth.LONG_128K, 5003, layers=4)
    run = parity.DeviceRun(kv, wl)
    qh, kh, vh = _host_copies(run.dw)
    vh[0, 1, 500, 7] = 1.0e5
    pipe = kv.HostPipeline(run.prob, run.budgets, group_layers=1)
    with pytest.raises(kv.KvError) as e:
        pipe.run(qh, kh, vh)
    assert e.value.code == kv.KV_ERR_UNSUPPORTED


def test_host_pipeline_rejects_bad_budgets_before_copying(cuda_lib):
    kv = cuda_lib
    wl = synth.small_variant(synth.LLAMA8B_32K, 1200, layers=2)
    run = parity.DeviceRun(kv, wl)
    qh, kh, vh = _host_copies(run.dw)
    pipe = kv.HostPipeline(run.prob, run.budgets, group_layers=1)
    bad = np.array(run.budgets).reshape(-1).copy()
    bad[1] = 3
    offs = np.zeros(wl.num_units + 1, dtype=np.int64)
    with pytest.raises(kv.KvError) as e:
        kv.kv_evict_host(run.prob, pipe.plan, qh, kh, vh, bad, offs, pipe.sel_host,
                         pipe.k_out_host, pipe.v_out_host, pipe.workspace)
    assert e.value.code == kv.KV_ERR_BUDGET
