"""kv_score_noalloc: scoring for callers that cannot allocate device memory.

Such callers (a process that reserves all device memory at start-up, a plugin
whose host application owns the allocator) cannot pass a workspace; the entry
point uses a fixed array inside the library instead.  This file is collected
last so that a run stopping at its first failure has already run every other
test.  The check: two calls in a row through the C ABI give the same scores
as kv_score with a caller-allocated workspace.  Both run the same kernels on
the same problem, so the scores must agree bit for bit (a looser check would
also be within the 1e-3 score tolerance of the parity tests).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

RTOL = 1e-3


@pytest.mark.parametrize("wl", [
    synth.TINY,
    synth.small_variant(synth.QWEN7B_128K, 3000, kv_heads=1),        # 4 row chunks
    synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 2300]),
], ids=lambda w: w.name)
def test_noalloc_matches_kv_score_twice(cuda_lib, wl):
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    lib = kv.load()
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    stream = torch.cuda.current_stream()
    shape = (wl.num_layers, wl.num_kv_heads, dw.N_tot)
    ref = torch.empty(shape, dtype=torch.float32, device="cuda")
    ws = torch.zeros(kv.kv_score_workspace_size(prob), dtype=torch.uint8, device="cuda")
    kv.kv_score(prob, dw.q, dw.k, dw.v, ref, ws, stream)
    for _ in range(2):
        out = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.kv_score_noalloc(prob.c, dw.q.data_ptr(), dw.k.data_ptr(), dw.v.data_ptr(),
                                  out.data_ptr(), stream.cuda_stream)
        assert rc == kv.KV_OK, kv.status_string(rc)
        torch.cuda.synchronize()
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(a))
        np.testing.assert_allclose(a, b, rtol=RTOL, atol=1e-30)
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    kv = cuda_lib
    wl = synth.LONG_128K
    prob = kv.Problem.for_workload(wl)
    assert kv.kv_score_workspace_size(prob) > (64 << 20)
    rc = kv.load().kv_score_noalloc(prob.c, 256, 256, 256, 256, None)
    assert rc == kv.KV_ERR_WORKSPACE
