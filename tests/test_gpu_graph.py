"""The eviction path captured into a CUDA graph and replayed.

Every call of the path is asynchronous on the caller's stream and allocates
nothing, so a whole step (scoring, selection, compaction; or the fused launch)
can be captured once and replayed, which removes the per-launch host cost that
bounds small problems.  A replay must give exactly what the same calls give
when issued directly, also after the inputs are rewritten in place between
replays.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    return t.contiguous().view(torch.int32 if t.element_size() == 4 else torch.int16).cpu().numpy()


def _outputs(bufs):
    n = bufs.total_rows
    return [_bits(bufs.scores), _bits(bufs.sel[:n]), _bits(bufs.k_out[:n]), _bits(bufs.v_out[:n])]


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("wl", [synth.TINY,
                                synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[1500, 2300]),
                                synth.small_variant(synth.LONG_128K, 3001)],
                         ids=lambda w: w.name)
def test_path_replays_from_a_cuda_graph(cuda_lib, wl, fused):
    import torch
    from synth.device import DeviceWorkload
    kv = cuda_lib
    dw = DeviceWorkload(wl)
    prob = kv.Problem.for_workload(wl)
    budgets = np.full((wl.num_requests, wl.num_layers, wl.num_kv_heads),
                      wl.num_sinks + wl.window + 100, dtype=np.int32)
    ref = kv.Buffers(prob, budgets)
    bufs = kv.Buffers(prob, budgets)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kv.evict(prob, dw.q, dw.k, dw.v, bufs, fused=fused)   # first calls outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kv.evict(prob, dw.q, dw.k, dw.v, bufs, fused=fused)
    for replay in range(2):
        if replay == 1:   # new window queries, written in place between replays
            dw.q.copy_(torch.flip(dw.q, dims=[-2]))
        for t in (bufs.scores, bufs.sel, bufs.k_out, bufs.v_out):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert kv.kv_check_status(bufs.score_ws) == kv.KV_OK
        if not fused:
            assert kv.kv_check_status(bufs.select_ws) == kv.KV_OK
        kv.evict(prob, dw.q, dw.k, dw.v, ref, fused=fused)
        torch.cuda.synchronize()
        for a, b in zip(_outputs(bufs), _outputs(ref)):
            np.testing.assert_array_equal(a, b)
