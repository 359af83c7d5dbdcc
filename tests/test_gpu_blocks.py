"""GPU parity of block eviction (BellowsKV blog, eviction operator) against the oracle.

One decision per block of consecutive layers: scores summed over the block's
layers and heads, max-pooled (13), the sinks, the window and the fraction q of
the rest kept, and every layer and head of the block compacted with the
block's tokens.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block_layers,q,kernel", [(2, 0.1, 13), (1, 0.3, 13), (2, 0.5, 1)],
                         ids=["blk2_q0.1_k13", "blk1_q0.3_k13", "blk2_q0.5_nopool"])
@pytest.mark.parametrize("wl", [
    synth.small_variant(synth.LONG_128K, 5003, layers=4),
    synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=2, requests=[1500, 4097, 2222]),
], ids=lambda w: w.name)
def test_block_eviction_matches_oracle(cuda_lib, wl, block_layers, q, kernel):
    import torch
    kv = cuda_lib
    run = parity.DeviceRun(kv, wl, score_rule=oracle.RULE_ATTN_SUM)
    assert run.status_score == 0
    bb = kv.BlockBuffers(run.prob, block_layers, q, pool_kernel=kernel)
    sel, k_out, v_out, offsets = kv.evict_blocks(run.prob, run.bufs.scores, run.dw.k, run.dw.v,
                                                 bb)
    torch.cuda.synchronize()
    assert kv.kv_check_status(bb.select_ws) == 0
    scores = run.bufs.scores.cpu().numpy().astype(np.float64)
    blk = bb.block_scores.cpu().numpy()[:, 0]
    pooled = bb.pooled.cpu().numpy()[:, 0] if bb.pooled is not None else blk
    sel = sel.cpu().numpy()
    ko = k_out.cpu().view(torch.int16).numpy().view(np.uint16)
    vo = v_out.cpu().view(torch.int16).numpy().view(np.uint16)
    cu = run.dw.cu_host
    L, H, w, s = wl.num_layers, wl.num_kv_heads, wl.window, wl.num_sinks
    nblk = L // block_layers
    for r in range(wl.num_requests):
        c0, c1 = int(cu[r]), int(cu[r + 1])
        n = c1 - c0
        for b in range(nblk):
            ub = r * nblk + b
            layers = range(b * block_layers, (b + 1) * block_layers)
            # block sums: against the GPU's own scores (fp32 sum order) and the oracle's
            g_blk = blk[b, c0:c1]
            np.testing.assert_allclose(
                g_blk, oracle.block_scores(scores[b * block_layers:(b + 1) * block_layers, :, c0:c1]),
                rtol=1e-5)
            So = oracle.block_scores(np.stack([
                np.stack([parity.oracle_unit(wl, run.dw, r, l, h, oracle.RULE_ATTN_SUM)[3]
                          for h in range(H)]) for l in layers]))
            rel = np.abs(g_blk - So) / So
            assert rel.max() <= parity.SCORE_RTOL
            # pooling bit-exact on the GPU's block scores; selection exact on the GPU's pooled
            g_pool = pooled[b, c0:c1]
            if kernel > 1:
                np.testing.assert_array_equal(g_pool, oracle.pool_unit(g_blk.astype(np.float64),
                                                                       w, kernel))
            budget = oracle.block_budget(n, w, s, q)
            o0, o1 = int(bb.block_offsets_host[ub]), int(bb.block_offsets_host[ub + 1])
            assert o1 - o0 == budget
            g_sel = sel[o0:o1]
            np.testing.assert_array_equal(
                g_sel, oracle.select(g_pool.astype(np.float64), w, s, budget))
            # against the oracle's own scores, differences only inside the tie band
            Sp = oracle.pool_unit(So, w, kernel) if kernel > 1 else So
            ref = oracle.select(Sp, w, s, budget)
            take = budget - s - w
            diff = set(ref.tolist()) ^ set(g_sel.tolist())
            if diff:
                mid = np.arange(s, n - w)
                theta = Sp[mid[np.lexsort((mid, -Sp[mid]))][take - 1]]
                for j in diff:
                    assert abs(Sp[j] - theta) <= parity.SCORE_RTOL * theta
            # every layer and head of the block keeps the block's tokens, bit for bit
            for l in layers:
                for h in range(H):
                    u = wl.unit_index(r, l, h)
                    a0, a1 = int(bb.unit_offsets_host[u]), int(bb.unit_offsets_host[u + 1])
                    _, k, v = run.dw.unit_host(r, l, h)
                    np.testing.assert_array_equal(ko[a0:a1], k[g_sel])
                    np.testing.assert_array_equal(vo[a0:a1], v[g_sel])


def test_block_scores_random_input(cuda_lib):
    import torch
    kv = cuda_lib
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, layers=4, requests=[700, 3001])
    prob = kv.Problem.for_workload(wl)
    g = torch.Generator(device="cuda").manual_seed(5)
    s = torch.rand((wl.num_layers, wl.num_kv_heads, prob.total_tokens), generator=g,
                   device="cuda")
    out = torch.empty((2, 1, prob.total_tokens), device="cuda")
    kv.kv_block_scores(prob, 2, s, out)
    torch.cuda.synchronize()
    ref = s.double().reshape(2, 2 * wl.num_kv_heads, -1).sum(dim=1)
    torch.testing.assert_close(out[:, 0].double(), ref, rtol=1e-6, atol=0)


def test_block_eviction_head_dim_64(cuda_lib):
    """The d = 64 instances (pass 1, rescoring, block compaction) on a two-layer block."""
    import torch
    kv = cuda_lib
    wl = synth.TINY.scaled(name="tiny_2L_2kv_d64_n3000", num_layers=2, num_kv_heads=2,
                           num_q_heads=8, lengths=(3000,))
    run = parity.DeviceRun(kv, wl, score_rule=oracle.RULE_ATTN_SUM)
    assert run.status_score == 0
    bb = kv.BlockBuffers(run.prob, 2, 0.2, pool_kernel=13)
    sel, k_out, v_out, _ = kv.evict_blocks(run.prob, run.bufs.scores, run.dw.k, run.dw.v, bb)
    torch.cuda.synchronize()
    assert kv.kv_check_status(bb.select_ws) == 0
    sel = sel.cpu().numpy()
    ko = k_out.cpu().view(torch.int16).numpy().view(np.uint16)
    w, s, n = wl.window, wl.num_sinks, 3000
    g_pool = bb.pooled.cpu().numpy()[0, 0].astype(np.float64)
    np.testing.assert_array_equal(sel, oracle.select(g_pool, w, s, oracle.block_budget(n, w, s, 0.2)))
    for l in range(2):
        for h in range(2):
            u = wl.unit_index(0, l, h)
            a0, a1 = int(bb.unit_offsets_host[u]), int(bb.unit_offsets_host[u + 1])
            _, k, _ = run.dw.unit_host(0, l, h)
            np.testing.assert_array_equal(ko[a0:a1], k[sel])
