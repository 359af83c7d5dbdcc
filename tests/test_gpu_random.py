"""Seeded random shapes: the whole path against the oracle, and the fused launch against
the separate calls, over problem shapes the named workloads do not reach.

Each case draws (from its own seed, so the list is fixed) the head dim, KV heads, GQA group
and window -- window-row counts G*w from 1 to 512, including counts below one 32-row MMA
group and odd windows -- the layers, one to three requests whose lengths go down to
sinks + window, a budget per (request, layer, head) anywhere in [sinks + window, n], and
the score rule.  Every unit is compared with the oracle (parity.check_units), and the
fused launch must reproduce every output of the separate calls bit for bit.
"""
import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = 64


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice([64, 128]))
    H = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 3, 4, 7, 8]))
    w = int(rng.integers(1, 65))
    while G * w > 512:
        w //= 2
    L = int(rng.choice([1, 2]))
    R = int(rng.integers(1, 4))
    s = 4
    lengths = []
    for _ in range(R):
        lo = s + w
        lengths.append(int(lo if rng.random() < 0.2 else rng.integers(lo, 2600)))
    rule = int(rng.choice([0, 1, 2]))
    budgets = np.zeros((R, L, H), dtype=np.int32)
    for r, n in enumerate(lengths):
        budgets[r] = rng.integers(s + w, n + 1, size=(L, H))
    wl = synth.TINY.scaled(
        name="rand%02d_d%d_h%d_g%d_w%d_l%d_r%d_rule%d" % (seed, d, H, G, w, L, R, rule),
        num_layers=L, num_kv_heads=H, num_q_heads=H * G, head_dim=d, window=w,
        lengths=tuple(lengths), ragged_range=None, num_sinks=s, seed=2000 + seed,
        num_heavy=0 if min(lengths) < 200 else 4, budget_tokens=None, budget_ratio=0.1)
    return wl, budgets, rule


@pytest.mark.parametrize("seed", range(CASES))
def test_random_shapes(cuda_lib, seed):
    import torch
    wl, budgets, rule = _case(seed)
    sep = parity.DeviceRun(cuda_lib, wl, budgets=budgets, score_rule=rule)
    assert sep.status_score == 0 and sep.status_select == 0, wl.name
    res = parity.check_units(sep, list(range(wl.num_units)))
    assert max(r["max_rel"] for r in res.values()) <= parity.SCORE_RTOL, wl.name
    fus = parity.DeviceRun(cuda_lib, wl, budgets=budgets, dw=sep.dw, score_rule=rule,
                           fused=True)
    assert fus.status_score == 0, wl.name
    n = sep.bufs.total_rows
    assert torch.equal(sep.bufs.scores.view(torch.int32), fus.bufs.scores.view(torch.int32))
    assert torch.equal(sep.bufs.sel[:n], fus.bufs.sel[:n])
    assert torch.equal(sep.bufs.k_out[:n].view(torch.int16), fus.bufs.k_out[:n].view(torch.int16))
    assert torch.equal(sep.bufs.v_out[:n].view(torch.int16), fus.bufs.v_out[:n].view(torch.int16))


@pytest.mark.parametrize("seed", range(0, CASES, 2))
def test_random_shapes_pooling_and_head_budgets(cuda_lib, seed):
    """The same shapes with max pooling of a random odd width before the selection and, on
    every other case, per-head budgets: pooled scores, the heads' budgets (against the
    oracle's allocation over the GPU's ranked scores), selection and compaction."""
    import oracle
    wl, budgets, rule = _case(seed)
    rng = np.random.default_rng(5000 + seed)
    kernel = int(rng.choice([1, 3, 5, 11, 13, 31]))
    heads = bool(seed % 4 == 0)
    run = parity.DeviceRun(cuda_lib, wl, budgets=budgets, score_rule=rule, pool_kernel=kernel,
                           head_budgets=heads)
    assert run.status_score == 0 and run.status_select == 0, wl.name
    if heads:
        ranked = run.ranked_scores()
        H, w, s = wl.num_kv_heads, wl.window, wl.num_sinks
        inb = np.asarray(budgets).reshape(-1)
        cu = run.dw.cu_host
        for r in range(wl.num_requests):
            for l in range(wl.num_layers):
                u0 = wl.unit_index(r, l, 0)
                S = ranked[l, :, int(cu[r]):int(cu[r + 1])].astype(np.float64)
                want = oracle.head_budgets(S, w, s, inb[u0:u0 + H])
                np.testing.assert_array_equal(run.eff_budgets[u0:u0 + H], want, err_msg=wl.name)
        np.testing.assert_array_equal(run.eff_offsets, oracle.offsets(run.eff_budgets))
    parity.check_units(run, list(range(wl.num_units)))
