"""GPU-vs-oracle parity harness used by the ``-m gpu`` tests.

Runs the CUDA path through the C ABI on a device-generated workload and
compares, unit by unit, against the fp64 oracle run on inputs regenerated on
the host from the same seed (no oracle input is read back from the GPU):

* scores: |gpu - oracle| <= 1e-3 * oracle elementwise (relative), or
  <= 1e-30 absolute where the oracle score is below 1e-30;
* selection: exact equality with the oracle's selection rule applied to the
  GPU's own scores, and equality with the oracle's selection on oracle scores
  except for tokens within 1e-3 relative of the oracle's k-th score;
* compaction: the packed rows equal the input rows at the GPU's indices, bit
  for bit;
* pooling (when a pool kernel is set): the pooled scores equal the oracle's
  pooling of the GPU's own raw scores bit for bit (a max of fp32 values is
  exact), and the oracle's pooling of oracle scores within the score
  tolerance; selection is then checked on the pooled scores.

Every score rule is checked the same way against oracle.unit_scores_rule.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle
import synth

SCORE_RTOL = 1e-3
SCORE_ATOL = 1e-30


def product_budgets(kv, wl, profile=None) -> np.ndarray:
    """int32 [req][L][H] from the library's host budget helpers."""
    L, H = wl.num_layers, wl.num_kv_heads
    rows = []
    for B in wl.mean_budgets():
        if wl.budget_policy == "uniform":
            bl = kv.kv_budgets_uniform(L, B)
        elif wl.budget_policy == "pyramid":
            bl = kv.kv_budgets_pyramid(L, B, wl.pyramid_max, wl.pyramid_min)
        else:
            bl = kv.kv_budgets_ripple(L, B, profile, wl.ripple_beta)
        rows.append(np.repeat(np.asarray(bl, np.int32)[:, None], H, axis=1))
    return np.asarray(rows, dtype=np.int32)


class DeviceRun:
    """The three C-ABI calls (or, with fused=True, kv_evict_fused) on one workload,
    results kept on the device."""

    def __init__(self, kv, wl, budgets=None, dw=None, score_rule=0, pool_kernel=1,
                 head_budgets=False, fused=False):
        import torch
        from synth.device import DeviceWorkload
        self.wl = wl
        self.rule = score_rule
        self.pool = pool_kernel
        self.dw = dw or DeviceWorkload(wl)
        self.prob = kv.Problem.for_workload(wl, score_rule=score_rule, pool_kernel=pool_kernel,
                                            head_budgets=head_budgets)
        prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
        self.profile = prof
        if budgets is None:
            budgets = product_budgets(kv, wl, prof)
        self.budgets = budgets
        self.bufs = kv.Buffers(self.prob, budgets)
        kv.evict(self.prob, self.dw.q, self.dw.k, self.dw.v, self.bufs, fused=fused)
        torch.cuda.synchronize()
        self.status_score = kv.kv_check_status(self.bufs.score_ws)
        # the fused launch posts the selection's errors to the score workspace
        self.status_select = self.status_score if fused else kv.kv_check_status(self.bufs.select_ws)
        # budgets and offsets selection and compaction used (per-head ones if computed)
        if head_budgets:
            self.eff_budgets = self.bufs.head_budgets.cpu().numpy().reshape(-1)
            self.eff_offsets = self.bufs.head_offsets.cpu().numpy()
        else:
            self.eff_budgets = np.asarray(budgets).reshape(-1)
            self.eff_offsets = self.bufs.offsets_host

    def ranked_scores(self):
        """The scores selection ranked (pooled if pooling ran), float32 [L][H][N]."""
        b = self.bufs
        return (b.pooled if b.pooled is not None else b.scores).cpu().numpy()

    def unit_results(self, r, l, h):
        wl, b = self.wl, self.bufs
        cu = self.dw.cu_host
        u = wl.unit_index(r, l, h)
        n = int(cu[r + 1] - cu[r])
        scores = b.scores[l, h, int(cu[r]):int(cu[r + 1])].cpu().numpy()
        if b.pooled is not None:
            pooled = b.pooled[l, h, int(cu[r]):int(cu[r + 1])].cpu().numpy()
            scores = (scores, pooled)
        o0, o1 = int(self.eff_offsets[u]), int(self.eff_offsets[u + 1])
        sel = b.sel[o0:o1].cpu().numpy()
        kout = b.k_out[o0:o1].cpu().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        vout = b.v_out[o0:o1].cpu().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        return n, scores, sel, kout, vout, int(self.eff_budgets[u])


def oracle_unit(wl, dw, r, l, h, rule=0):
    q, k, v = dw.unit_host(r, l, h)
    S = oracle.unit_scores_rule(q, k, v, wl.group, wl.window, rule)
    return q, k, v, S


def _check_scores(g, S, what):
    big = S >= SCORE_ATOL
    rel = np.abs(g[big].astype(np.float64) - S[big]) / S[big]
    assert np.all(np.isfinite(g)), "non-finite GPU score"
    max_rel = float(rel.max()) if rel.size else 0.0
    assert max_rel <= SCORE_RTOL, "%s: score rel err %.3g" % (what, max_rel)
    assert np.all(np.abs(g[~big].astype(np.float64) - S[~big]) <= SCORE_ATOL)
    return max_rel


def check_unit(run: DeviceRun, r, l, h, oracle_out=None):
    """Asserts parity of one unit; returns a small dict of error figures."""
    wl = run.wl
    n, g_scores, g_sel, kout, vout, b = run.unit_results(r, l, h)
    q, k, v, S = oracle_out if oracle_out is not None else \
        oracle_unit(wl, run.dw, r, l, h, run.rule)
    where = "unit (%d,%d,%d)" % (r, l, h)
    # scores
    if isinstance(g_scores, tuple):
        g_raw, g_scores = g_scores
        max_rel = _check_scores(g_raw, S, where)
        np.testing.assert_array_equal(
            g_scores, oracle.pool_unit(g_raw.astype(np.float64), wl.window, run.pool),
            err_msg="%s: pooling of the GPU's own scores" % where)
        S = oracle.pool_unit(S, wl.window, run.pool)
        _check_scores(g_scores, S, where + " pooled")
    else:
        max_rel = _check_scores(g_scores, S, where)
    # selection: the GPU's rule on its own scores is exact
    mine = oracle.select(g_scores.astype(np.float64), wl.window, wl.num_sinks, b)
    np.testing.assert_array_equal(g_sel, mine, err_msg="selection rule on GPU scores")
    # selection vs oracle scores, within the tie band
    ref = oracle.select(S, wl.window, wl.num_sinks, b)
    diff = set(ref.tolist()) ^ set(g_sel.tolist())
    take = b - wl.num_sinks - wl.window
    if diff:
        assert take > 0
        mid = np.arange(wl.num_sinks, n - wl.window)
        order = mid[np.lexsort((mid, -S[mid]))]
        theta = S[order[take - 1]]
        for j in diff:
            assert abs(S[j] - theta) <= SCORE_RTOL * theta, \
                "unit (%d,%d,%d): token %d outside the tie band" % (r, l, h, j)
    # compaction: bit copy of the GPU's own indices
    np.testing.assert_array_equal(kout, k[g_sel])
    np.testing.assert_array_equal(vout, v[g_sel])
    return {"max_rel": max_rel, "swapped": len(diff) // 2}


def check_units(run: DeviceRun, units, threads=None):
    """Oracle for several units in parallel threads (ctypes releases the GIL)."""
    wl = run.wl
    threads = threads or min(len(units), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {u: ex.submit(oracle_unit, wl, run.dw, *wl.unit_coords(u), run.rule)
                for u in units}
        out = {}
        for u in units:
            out[u] = check_unit(run, *wl.unit_coords(u), oracle_out=futs[u].result())
    return out


def sample_units(wl, count, seed=1234):
    u = synth.uniform01(synth.stream_key(seed, 99), 0, 4 * count)
    picks = []
    for x in u:
        c = int(x * wl.num_units)
        if c not in picks:
            picks.append(c)
        if len(picks) == count:
            break
    return picks


def check_every_unit_select_compact(run: DeviceRun, host_rows=64, threads=None, seed=4321):
    """Selection and compaction of EVERY unit, at any size, without oracle scoring:

    * selection: equal to the oracle's selection rule (oracle.select) applied to the
      GPU's own (ranked) scores of the unit;
    * compaction: every kept row equals the row of the device K/V at the kept index
      (a torch gather, bit for bit), and `host_rows` kept rows of every unit (its
      first and last four and a seeded sample of the rest) equal the host
      regeneration of those rows from the seed (synth.kv_rows), which ties the
      device K/V to the generator.
    Returns the number of units checked."""
    import torch
    wl, b = run.wl, run.bufs
    cu = run.dw.cu_host
    L, H = wl.num_layers, wl.num_kv_heads
    units = wl.num_units
    offs = np.asarray(run.eff_offsets, dtype=np.int64)
    bud = np.asarray(run.eff_budgets, dtype=np.int64)
    total = int(offs[-1])
    ranked = (b.pooled if b.pooled is not None else b.scores)
    scores = ranked.cpu().numpy()
    sel = b.sel[:total].cpu().numpy()

    def one_select(u):
        r, l, h = wl.unit_coords(u)
        g = scores[l, h, int(cu[r]):int(cu[r + 1])].astype(np.float64)
        mine = oracle.select(g, wl.window, wl.num_sinks, int(bud[u]))
        got = sel[offs[u]:offs[u + 1]]
        if not np.array_equal(got, mine):
            raise AssertionError("unit %d (%d,%d,%d): selection differs from the oracle's "
                                 "rule on the GPU's scores" % (u, r, l, h))
        return True

    threads = threads or min(32, os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        assert all(ex.map(one_select, range(units)))

    # every kept row against the device K/V, gathered by torch on the device
    dev = b.sel.device
    N_tot = int(cu[-1])
    r_of = np.repeat(np.arange(wl.num_requests), L * H)
    lh = np.tile(np.arange(L * H), wl.num_requests)
    row0 = lh * N_tot + cu[r_of]                       # first K/V row of each unit
    counts = torch.from_numpy(offs[1:] - offs[:-1]).to(dev)
    base = torch.repeat_interleave(torch.from_numpy(row0).to(dev), counts)
    idx = base + b.sel[:total].long()
    d = wl.head_dim
    kf = run.dw.k.reshape(-1, d)
    vf = run.dw.v.reshape(-1, d)
    as16 = lambda t: t.view(torch.int16)
    assert torch.equal(as16(kf[idx]), as16(b.k_out[:total])), "compacted K differs from K[sel]"
    assert torch.equal(as16(vf[idx]), as16(b.v_out[:total])), "compacted V differs from V[sel]"

    # a sample of kept rows of every unit against the host generator
    outl = synth.outlier_channels(wl)
    hp = synth.heavy_positions(wl)
    hv = synth.heavy_rows(wl, synth.q_window(wl)) if wl.num_heavy else None
    picks = []
    for u in range(units):
        n_u = int(bud[u])
        if n_u <= host_rows:
            pos = np.arange(n_u)
        else:
            rng = synth.uniform01(synth.stream_key(seed, u), 0, host_rows)
            mid = 4 + np.floor(rng * (n_u - 8)).astype(np.int64)
            pos = np.unique(np.concatenate([np.arange(4), np.arange(n_u - 4, n_u),
                                            mid[:host_rows - 8]]))
        picks.append(pos)
    flat = torch.from_numpy(np.concatenate([offs[u] + picks[u] for u in range(units)])).to(dev)
    k_s = as16(b.k_out[flat]).cpu().numpy().view(np.uint16)
    v_s = as16(b.v_out[flat]).cpu().numpy().view(np.uint16)
    starts = np.concatenate([[0], np.cumsum([len(p) for p in picks])])

    def one_rows(u):
        r, l, h = wl.unit_coords(u)
        toks = sel[offs[u] + picks[u]]
        kr, vr = synth.kv_rows(wl, r, l, h, toks, outl=outl, heavy_pos=hp, heavy_vec=hv)
        a, z = starts[u], starts[u + 1]
        if not (np.array_equal(k_s[a:z], kr) and np.array_equal(v_s[a:z], vr)):
            raise AssertionError("unit %d (%d,%d,%d): compacted rows differ from the host "
                                 "generator" % (u, r, l, h))
        return True

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        assert all(ex.map(one_rows, range(units)))
    return units
