"""Plain fp64 CPU oracle of the KV-cache eviction path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``kv_cache_eviction_split_gb300``) never does, and this
package imports nothing from it.

* ``oracle.c`` (compiled here with gcc) holds the window attention, the
  DropKV removal score and the budgeted selection of one unit, in fp64.
* This file adds the ctypes wrapper, the per-layer budget policies (plain
  Python ``math`` in fp64) and the offsets scan and gather of the compaction,
  which are plain numpy indexing.

Every function cites the passage it follows.  Parity of each function is
pinned by ``tests/test_oracle_pins.py`` against brute force, closed forms and
invariants that the pages and the mathematics fix.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_liboracle.so`` (plain gcc, no fused multiply-add)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or \
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC",
                                   "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        ci = ctypes.c_int
        lib.oracle_window_attention.argtypes = [ci, ci, ci, ci, ctypes.c_double, u16p, u16p,
                                                u16p, f64p, f64p, f64p]
        lib.oracle_unit_scores.argtypes = [ci, ci, ci, ci, ctypes.c_double, u16p, u16p, u16p,
                                           f64p]
        lib.oracle_select.argtypes = [ci, ci, ci, ci, f64p, i32p]
        lib.oracle_unit_scores_rule.argtypes = [ci, ci, ci, ci, ctypes.c_double, ci, u16p, u16p,
                                                u16p, f64p]
        lib.oracle_max_pool.argtypes = [ci, ci, f64p, f64p]
        for f in (lib.oracle_window_attention, lib.oracle_unit_scores, lib.oracle_select):
            f.restype = ci
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _unit_args(q, k, v):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    n, d = k.shape
    assert v.shape == (n, d) and q.shape[-1] == d
    return q, k, v, n, d


def window_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, G: int, w: int,
                     scale: float | None = None):
    """Causal window attention of one unit (DropKV, "Methodology in Plain English").

    q: bf16 bits [G*w][d] (or [G][w][d]); k, v: bf16 bits [n][d].
    Returns (m[R], l[R], a[R][d]) in fp64 with m the logit row max and
    l = sum_j exp(s_j - m).
    """
    q, k, v, n, d = _unit_args(q, k, v)
    R = G * w
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    m = np.zeros(R)
    l = np.zeros(R)
    a = np.zeros((R, d))
    rc = _load().oracle_window_attention(n, d, G, w, scale, _ptr(q, ctypes.c_uint16),
                                         _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                                         _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double),
                                         _ptr(a, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_window_attention failed (%d)" % rc)
    return m, l, a


def unit_scores(q: np.ndarray, k: np.ndarray, v: np.ndarray, G: int, w: int,
                scale: float | None = None) -> np.ndarray:
    """DropKV removal score of every key of one unit, fp64 [n].

    S_j = sum over the G*w window rows that see j of p/(1-p) * ||a - v_j||_2
    (DropKV, "Key Contributions" 1; the unsquared sum over the window and the
    GQA group is the aggregation this implementation fixes).
    """
    q, k, v, n, d = _unit_args(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    S = np.zeros(n)
    rc = _load().oracle_unit_scores(n, d, G, w, scale, _ptr(q, ctypes.c_uint16),
                                    _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                                    _ptr(S, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_unit_scores failed (%d)" % rc)
    return S


# aggregation rules: 0 = DropKV removal score (unit_scores), 1 = its squared form,
# 2 = attention sum
RULE_DROPKV, RULE_DROPKV_SQUARED, RULE_ATTN_SUM = 0, 1, 2


def unit_scores_rule(q: np.ndarray, k: np.ndarray, v: np.ndarray, G: int, w: int, rule: int,
                     scale: float | None = None) -> np.ndarray:
    """Score of every key of one unit under `rule`, fp64 [n].

    rule 0: unit_scores.  rule 1: sum over the window rows of (p/(1-p))^2 *
    ||a - v_j||^2 (DropKV, "Methodology in Plain English": accumulated over the
    window and squared).  rule 2: sum of p over the window rows and heads
    (PyramidKV guide, "Observation Window and Aggregated Attention Eviction").
    """
    if rule == RULE_DROPKV:
        return unit_scores(q, k, v, G, w, scale)
    q, k, v, n, d = _unit_args(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    S = np.zeros(n)
    rc = _load().oracle_unit_scores_rule(n, d, G, w, scale, int(rule), _ptr(q, ctypes.c_uint16),
                                         _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                                         _ptr(S, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_unit_scores_rule failed (%d)" % rc)
    return S


def max_pool(S: np.ndarray, kernel: int) -> np.ndarray:
    """out[j] = max of S over the `kernel` positions centred on j, clipped to the unit
    (DropKV page: kernel 11; BellowsKV blog: 13)."""
    S = np.ascontiguousarray(S, dtype=np.float64)
    out = np.empty_like(S)
    rc = _load().oracle_max_pool(S.shape[0], int(kernel), _ptr(S, ctypes.c_double),
                                 _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_max_pool failed (%d)" % rc)
    return out


def pool_unit(S: np.ndarray, w: int, kernel: int) -> np.ndarray:
    """Pooling of one unit's scores in the SnapKV convention the DropKV page follows: the
    keys outside the observation window, [0, n - w), are max-pooled among themselves; the
    w window keys (kept by selection anyway) are copied."""
    S = np.asarray(S, dtype=np.float64)
    out = S.copy()
    c = S.shape[0] - w
    if c > 0:
        out[:c] = max_pool(S[:c], kernel)
    return out


def select(S: np.ndarray, w: int, sinks: int, b: int) -> np.ndarray:
    """Kept indices of one unit, ascending int32 [b] (sinks + top middle + window)."""
    S = np.ascontiguousarray(S, dtype=np.float64)
    n = S.shape[0]
    out = np.zeros(b, dtype=np.int32)
    rc = _load().oracle_select(n, w, sinks, b, _ptr(S, ctypes.c_double),
                               _ptr(out, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle_select: inconsistent sizes n=%d w=%d sinks=%d b=%d"
                         % (n, w, sinks, b))
    return out


# --------------------------------------------------------------------------
# per-layer budgets
# --------------------------------------------------------------------------
def _plain_sum(xs) -> float:
    """Left-to-right float sum (Python's ``sum`` compensates rounding since 3.12)."""
    acc = 0.0
    for t in xs:
        acc += t
    return acc


def largest_remainder(L: int, B: int, mult: list) -> list:
    """Integer budgets b_l close to B*m_l with sum exactly L*B.

    RippleKV, Eq. (5) requires the layer budgets to sum to the global budget;
    Eq. (12) rounds each B*w_l, which can miss that sum.  Reading taken here:
    floor every B*m_l, then give one more token to the layers with the
    largest fractional parts (ties to the lower layer) until the sum is L*B.
    """
    x = [B * m for m in mult]
    f = [math.floor(t) for t in x]
    deficit = L * B - sum(f)
    if deficit < 0 or deficit > L:
        raise ValueError("multipliers do not average to one")
    order = sorted(range(L), key=lambda i: (-(x[i] - f[i]), i))
    for i in order[:deficit]:
        f[i] += 1
    return [int(t) for t in f]


def budgets_uniform(L: int, B: int) -> list:
    """Uniform allocation: every layer keeps B tokens per head."""
    return [int(B)] * L


def pyramid_multipliers(L: int, hi: float = 1.8, lo: float = 0.2, gamma: float = 1.0) -> list:
    """PyramidKV blog, "Layer-Adaptive Dynamic Budget Allocation":
    C_l = C_min + (C_max - C_min) * (1 - (l-1)/(L-1))**gamma for 1-based l;
    written here 0-based as multipliers of the mean, rescaled to mean one."""
    if L == 1:
        return [1.0]
    raw = [lo + (hi - lo) * (1.0 - l / (L - 1)) ** gamma for l in range(L)]
    mean = _plain_sum(raw) / L
    return [t / mean for t in raw]


def budgets_pyramid(L: int, B: int, hi: float = 1.8, lo: float = 0.2, gamma: float = 1.0) -> list:
    return largest_remainder(L, B, pyramid_multipliers(L, hi, lo, gamma))


def ripple_multipliers(profile, beta: float = 2.0, gamma: float = math.inf) -> list:
    """RippleKV, Eq. (9)-(11):
    s_hat = (s - min) / (max - min) (all zero for a constant profile, Eq. (9));
    w~ = exp(log r * s_hat) with log r = beta (Eq. (10));
    ClipNormalize: clip to [1/gamma, gamma], then rescale to mean one (Eq. (11))."""
    s = [float(t) for t in profile]
    L = len(s)
    smin, smax = min(s), max(s)
    if smax == smin:
        shat = [0.0] * L
    else:
        shat = [(t - smin) / (smax - smin) for t in s]
    wt = [math.exp(beta * t) for t in shat]
    if math.isfinite(gamma):
        wt = [min(max(t, 1.0 / gamma), gamma) for t in wt]
    mean = _plain_sum(wt) / L
    return [t / mean for t in wt]


def budgets_ripple(L: int, B: int, profile, beta: float = 2.0, gamma: float = math.inf) -> list:
    """RippleKV, Eq. (12) with the exact-sum rounding of ``largest_remainder``."""
    return largest_remainder(L, B, ripple_multipliers(profile, beta, gamma))


def segment_budgets(wl, profile=None) -> np.ndarray:
    """int32 [req][L][H] budgets of a synthetic workload (uniform over KV heads)."""
    L, H = wl.num_layers, wl.num_kv_heads
    out = []
    for B in wl.mean_budgets():
        if wl.budget_policy == "uniform":
            bl = budgets_uniform(L, B)
        elif wl.budget_policy == "pyramid":
            bl = budgets_pyramid(L, B, wl.pyramid_max, wl.pyramid_min)
        elif wl.budget_policy == "ripple":
            bl = budgets_ripple(L, B, profile, wl.ripple_beta)
        else:
            raise ValueError(wl.budget_policy)
        out.append([[b] * H for b in bl])
    return np.asarray(out, dtype=np.int32)


def offsets(budgets: np.ndarray) -> np.ndarray:
    """Exclusive scan of the segment budgets (GraceKV "physical cache packing":
    one independent length per layer-KV-head), int64 [segments + 1]."""
    b = np.asarray(budgets, dtype=np.int64).reshape(-1)
    return np.concatenate([[0], np.cumsum(b)]).astype(np.int64)


def compact(k: np.ndarray, v: np.ndarray, idx: np.ndarray):
    """Rows of k and v at the kept indices (a plain gather of the bf16 bits)."""
    return k[idx], v[idx]


# --------------------------------------------------------------------------
# per-head budgets (AdaDropKV) and block eviction (BellowsKV)
# --------------------------------------------------------------------------
def head_budgets(S_heads: np.ndarray, w: int, sinks: int, b_heads) -> np.ndarray:
    """Per-head budgets of one (request, layer), int32 [H].

    DropKV page, Key Contributions ("Adaptive head budgets"): DropKV scores with
    AdaKV's head budget allocation.  Reading: the layer keeps sum(b_heads) tokens;
    every head keeps its sinks and window, and the remaining slots go to the
    largest middle-candidate scores [sinks, n - w) over all heads together, equal
    scores to the lower head, then the lower index.  A head's budget is its sinks
    + window + the slots it won.
    """
    S = np.asarray(S_heads, dtype=np.float64)
    H, n = S.shape
    b_heads = [int(b) for b in b_heads]
    if len(b_heads) != H or any(b < sinks + w or b > n for b in b_heads):
        raise ValueError("head_budgets: budgets outside [sinks + w, n]")
    k = sum(b_heads) - H * (sinks + w)
    mid = np.arange(sinks, n - w)
    vals = S[:, sinks:n - w].reshape(-1)
    hh = np.repeat(np.arange(H), mid.size)
    jj = np.tile(mid, H)
    order = np.lexsort((jj, hh, -vals))          # score desc, then head, then index
    counts = np.bincount(hh[order[:k]], minlength=H)
    return (sinks + w + counts).astype(np.int32)


def block_scores(S_block: np.ndarray) -> np.ndarray:
    """BellowsKV blog, eviction operator: a token's block score is its score summed
    over all layers and heads of the block.  S_block [layers][heads][n] -> [n]."""
    S = np.asarray(S_block, dtype=np.float64)
    return S.reshape(-1, S.shape[-1]).sum(axis=0)


def block_budget(n: int, w: int, sinks: int, q: float) -> int:
    """BellowsKV blog, eviction operator: the first `sinks` and last `w` positions
    are kept, and the fraction q of the remaining positions with the highest
    scores survives (rounded down)."""
    return sinks + w + int(math.floor(q * (n - sinks - w)))
