"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Nothing here re-types the oracle's own formula: the score is checked against
a brute-force recomputation of attention with each token deleted (the
definition the DropKV page derives its closed form from), against a hand
closed form for two keys, and against invariants (softmax rows sum to one,
causality).  Selection is checked against a brute-force sort and its
invariants; budgets against the sums and ratios RippleKV and PyramidKV state.
The squared and attention-sum aggregation rules are checked against literal
token deletion and a direct softmax, closed forms and the row-sum invariant;
max pooling against a sliding-window brute force and scipy's maximum filter.
A final group compiles mutated copies of the oracle (a dropped factor, a
squared norm, a lost causal mask, a wrong tie-break, a short pooling window)
and checks that some pin rejects each.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synth


def _bf16(rng, shape, scale=1.0):
    return synth.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _softmax_out(qv, K, V, keys, scale):
    s = np.array([scale * float(qv @ K[j]) for j in keys])
    e = np.exp(s - s.max())
    p = e / e.sum()
    return p @ V[list(keys)], dict(zip(keys, p))


def brute_force_scores(q, k, v, G, w, scale=None):
    """sum over rows of || attention without j  -  attention with all keys ||, per j.

    DropKV, "Methodology in Plain English": deleting a token renormalises the
    softmax over the survivors; the score is the size of the resulting output
    shift.  Computed by literally deleting the token and recomputing.
    """
    Q, K, V = _f64(q).reshape(G * w, -1), _f64(k), _f64(v)
    n, d = K.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    S = np.zeros(n)
    for i in range(G * w):
        pos = n - w + i % w
        keys = list(range(pos + 1))
        a_full, _ = _softmax_out(Q[i], K, V, keys, scale)
        for j in keys:
            rest = [t for t in keys if t != j]
            a_minus, _ = _softmax_out(Q[i], K, V, rest, scale)
            S[j] += np.linalg.norm(a_minus - a_full)
    return S


# --------------------------------------------------------------------------
# score pins
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,d", [(5, 4), (17, 8), (64, 16)])
def test_single_query_removal_identity(n, d):
    """One query: the closed-form score equals the brute-force removal shift."""
    rng = np.random.default_rng(n * 31 + d)
    q, k, v = _bf16(rng, (1, d)), _bf16(rng, (n, d)), _bf16(rng, (n, d))
    S = oracle.unit_scores(q, k, v, G=1, w=1)
    ref = brute_force_scores(q, k, v, 1, 1)
    np.testing.assert_allclose(S, ref, rtol=1e-11, atol=0)


@pytest.mark.parametrize("G,w,n", [(2, 3, 11), (4, 4, 24), (3, 5, 9)])
def test_window_and_group_removal_identity(G, w, n):
    """Sum over the window rows and GQA heads, each causal, of the removal shift."""
    rng = np.random.default_rng(G * 100 + w * 10 + n)
    d = 8
    q, k, v = _bf16(rng, (G * w, d)), _bf16(rng, (n, d)), _bf16(rng, (n, d))
    S = oracle.unit_scores(q, k, v, G=G, w=w)
    ref = brute_force_scores(q, k, v, G, w)
    np.testing.assert_allclose(S, ref, rtol=1e-11, atol=0)


def test_two_key_closed_form():
    """n=2, one query: S_0 = p_0 * ||v_1 - v_0||, S_1 = p_1 * ||v_1 - v_0||.

    Derivation: a - v_0 = p_1 (v_1 - v_0), so p_0/(1-p_0) * ||a - v_0||
    = (p_0/p_1) * p_1 ||v_1 - v_0||.
    """
    rng = np.random.default_rng(5)
    d = 16
    q, k, v = _bf16(rng, (1, d)), _bf16(rng, (2, d)), _bf16(rng, (2, d))
    Q, K, V = _f64(q)[0], _f64(k), _f64(v)
    s0, s1 = (Q @ K[0]) / 4.0, (Q @ K[1]) / 4.0
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    p1 = 1.0 - p0
    gap = math.sqrt(sum((V[1, c] - V[0, c]) ** 2 for c in range(d)))
    S = oracle.unit_scores(q, k, v, G=1, w=1)
    assert S[0] == pytest.approx(p0 * gap, rel=1e-12)
    assert S[1] == pytest.approx(p1 * gap, rel=1e-12)


def test_softmax_rows_sum_to_one():
    """With every value row equal to ones, a = sum_j p_j = 1 for each row."""
    rng = np.random.default_rng(6)
    G, w, n, d = 4, 8, 300, 32
    q, k = _bf16(rng, (G * w, d), 3.0), _bf16(rng, (n, d), 3.0)
    ones = synth.f32_to_bf16_bits(np.ones((n, d), np.float32))
    m, l, a = oracle.window_attention(q, k, ones, G, w)
    np.testing.assert_allclose(a, 1.0, rtol=0, atol=1e-13)
    assert np.all(l >= 1.0 - 1e-15)
    # m is the largest causal logit of the row
    Q, K = _f64(q), _f64(k)
    for i in range(G * w):
        pos = n - w + i % w
        assert m[i] == pytest.approx((K[:pos + 1] @ Q[i]).max() / math.sqrt(d), rel=1e-14)


def test_attention_is_causal():
    """Row at window slot t never sees keys after position n - w + t."""
    rng = np.random.default_rng(7)
    G, w, n, d = 2, 6, 40, 8
    q, k, v = _bf16(rng, (G * w, d)), _bf16(rng, (n, d)), _bf16(rng, (n, d))
    _, _, a1 = oracle.window_attention(q, k, v, G, w)
    k2, v2 = k.copy(), v.copy()
    k2[n - w + 1:] = _bf16(rng, (w - 1, d), 5.0)
    v2[n - w + 1:] = _bf16(rng, (w - 1, d), 5.0)
    _, _, a2 = oracle.window_attention(q, k2, v2, G, w)
    slot0 = [i for i in range(G * w) if i % w == 0]
    np.testing.assert_array_equal(a1[slot0], a2[slot0])
    assert not np.allclose(a1, a2)


def test_attention_matches_definition():
    rng = np.random.default_rng(8)
    G, w, n, d = 3, 4, 50, 16
    q, k, v = _bf16(rng, (G * w, d)), _bf16(rng, (n, d)), _bf16(rng, (n, d))
    m, l, a = oracle.window_attention(q, k, v, G, w)
    Q, K, V = _f64(q), _f64(k), _f64(v)
    for i in range(G * w):
        pos = n - w + i % w
        ref, _ = _softmax_out(Q[i], K, V, list(range(pos + 1)), 1.0 / math.sqrt(d))
        np.testing.assert_allclose(a[i], ref, rtol=1e-12, atol=1e-15)


def test_single_visible_key_is_rejected():
    """w = n: the first window row sees one key, p = 1, the shift is unbounded."""
    rng = np.random.default_rng(9)
    q, k, v = _bf16(rng, (3, 4)), _bf16(rng, (3, 4)), _bf16(rng, (3, 4))
    with pytest.raises(ValueError):
        oracle.unit_scores(q, k, v, G=1, w=3)


# --------------------------------------------------------------------------
# pins of the other aggregation rules and of max pooling
# --------------------------------------------------------------------------
def brute_force_rule_scores(q, k, v, G, w, rule):
    """rule 1: sum over rows of the SQUARED removal shift, by literal deletion;
    rule 2: sum over rows of the softmax weight, from a direct softmax."""
    Q, K, V = _f64(q).reshape(G * w, -1), _f64(k), _f64(v)
    n, d = K.shape
    scale = 1.0 / math.sqrt(d)
    S = np.zeros(n)
    for i in range(G * w):
        pos = n - w + i % w
        keys = list(range(pos + 1))
        a_full, p = _softmax_out(Q[i], K, V, keys, scale)
        for j in keys:
            if rule == oracle.RULE_ATTN_SUM:
                S[j] += p[j]
                continue
            rest = [t for t in keys if t != j]
            a_minus, _ = _softmax_out(Q[i], K, V, rest, scale)
            S[j] += float(np.sum((a_minus - a_full) ** 2))
    return S


@pytest.mark.parametrize("rule", [oracle.RULE_DROPKV_SQUARED, oracle.RULE_ATTN_SUM])
@pytest.mark.parametrize("G,w,n", [(1, 1, 13), (2, 3, 11), (4, 4, 24)])
def test_rule_scores_match_brute_force(rule, G, w, n):
    rng = np.random.default_rng(1000 * rule + G * 100 + w * 10 + n)
    d = 8
    q, k, v = _bf16(rng, (G * w, d), 2.0), _bf16(rng, (n, d)), _bf16(rng, (n, d))
    S = oracle.unit_scores_rule(q, k, v, G=G, w=w, rule=rule)
    ref = brute_force_rule_scores(q, k, v, G, w, rule)
    np.testing.assert_allclose(S, ref, rtol=1e-10, atol=1e-300)


def test_attention_sum_totals_rows():
    """Each window row's weights sum to one, so sum_j S_j = G * w."""
    rng = np.random.default_rng(21)
    G, w, n, d = 4, 8, 300, 32
    q, k, v = _bf16(rng, (G * w, d), 3.0), _bf16(rng, (n, d), 3.0), _bf16(rng, (n, d))
    S = oracle.unit_scores_rule(q, k, v, G, w, oracle.RULE_ATTN_SUM)
    assert S.sum() == pytest.approx(G * w, rel=1e-13)
    assert np.all(S >= 0)
    # keys after the first window slot are seen by fewer rows
    assert np.all(S[n - w + 1:] <= G * 1.0 + 1e-12)


def test_rule_two_key_closed_forms():
    """n=2, one query: squared S_0 = (p_0 ||v_1 - v_0||)^2; attention sum S_0 = p_0."""
    rng = np.random.default_rng(22)
    d = 16
    q, k, v = _bf16(rng, (1, d)), _bf16(rng, (2, d)), _bf16(rng, (2, d))
    Q, K, V = _f64(q)[0], _f64(k), _f64(v)
    p0 = 1.0 / (1.0 + math.exp((Q @ K[1] - Q @ K[0]) / 4.0))
    gap2 = float(((V[1] - V[0]) ** 2).sum())
    sq = oracle.unit_scores_rule(q, k, v, 1, 1, oracle.RULE_DROPKV_SQUARED)
    at = oracle.unit_scores_rule(q, k, v, 1, 1, oracle.RULE_ATTN_SUM)
    assert sq[0] == pytest.approx(p0 * p0 * gap2, rel=1e-12)
    assert sq[1] == pytest.approx((1 - p0) ** 2 * gap2, rel=1e-12)
    assert at[0] == pytest.approx(p0, rel=1e-13) and at[1] == pytest.approx(1 - p0, rel=1e-12)


def test_squared_rule_ranks_like_dropkv_for_one_row():
    """One row: the squared rule is the DropKV score squared, so the ranking is the same."""
    rng = np.random.default_rng(23)
    n, d = 200, 16
    q, k, v = _bf16(rng, (1, d), 2.0), _bf16(rng, (n, d)), _bf16(rng, (n, d))
    base = oracle.unit_scores(q, k, v, 1, 1)
    sq = oracle.unit_scores_rule(q, k, v, 1, 1, oracle.RULE_DROPKV_SQUARED)
    np.testing.assert_allclose(sq, base ** 2, rtol=1e-12)
    assert list(oracle.select(sq, 1, 4, 50)) == list(oracle.select(base, 1, 4, 50))


def test_squared_rule_rejects_single_visible_key():
    rng = np.random.default_rng(24)
    q, k, v = _bf16(rng, (3, 4)), _bf16(rng, (3, 4)), _bf16(rng, (3, 4))
    with pytest.raises(ValueError):
        oracle.unit_scores_rule(q, k, v, 1, 3, oracle.RULE_DROPKV_SQUARED)
    # the attention sum has no 1 - p and is defined there
    S = oracle.unit_scores_rule(q, k, v, 1, 3, oracle.RULE_ATTN_SUM)
    assert S.sum() == pytest.approx(3.0, rel=1e-14)


@pytest.mark.parametrize("n,kernel", [(1, 1), (1, 13), (5, 3), (40, 11), (40, 13), (97, 7)])
def test_max_pool_matches_brute_force(n, kernel):
    rng = np.random.default_rng(n * 7 + kernel)
    S = rng.standard_normal(n)
    r = kernel // 2
    ref = np.array([S[max(0, j - r):j + r + 1].max() for j in range(n)])
    np.testing.assert_array_equal(oracle.max_pool(S, kernel), ref)


def test_max_pool_library_and_special_cases():
    """Agrees with scipy's maximum filter (edge padding repeats a value already in the
    clipped window); kernel 1 is the identity; a kernel wider than 2n-1 is the global max."""
    scipy_nd = pytest.importorskip("scipy.ndimage")
    rng = np.random.default_rng(25)
    S = rng.standard_normal(300)
    for kernel in (3, 11, 13):
        np.testing.assert_array_equal(oracle.max_pool(S, kernel),
                                      scipy_nd.maximum_filter1d(S, kernel, mode="nearest"))
    np.testing.assert_array_equal(oracle.max_pool(S, 1), S)
    np.testing.assert_array_equal(oracle.max_pool(S[:20], 41), np.full(20, S[:20].max()))
    with pytest.raises(ValueError):
        oracle.max_pool(S, 4)


def test_pool_unit_keeps_window_out_of_the_pool():
    """The window keys are copied and never raise a candidate's pooled score."""
    S = np.zeros(30)
    S[25:] = 100.0          # window w = 5, large scores
    S[3] = 2.0
    out = oracle.pool_unit(S, 5, 11)
    np.testing.assert_array_equal(out[25:], S[25:])
    np.testing.assert_array_equal(out[:9], 2.0)        # 3 +- 5, clipped at 0
    np.testing.assert_array_equal(out[9:25], 0.0)      # nothing leaks from the window
    np.testing.assert_array_equal(oracle.pool_unit(S[:5], 5, 11), S[:5])   # no candidates


# --------------------------------------------------------------------------
# per-head budgets (AdaDropKV) and block eviction (BellowsKV) pins
# --------------------------------------------------------------------------
def brute_head_budgets(S, w, sinks, b_heads):
    """Picks the k layer-wide winners one at a time: the largest remaining middle score,
    ties to the lower head, then the lower index."""
    H, n = S.shape
    k = sum(b_heads) - H * (sinks + w)
    taken = set()
    counts = [0] * H
    for _ in range(k):
        best = None
        for h in range(H):
            for j in range(sinks, n - w):
                if (h, j) in taken:
                    continue
                if best is None or S[h, j] > S[best] or (S[h, j] == S[best] and (h, j) < best):
                    best = (h, j)
        taken.add(best)
        counts[best[0]] += 1
    return [sinks + w + c for c in counts], taken


@pytest.mark.parametrize("H,n,w,sinks,b", [(4, 40, 4, 4, 12), (3, 25, 2, 0, 10), (2, 30, 8, 4, 30),
                                           (5, 17, 1, 4, 5), (1, 50, 4, 4, 20)])
def test_head_budgets_match_brute_force(H, n, w, sinks, b):
    rng = np.random.default_rng(H * 1000 + n)
    S = rng.integers(0, 5, (H, n)).astype(np.float64)      # many cross-head ties
    got = oracle.head_budgets(S, w, sinks, [b] * H)
    ref, taken = brute_head_budgets(S, w, sinks, [b] * H)
    assert list(got) == ref
    assert int(got.sum()) == H * b and got.min() >= sinks + w and got.max() <= n
    # each head's own top-b_h selection is exactly the head's share of the layer winners
    for h in range(H):
        sel = set(oracle.select(S[h], w, sinks, int(got[h])).tolist())
        mid = {j for j in sel if sinks <= j < n - w}
        assert mid == {j for (hh, j) in taken if hh == h}


def test_head_budgets_special_cases():
    # one head: nothing to redistribute
    S = np.random.default_rng(1).random((1, 64))
    assert list(oracle.head_budgets(S, 8, 4, [30])) == [30]
    # equal scores everywhere: the lower heads win the ties and fill up first
    S = np.ones((3, 20))
    assert list(oracle.head_budgets(S, 2, 2, [10, 10, 10])) == [20, 6, 4]
    # a head whose every candidate beats the others takes all it can
    S = np.zeros((2, 30))
    S[1] = 1.0
    assert list(oracle.head_budgets(S, 4, 4, [12, 12])) == [8, 16]
    with pytest.raises(ValueError):
        oracle.head_budgets(S, 4, 4, [7, 12])


def test_block_scores_and_budget():
    rng = np.random.default_rng(3)
    S = rng.random((2, 3, 50))
    np.testing.assert_allclose(oracle.block_scores(S), S[0].sum(0) + S[1].sum(0), rtol=1e-15)
    assert oracle.block_budget(1000, 64, 4, 0.1) == 4 + 64 + 93   # floor(0.1 * 932)
    assert oracle.block_budget(68, 64, 4, 0.5) == 68
    assert oracle.block_budget(1000, 64, 4, 1.0) == 1000


# --------------------------------------------------------------------------
# selection pins
# --------------------------------------------------------------------------
def brute_select(S, w, sinks, b):
    n = len(S)
    mid = sorted(range(sinks, n - w), key=lambda j: (-S[j], j))[: b - sinks - w]
    return sorted(list(range(sinks)) + mid + list(range(n - w, n)))


@pytest.mark.parametrize("n,w,sinks,b", [(100, 8, 4, 30), (50, 4, 4, 8), (50, 4, 4, 50),
                                         (9, 5, 4, 9), (64, 16, 4, 20), (33, 1, 0, 7)])
def test_select_matches_brute_force(n, w, sinks, b):
    rng = np.random.default_rng(n + b)
    S = rng.integers(0, 6, n).astype(np.float64)  # many ties
    got = oracle.select(S, w, sinks, b)
    assert list(got) == brute_select(S, w, sinks, b)
    assert len(got) == b and np.all(np.diff(got) > 0)
    assert set(range(sinks)) <= set(got) and set(range(n - w, n)) <= set(got)


def test_select_tie_break_lower_index():
    S = np.zeros(20)
    S[[6, 9, 12]] = 1.0
    got = oracle.select(S, w=2, sinks=4, b=4 + 2 + 5)
    # three ones, then the two lowest-index zeros of the middle [4, 18)
    assert list(got) == [0, 1, 2, 3, 4, 5, 6, 9, 12, 18, 19]


def test_select_rejects_small_budget():
    with pytest.raises(ValueError):
        oracle.select(np.zeros(40), w=8, sinks=4, b=11)
    with pytest.raises(ValueError):
        oracle.select(np.zeros(40), w=8, sinks=4, b=41)


# --------------------------------------------------------------------------
# budget pins
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L,B", [(32, 13107), (28, 6553), (1, 256), (2, 100), (80, 999)])
def test_budgets_sum_to_L_times_B(L, B):
    """RippleKV Eq. (5): the layer budgets sum to the global budget."""
    prof = synth.ripple_profile(synth.QWEN7B_128K.scaled(num_layers=L))
    for b in (oracle.budgets_uniform(L, B), oracle.budgets_pyramid(L, B),
              oracle.budgets_ripple(L, B, prof, 2.0), oracle.budgets_ripple(L, B, prof, 0.7, 1.5)):
        assert sum(b) == L * B and len(b) == L


def test_pyramid_is_linear_from_1p8_to_0p2():
    m = oracle.pyramid_multipliers(32)
    assert m[0] == pytest.approx(1.8, rel=1e-14) and m[-1] == pytest.approx(0.2, rel=1e-13)
    assert sum(m) / 32 == pytest.approx(1.0, rel=1e-15)
    steps = np.diff(m)
    np.testing.assert_allclose(steps, -1.6 / 31, rtol=1e-12)
    b = oracle.budgets_pyramid(32, 13107)
    assert all(x > y for x, y in zip(b, b[1:]))
    assert abs(b[0] - 1.8 * 13107) < 1 and abs(b[-1] - 0.2 * 13107) < 1


def test_ripple_ratio_is_r():
    """RippleKV after Eq. (10): max/min multiplier before clipping is exactly r = e^beta."""
    prof = synth.ripple_profile(synth.QWEN7B_128K)
    for beta in (0.5, 2.0, math.log(1.5)):
        m = oracle.ripple_multipliers(prof, beta)
        assert max(m) / min(m) == pytest.approx(math.exp(beta), rel=1e-13)
        assert sum(m) / len(m) == pytest.approx(1.0, rel=1e-14)
        # monotone in the profile
        order = np.argsort(prof)
        assert np.all(np.diff(np.asarray(m)[order]) >= -1e-15)


def test_ripple_special_cases():
    """Eq. (9): constant profile -> uniform; r = 1 -> uniform; invariant to s -> a*s + c."""
    L, B = 28, 6553
    assert oracle.budgets_ripple(L, B, [0.3] * L, 2.0) == [B] * L
    prof = synth.ripple_profile(synth.QWEN7B_128K)
    assert oracle.budgets_ripple(L, B, prof, 0.0) == [B] * L
    np.testing.assert_allclose(oracle.ripple_multipliers(prof * 3.5 + 7.0, 2.0),
                               oracle.ripple_multipliers(prof, 2.0), rtol=1e-13)


def test_ripple_clip_bounds():
    """Eq. (11): with gamma finite, pre-normalisation multipliers lie in [1/gamma, gamma]."""
    prof = synth.ripple_profile(synth.QWEN7B_128K)
    m = oracle.ripple_multipliers(prof, 3.0, gamma=4.0)
    scale = max(m) / 4.0   # the largest was clipped to gamma
    assert min(m) / scale >= 1.0 - 1e-12


def test_ripple_profile_is_non_monotonic():
    s = synth.ripple_profile(synth.QWEN7B_128K)
    interior_max = any(s[i] > s[i - 1] and s[i] > s[i + 1] for i in range(1, len(s) - 1))
    assert interior_max and np.argmax(s) not in (0, len(s) - 1)


def test_largest_remainder_close_to_real():
    mult = oracle.pyramid_multipliers(32)
    b = oracle.largest_remainder(32, 1638, mult)
    assert all(abs(bi - 1638 * m) < 1 for bi, m in zip(b, mult))


def test_offsets_is_exclusive_scan():
    o = oracle.offsets(np.array([[3, 4], [5, 6]]))
    assert list(o) == [0, 3, 7, 12, 18]


# --------------------------------------------------------------------------
# planted mistakes: each mutated oracle must fail one of the pins above
# --------------------------------------------------------------------------
MUTATIONS = {
    "drop_1_minus_p": ("S[j] += p / (1.0 - p) * sqrt(dist2);", "S[j] += p * sqrt(dist2);"),
    "squared_norm": ("S[j] += p / (1.0 - p) * sqrt(dist2);", "S[j] += p / (1.0 - p) * dist2;"),
    "not_causal": ("const int pos = n - w + (i % w);\n        const uint16_t *qrow = q + (size_t)i * d;\n        const double mx = row_logits(pos, d, scale, qrow, k, s);\n        double sum = 0.0;\n        for (int j = 0; j <= pos; ++j) {\n            s[j] = exp(s[j] - mx);\n            sum += s[j];\n        }\n        for (int c = 0; c < d; ++c) a[c] = 0.0;",
                   "const int pos = n - 1;\n        const uint16_t *qrow = q + (size_t)i * d;\n        const double mx = row_logits(pos, d, scale, qrow, k, s);\n        double sum = 0.0;\n        for (int j = 0; j <= pos; ++j) {\n            s[j] = exp(s[j] - mx);\n            sum += s[j];\n        }\n        for (int c = 0; c < d; ++c) a[c] = 0.0;"),
    "tie_to_higher_index": ("return (a->idx > b->idx) - (a->idx < b->idx);",
                            "return (a->idx < b->idx) - (a->idx > b->idx);"),
    "sign_of_v": ("const double diff = a[c] - bf16_value(vj[c]);\n                dist2 += diff * diff;\n            }\n            S[j] += p / (1.0 - p)",
                  "const double diff = a[c] + bf16_value(vj[c]);\n                dist2 += diff * diff;\n            }\n            S[j] += p / (1.0 - p)"),
    "squared_rule_unsquared_ratio": ("S[j] += r * r * dist2;", "S[j] += r * dist2;"),
    "squared_rule_sign_of_v": ("const double diff = a[c] - bf16_value(vj[c]);\n                dist2 += diff * diff;\n            }\n            const double r",
                               "const double diff = a[c] + bf16_value(vj[c]);\n                dist2 += diff * diff;\n            }\n            const double r"),
    "attn_sum_unnormalised": ("S[j] += s[j] / sum;", "S[j] += s[j];"),
    "pool_radius_short": ("for (int i = j - r; i <= j + r; ++i)", "for (int i = j - r; i < j + r; ++i)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path, monkeypatch):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    bad = tmp_path / "oracle.c"
    bad.write_text(src.replace(old, new))
    so = tmp_path / "_liboracle.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(bad), "-lm"])
    monkeypatch.setattr(oracle, "_LIB_PATH", str(so))
    monkeypatch.setattr(oracle, "_SRC", str(bad))
    monkeypatch.setattr(oracle, "_lib", None)
    pins = [lambda: test_single_query_removal_identity(17, 8),
            lambda: test_window_and_group_removal_identity(2, 3, 11),
            lambda: test_two_key_closed_form(),
            lambda: test_select_tie_break_lower_index(),
            lambda: test_rule_scores_match_brute_force(oracle.RULE_DROPKV_SQUARED, 2, 3, 11),
            lambda: test_rule_two_key_closed_forms(),
            lambda: test_attention_sum_totals_rows(),
            lambda: test_max_pool_matches_brute_force(40, 11)]
    failed = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            failed += 1
    monkeypatch.setattr(oracle, "_lib", None)
    assert failed >= 1, "planted mistake %r passed every pin" % name
