"""CPU checks of the C-ABI library: it builds, loads, exports every declared
symbol, and its host-side logic (argument checks, offsets, budgets) behaves.
No kernel is launched here."""
import ctypes
import math
import re

import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module")
def kv():
    import kv_cache_eviction_split_gb300 as kv
    kv.build()
    kv.load()
    return kv


def _declared_functions():
    src = open(__import__("os").path.join(__import__("os").path.dirname(__file__), "..",
                                          "include", "kvevict.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(kv):
    declared = _declared_functions()
    assert len(declared) >= 12
    lib = kv.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(kv.EXPORTED_SYMBOLS) == declared


def test_wait_limit_knob_round_trip(kv):
    default = kv.kv_get_wait_limit_ns()
    assert default == 2_000_000_000
    try:
        kv.kv_set_wait_limit_ns(12345)
        assert kv.kv_get_wait_limit_ns() == 12345
        kv.kv_set_wait_limit_ns(0)
        assert kv.kv_get_wait_limit_ns() == 0
    finally:
        kv.kv_set_wait_limit_ns(default)
    assert kv.kv_get_wait_limit_ns() == default


def _prob(kv, **kw):
    args = dict(lengths=[1000, 2000], num_layers=2, num_kv_heads=2, num_q_heads=8, head_dim=128,
                window=32, num_sinks=4, device="cpu")
    args.update(kw)
    return kv.Problem(**args)


def test_workspace_size_and_shape_checks(kv):
    assert kv.kv_score_workspace_size(_prob(kv)) > 0
    assert kv.kv_select_workspace_size(_prob(kv)) >= 4
    for bad, code in [(dict(head_dim=96), kv.KV_ERR_UNSUPPORTED),
                      (dict(num_q_heads=7), kv.KV_ERR_INVALID_ARG),
                      (dict(window=0), kv.KV_ERR_INVALID_ARG),
                      (dict(lengths=[20, 2000]), kv.KV_ERR_INVALID_ARG),
                      (dict(num_q_heads=2 * 17, window=32), kv.KV_ERR_UNSUPPORTED),
                      # 2^31 packed K/V rows: beyond the 32-bit TMA row coordinates
                      (dict(lengths=[1 << 30, 1 << 30], num_layers=1, num_kv_heads=1,
                            num_q_heads=4), kv.KV_ERR_UNSUPPORTED)]:
        with pytest.raises(kv.KvError) as e:
            kv.kv_score_workspace_size(_prob(kv, **bad))
        assert e.value.code == code, bad


def test_score_argument_checks_before_launch(kv):
    lib = kv.load()
    p = _prob(kv)
    ws = kv.kv_score_workspace_size(p)
    fake = 1 << 20  # never dereferenced: the checks fail first
    assert lib.kv_score(p.c, None, fake, fake, fake, fake, ws, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_score(p.c, fake + 4, fake, fake, fake, fake, ws, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_score(p.c, fake, fake, fake, fake, fake, ws - 1, None) == kv.KV_ERR_WORKSPACE
    assert lib.kv_select_topk(p.c, fake, fake, fake, fake, fake, 3, None) == kv.KV_ERR_WORKSPACE
    assert lib.kv_compact(p.c, fake, fake, fake, fake, -1, fake, fake, None) == kv.KV_ERR_INVALID_ARG
    empty = _prob(kv, lengths=[])
    assert lib.kv_score(empty.c, None, None, None, None, None, 0, None) == kv.KV_OK
    assert lib.kv_compact(empty.c, None, None, None, None, 0, None, None, None) == kv.KV_OK


def test_fused_argument_checks_before_launch(kv):
    """kv_evict_fused validates like kv_score, kv_select_topk and kv_compact together,
    before anything is launched."""
    lib = kv.load()
    p = _prob(kv)
    ws = kv.kv_score_workspace_size(p)
    f = 1 << 20  # never dereferenced: the checks fail first
    call = lib.kv_evict_fused
    ok_args = [p.c, f, f, f, f, f, 64, f, f, f, f, f, ws, None]

    def with_(i, value):
        a = list(ok_args)
        a[i] = value
        return call(*a)

    assert with_(1, None) == kv.KV_ERR_INVALID_ARG        # q_win
    assert with_(1, f + 4) == kv.KV_ERR_INVALID_ARG       # misaligned q_win
    assert with_(12, ws - 1) == kv.KV_ERR_WORKSPACE       # score workspace too small
    assert with_(4, None) == kv.KV_ERR_INVALID_ARG        # budgets
    assert with_(5, None) == kv.KV_ERR_INVALID_ARG        # offsets
    assert with_(6, -1) == kv.KV_ERR_INVALID_ARG          # total_rows
    assert with_(7, None) == kv.KV_ERR_INVALID_ARG        # scores
    assert with_(8, None) == kv.KV_ERR_INVALID_ARG        # sel_idx
    assert with_(9, None) == kv.KV_ERR_INVALID_ARG        # k_out with rows to copy
    assert with_(10, f + 2) == kv.KV_ERR_INVALID_ARG      # misaligned v_out
    empty = _prob(kv, lengths=[])
    assert call(empty.c, None, None, None, None, None, 0, None, None, None, None, None, 0,
                None) == kv.KV_OK


def test_make_offsets(kv):
    p = _prob(kv)
    b = np.array([36, 40, 100, 1000, 36, 2000, 37, 50], np.int32)
    np.testing.assert_array_equal(kv.kv_make_offsets(p, b), oracle.offsets(b))
    for bad in (35, 1001):
        b2 = b.copy()
        b2[3] = bad
        with pytest.raises(kv.KvError) as e:
            kv.kv_make_offsets(p, b2)
        assert e.value.code == kv.KV_ERR_BUDGET


@pytest.mark.parametrize("L,B", [(32, 13107), (28, 6553), (1, 256), (2, 100), (80, 999), (5, 3)])
def test_budget_helpers_equal_oracle(kv, L, B):
    prof = synth.ripple_profile(synth.QWEN7B_128K.scaled(num_layers=L))
    np.testing.assert_array_equal(kv.kv_budgets_pyramid(L, B), oracle.budgets_pyramid(L, B))
    np.testing.assert_array_equal(kv.kv_budgets_pyramid(L, B, 2.0, 0.25, 0.8),
                                  oracle.budgets_pyramid(L, B, 2.0, 0.25, 0.8))
    for beta, gamma in [(2.0, math.inf), (math.log(1.5), math.inf), (3.0, 4.0)]:
        np.testing.assert_array_equal(kv.kv_budgets_ripple(L, B, prof, beta, gamma),
                                      oracle.budgets_ripple(L, B, prof, beta, gamma))


def test_config_budgets_equal_oracle(kv):
    from tests import parity
    for wl in synth.CONFIGS:
        prof = synth.ripple_profile(wl) if wl.budget_policy == "ripple" else None
        np.testing.assert_array_equal(parity.product_budgets(kv, wl, prof),
                                      oracle.segment_budgets(wl, prof))


def test_score_rule_and_pool_argument_checks(kv):
    lib = kv.load()
    for rule in (kv.KV_SCORE_DROPKV, kv.KV_SCORE_DROPKV_SQUARED, kv.KV_SCORE_ATTN_SUM):
        assert kv.kv_score_workspace_size(_prob(kv, score_rule=rule)) > 0
    for bad in (-1, 3):
        with pytest.raises(kv.KvError) as e:
            kv.kv_score_workspace_size(_prob(kv, score_rule=bad))
        assert e.value.code == kv.KV_ERR_INVALID_ARG
    p = _prob(kv)
    nbytes = 2 * 2 * 3000 * 4          # L * H * N_tot floats
    a, b = 1 << 24, (1 << 24) + (1 << 20)
    for kernel in (0, 2, 12, 257):      # even, or outside 1..255
        assert lib.kv_pool_scores(p.c, kernel, a, b, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_pool_scores(p.c, 11, None, b, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_pool_scores(p.c, 11, a + 4, b, None) == kv.KV_ERR_INVALID_ARG
    # overlapping input and output ranges
    assert lib.kv_pool_scores(p.c, 11, a, a, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_pool_scores(p.c, 11, a, a + nbytes - 16, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_pool_scores(p.c, 11, a + nbytes - 16, a, None) == kv.KV_ERR_INVALID_ARG
    empty = _prob(kv, lengths=[])
    assert lib.kv_pool_scores(empty.c, 11, None, None, None) == kv.KV_OK


def test_block_helpers_host_side(kv):
    lib = kv.load()
    p = _prob(kv, num_layers=4)
    bp = p.block_view(2)
    assert (bp.num_layers, bp.num_kv_heads, bp.num_q_heads) == (2, 1, 1)
    with pytest.raises(ValueError):
        p.block_view(3)
    b = kv.kv_budgets_fraction(bp, 0.1)
    want = [oracle.block_budget(n, 32, 4, 0.1) for n in (1000, 2000) for _ in range(2)]
    assert list(b) == want
    with pytest.raises(kv.KvError):
        kv.kv_budgets_fraction(bp, 1.5)
    fake = 1 << 20
    assert lib.kv_block_scores(p.c, 3, fake, fake, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_block_scores(p.c, 0, fake, fake, None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_compact_blocks(p.c, 3, fake, fake, fake, fake, fake, 10, fake, fake,
                                 None) == kv.KV_ERR_INVALID_ARG
    assert lib.kv_compact_blocks(p.c, 2, fake, fake, fake, fake, fake, -1, fake, fake,
                                 None) == kv.KV_ERR_INVALID_ARG


def test_host_pipeline_plan_checks(kv):
    """kv_evict_host_workspace_size / kv_evict_host argument checks (host only)."""
    prob = _prob(kv, lengths=[1000, 2000], num_layers=5)
    budgets = np.full(prob.num_units, 200, dtype=np.int32)
    good = kv._KvHostPlan(2, 1, 0, 0)
    one = kv.kv_evict_host_workspace_size(prob, good, budgets)
    # the workspace holds two slots of a 2-layer group: more than one layer's K and V
    N, d, H = prob.total_tokens, prob.head_dim, prob.num_kv_heads
    assert one > 2 * 2 * (2 * H * N * d * 2)
    for bad in (kv._KvHostPlan(0, 1, 0, 0), kv._KvHostPlan(6, 1, 0, 0),
                kv._KvHostPlan(2, 4, 0, 0), kv._KvHostPlan(2, 11, 0, 1),
                kv._KvHostPlan(2, 1, 1, 1)):
        with pytest.raises(kv.KvError) as e:
            kv.kv_evict_host_workspace_size(prob, bad, budgets)
        assert e.value.code == kv.KV_ERR_INVALID_ARG
    # a budget below sinks + window is refused on the host before anything is copied
    bad_b = budgets.copy()
    bad_b[3] = 10
    offs = np.zeros(prob.num_units + 1, dtype=np.int64)
    st = ctypes.c_int32()
    rc = kv.load().kv_evict_host(prob.c, ctypes.byref(good), 16, 16, 16,
                                 bad_b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                 offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), 16, 16, 16,
                                 256, one, None, ctypes.byref(st))
    assert rc == kv.KV_ERR_BUDGET


def test_host_pipeline_workspace_covers_every_group_shape(kv):
    """A smaller last group can choose smaller pass-1 splits (more partials per unit)
    than the full groups: the workspace must cover the largest need of any group."""
    prob = _prob(kv, lengths=[131072], num_layers=5, num_kv_heads=1, num_q_heads=4)
    budgets = np.full(prob.num_units, 2000, dtype=np.int32)
    plan = kv._KvHostPlan(4, 1, 0, 0)
    total = kv.kv_evict_host_workspace_size(prob, plan, budgets)
    sub4 = _prob(kv, lengths=[131072], num_layers=4, num_kv_heads=1, num_q_heads=4)
    sub1 = _prob(kv, lengths=[131072], num_layers=1, num_kv_heads=1, num_q_heads=4)
    s4, s1 = kv.kv_score_workspace_size(sub4), kv.kv_score_workspace_size(sub1)
    assert s1 > s4 / 4          # the one-layer group needs more than a quarter of four layers
    assert total >= 2 * max(s4, s1)
