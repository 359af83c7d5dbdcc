"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np

import synth


def test_irwin_hall_moments_and_support():
    z = synth.normals_f32(synth.stream_key(3, synth.S_K), 0, 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.var() - 1.0) < 5e-3
    assert z.min() >= -6.0 and z.max() <= 6.0
    # values are exact multiples of 2**-16
    assert np.all(z * 65536.0 == np.round(z * 65536.0))


def test_generator_is_counter_based():
    key = synth.stream_key(11, synth.S_V)
    a = synth.normals_f32(key, 1000, 5000)
    b = synth.normals_f32(key, 3000, 1000)
    np.testing.assert_array_equal(a[2000:3000], b)


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    assert list(synth.f32_to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F80]
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x[[0, 3]])),
                                  x[[0, 3]])


def test_workload_shapes():
    wl = synth.RAGGED_MISTRAL
    n = wl.seq_lengths()
    assert len(n) == 8 and all(16384 <= t <= 131072 for t in n)
    assert wl.cu_seqlens()[-1] == sum(n)
    assert synth.LLAMA8B_32K.mean_budgets() == [1638]
    assert synth.LONG_128K.mean_budgets() == [13107]
    assert synth.QWEN7B_128K.mean_budgets() == [6553]
    assert synth.QWEN7B_128K.rows == 448 and synth.LONG_128K.rows == 256


def test_heavy_and_outliers():
    wl = synth.small_variant(synth.LLAMA8B_32K, 3000)
    hp = synth.heavy_positions(wl)
    assert hp.shape == (1, 2, 2, 8)
    for seg in hp.reshape(-1, 8):
        assert len(set(seg)) == 8 and seg.min() >= 4 and seg.max() < 3000 - wl.window
    oc = synth.outlier_channels(wl)
    assert oc.shape == (2, 2, 4) and all(len(set(x)) == 4 for x in oc.reshape(-1, 4))
    q = synth.q_window(wl)
    k, v = synth.kv_unit(wl, 0, 1, 1)
    hv = synth.heavy_rows(wl, q)
    np.testing.assert_array_equal(k[hp[0, 1, 1]], np.broadcast_to(hv[0, 1, 1], (8, wl.head_dim)))
    # outlier channels carry 8x the scale
    kf = synth.bf16_bits_to_f32(np.delete(k, hp[0, 1, 1], axis=0))
    rms = np.sqrt((kf.astype(np.float64) ** 2).mean(axis=0))
    big = set(oc[1, 1])
    for c in range(wl.head_dim):
        assert (rms[c] > 4.0) == (c in big)


def test_kv_rows_equal_whole_unit_rows():
    """The row-level host regenerator gives the same bits as the whole-unit one,
    heavy rows and outlier channels included."""
    wl = synth.small_variant(synth.RAGGED_MISTRAL, 0, requests=[900, 1300], layers=2)
    for (r, l, h) in [(0, 0, 0), (1, 1, 1), (1, 0, 1)]:
        k, v = synth.kv_unit(wl, r, l, h)
        n = k.shape[0]
        rows = np.array([0, 3, 17, n // 2, n - 1] + list(synth.heavy_positions(wl)[r, l, h][:3]))
        kr, vr = synth.kv_rows(wl, r, l, h, rows)
        np.testing.assert_array_equal(kr, k[rows])
        np.testing.assert_array_equal(vr, v[rows])
