"""The seeded input generators: determinism, row regeneration, bf16 rounding and
the target distributions of the benchmarked configurations."""
import numpy as np

import workloads as wk


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e38, np.inf],
                 np.float32)
    bits = wk.f32_to_bf16_bits(f)
    back = wk.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: even is 1 + 2^-6
    assert list(back[:5]) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5]
    assert np.isinf(back[-1])


def test_bf16_rounding_error_bound():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    y = wk.bf16_bits_to_f32(wk.f32_to_bf16_bits(x))
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)


def test_rows_regenerate_exactly():
    full = wk.normal_matrix(3, wk.TID_LOGITS, 50, 70000, 3.0, True, threads=4)
    rows = [0, 13, 14, 49]
    np.testing.assert_array_equal(wk.normal_rows(3, wk.TID_LOGITS, rows, 70000, 3.0, True), full[rows])
    again = wk.normal_matrix(3, wk.TID_LOGITS, 50, 70000, 3.0, True, threads=1)
    np.testing.assert_array_equal(full, again)


def test_normal_moments():
    v = wk.bf16_bits_to_f32(wk.normal_matrix(0, wk.TID_X, 256, 4096, 3.0, True))
    assert abs(v.mean()) < 0.01 and abs(v.std() - 3.0) < 0.01


def test_uniform_targets_ignore_fraction():
    t = wk.uniform_targets(0, 16384, 128256, 0.05)
    frac = (t == wk.IGNORE_IDX).mean()
    assert 0.04 < frac < 0.06
    ok = t[t != wk.IGNORE_IDX]
    assert ok.min() >= 0 and ok.max() < 128256


def test_zipf_targets():
    t = wk.zipf_targets(0, 200000, 1000, 1.1)
    h = (np.arange(1, 1001, dtype=np.float64) ** -1.1).sum()
    assert abs((t == 0).mean() - 1 / h) < 0.01
    assert t.min() >= 0 and t.max() < 1000


def test_large_linear_workload_tail_is_ignored():
    t = wk.linear_targets(wk.LINEAR_LARGE)
    assert np.all(t[-903:] == wk.IGNORE_IDX)
    assert np.all(t[:-903] >= 0)
    assert (t != wk.IGNORE_IDX).sum() == 15481
