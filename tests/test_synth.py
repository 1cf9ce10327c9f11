"""Synthetic workload generator: counts and shapes follow the workload recipes."""
import numpy as np

from synth import WORKLOADS, make_m_splits, round_counts_to_128, bf16_bits_from_f32, f32_from_bf16_bits


def test_m_splits_contract():
    for w in WORKLOADS.values():
        m = make_m_splits(w)
        assert m.dtype == np.int64 and len(m) == w.E
        assert int(m.sum()) == w.M and np.all(m % 128 == 0) and np.all(m >= 0)
        assert np.array_equal(m, make_m_splits(w))          # seeded, repeatable
    assert list(make_m_splits(WORKLOADS["e4_h512_n1024_t512"])) == [128, 256, 0, 128]
    m5 = make_m_splits(WORKLOADS["e128_h7168_n2048_t128k_skew"])
    assert (m5 == 0).sum() == 32


def test_round_counts_largest_remainder():
    out = round_counts_to_128([100.0, 156.0, 0.0, 128.0], 384)
    assert list(out) == [128, 128, 0, 128]
    out = round_counts_to_128([64.0, 64.0, 128.0], 256)      # tie -> lower index
    assert list(out) == [128, 0, 128]


def test_bf16_bits_roundtrip():
    x = np.array([1.0, -2.5, 3.140625, 1e-40, 65504.0], np.float32)
    assert np.array_equal(f32_from_bf16_bits(bf16_bits_from_f32(x))[:3], x[:3])
