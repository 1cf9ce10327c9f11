"""CPU pins of the test-side operand builders in tests/_layouts.py: the
swizzled layouts they assemble from compact scales equal the oracle
quantizer's own swizzled output, and the random codes are valid E4M3."""
import numpy as np

import oracle as orc
from synth import bf16_bits_from_f32
from tests._layouts import random_codes, random_scales, swizzle_colwise_grouped, swizzle_rowwise


def test_swizzle_builders_reproduce_the_oracle_quantizer():
    rng = np.random.default_rng(3)
    ms = np.array([256, 0, 128, 384], np.int64)
    M, K = int(ms.sum()), 640
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    c = orc.group_quantize(x, ms)
    s = orc.group_quantize(x, ms, swizzled=True)
    assert np.array_equal(swizzle_rowwise(c["row_s"]), s["row_s"])
    assert np.array_equal(swizzle_colwise_grouped(c["col_s"], ms, K), s["col_s"])


def test_swizzle_builders_for_weights():
    rng = np.random.default_rng(4)
    E, N, K = 3, 256, 384
    w = bf16_bits_from_f32((0.02 * rng.standard_normal((E, N, K))).astype(np.float32))
    c = orc.quantize_weights(w)
    s = orc.quantize_weights(w, swizzled=True)
    assert np.array_equal(swizzle_rowwise(c["row_s"]), s["row_s"])
    assert np.array_equal(swizzle_colwise_grouped(c["col_s"], np.full(E, N), K), s["col_s"])


def test_random_codes_are_finite_e4m3():
    codes = random_codes(np.random.default_rng(5), 100_003, chunk=4096)
    assert codes.size == 100_003
    assert not np.any((codes & 0x7F) == 0x7F)
    vals = np.array([orc.e4m3_value(int(b)) for b in np.unique(codes)])
    assert np.all(np.isfinite(vals)) and np.max(np.abs(vals)) == 448.0
    assert len(np.unique(codes)) == 254  # every finite code appears
    s = random_scales(np.random.default_rng(6), (64, 64))
    assert s.min() >= 118 and s.max() <= 136


def test_weight_slab_atom_mapping():
    """The full-size weight test compares 128-row slabs: slab j of expert e, quantized by the
    oracle as a member of its own, must equal the same rows and scale atoms of the whole
    weight's quantization (rowwise atoms contiguous, colwise atom kb at
    e K N / 32 + (kb (N / 128) + j) * 512)."""
    import oracle as orc

    E, N, K = 3, 384, 512
    w = bf16_bits_from_f32((0.02 * np.random.default_rng(1).standard_normal((E, N, K))).astype(np.float32))
    full = orc.quantize_weights(w, swizzled=True)
    nkb = K // 128
    for e in range(E):
        for j in range(N // 128):
            r0 = e * N + 128 * j
            o = orc.quantize_weights(w[e, 128 * j:128 * j + 128][None], swizzled=True)
            assert np.array_equal(full["row_q"][r0:r0 + 128], o["row_q"])
            assert np.array_equal(full["col_q"][r0:r0 + 128], o["col_q"])
            a = (r0 // 128) * nkb * 512
            assert np.array_equal(full["row_s"][a:a + nkb * 512], o["row_s"])
            idx = e * K * N // 32 + (np.arange(nkb)[:, None] * (N // 128) + j) * 512 + np.arange(512)[None, :]
            assert np.array_equal(full["col_s"][idx.ravel()], o["col_s"])
