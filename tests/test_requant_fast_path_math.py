"""The exactness argument behind requant's f16x2 fast path, checked on the
CPU against the oracle's codecs. numpy's float16 product of two float16
values is the correctly rounded IEEE result (the exact product fits in
float32), as the packed hardware multiply's is.

- Pass 1: every nonzero E4M3 value times 2^k, k in [-5, 0], is an exact
  normal float16, so the colwise maximum of |val| 2^(rs - R) is exact.
- The column scale code read from that float16 maximum (exponent field ef,
  reference R), max(ef + R - 23, 0), is the oracle's E8M0 code of the exact
  maximum of |val| 2^(rs - 127); an all-zero column gives code 0.
- Pass 2: for every E4M3 value and every d in [-14, 15], 2^d is a normal
  float16, and wherever |val 2^d| < 512 (the column scale guarantees that
  bound for every value of its column) encoding the float16 product gives
  the oracle's code for the exact product."""
import numpy as np

import oracle as orc

CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.int64)  # every non-NaN code
VALS = np.array([orc.e4m3_value(int(c)) for c in CODES])


def test_pass1_products_are_exact_normal_float16():
    nz = VALS[VALS != 0]
    for k in range(-5, 1):
        p = (nz.astype(np.float16) * np.float16(2.0 ** k)).astype(np.float64)
        assert np.array_equal(p, nz * 2.0 ** k), k
        assert np.all(np.abs(p) >= 2.0 ** -14), k


def test_pass2_encode_through_float16_equals_the_exact_encode():
    for d in range(-14, 16):
        m = np.float16(2.0 ** d)
        assert float(m) == 2.0 ** d and int((m.view(np.uint16) >> 10) & 0x1F) == d + 15, d
        v = VALS[np.abs(VALS) * 2.0 ** d < 512]
        p16 = (v.astype(np.float16) * m).astype(np.float64)
        assert np.array_equal(orc.e4m3_encode_array(p16), orc.e4m3_encode_array(v * 2.0 ** d)), d


def test_column_scale_from_the_float16_maximum():
    rng = np.random.default_rng(2026)
    for trial in range(4000):
        R = int(rng.integers(0, 255)) if trial % 4 else int(rng.integers(0, 8))
        rs = np.maximum(R - rng.integers(0, 6, 32), 0)
        rs[int(rng.integers(32))] = R
        idx = rng.integers(0, len(CODES), 32)
        if trial % 5 == 0:
            idx[:] = 0                                   # an all-zero column (code 0x00)
        elif trial % 5 == 1:
            idx[rng.random(32) < 0.7] = 0
        v = VALS[idx]
        exact = float(np.max(np.abs(v) * 2.0 ** (rs.astype(np.float64) - 127)))
        want = orc.e8m0_exponent(exact) + 127
        m16 = np.max(np.abs(v.astype(np.float16) * (2.0 ** (rs - R)).astype(np.float16)))
        hb = int(np.float16(m16).view(np.uint16))
        got = 0 if hb == 0 else max((hb >> 10) + R - 23, 0)
        assert got == want, (trial, R, hb, want)
