"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- PyTorch's independent float8_e4m3fn decoder, bit-level brute force,
closed forms, invariants of the MX format, numpy's BLAS, finite differences.
A plausible slip in the oracle (a wrong rounding rule, a dropped clamp, a
transposed operand, a wrong index in a layout) fails at least one of them.
"""
import numpy as np
import pytest
import torch

from synth import bf16_bits_from_f32, f32_from_bf16_bits

# PyTorch's own E4M3 (fn) decoder: an independent table of code values.
TABLE = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
POS_CODES = np.arange(0, 0x7F)          # 0x00..0x7E: the 127 finite non-negative codes
POS_VALS = TABLE[POS_CODES]


def nearest_code_bruteforce(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code by enumeration of every code; ties -> even
    mantissa; |v| > 448 saturates; the sign is kept (negative zero = 0x80)."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    out = np.empty(v.shape, np.uint8)
    flat_a = a.ravel()
    res = np.empty(flat_a.shape, np.int64)
    for lo in range(0, flat_a.size, 4096):
        aa = flat_a[lo:lo + 4096, None]
        d = np.abs(POS_VALS[None, :] - aa)
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        even = cand & ((POS_CODES[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        res[lo:lo + 4096] = POS_CODES[pick]
    res = np.where(flat_a > 448.0, 0x7E, res)
    out = res.reshape(v.shape).astype(np.uint8)
    return out | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)


def floor_log2_bf16_bits(b: np.ndarray) -> np.ndarray:
    """floor(log2 |x|) for non-zero finite bf16 bit patterns, from the bit
    fields alone (exponent field, or leading one of a subnormal mantissa)."""
    b = np.asarray(b, np.int64) & 0x7FFF
    E = b >> 7
    m = b & 0x7F
    lead = np.array([int(x).bit_length() - 1 for x in m])
    return np.where(E > 0, E - 127, lead - 133)


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
FINITE_BF16 = ALL_BF16[((ALL_BF16.astype(np.int64) >> 7) & 0xFF) != 0xFF]


# ------------------------------------------------------------- E4M3 codec
def test_e4m3_decode_matches_torch(orc):
    for c in range(256):
        ref = TABLE[c]
        got = orc.e4m3_value(c)
        if np.isnan(ref):
            assert np.isnan(got)
        else:
            assert got == ref and np.signbit(got) == np.signbit(ref), c


def test_e4m3_known_points(orc):
    # Format facts of OCP MX v1.0 E4M3: 1.0 = 0x38, max finite 448 = 0x7E,
    # min normal 2^-6 = 0x08, min subnormal 2^-9 = 0x01.
    assert orc.e4m3_encode(1.0) == 0x38
    assert orc.e4m3_encode(448.0) == 0x7E
    assert orc.e4m3_encode(2.0 ** -6) == 0x08
    assert orc.e4m3_encode(2.0 ** -9) == 0x01
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(1e6) == 0x7E and orc.e4m3_encode(-1e6) == 0xFE
    assert orc.e4m3_encode(470.0) == 0x7E and orc.e4m3_encode(-511.0) == 0xFE


@pytest.mark.parametrize("shift", [-127, -20, -9, -8, -1, 0, 1, 8, 119])
def test_e4m3_encode_bruteforce_all_bf16(orc, shift):
    v = f32_from_bf16_bits(FINITE_BF16).astype(np.float64) * np.ldexp(1.0, -shift)
    got = orc.e4m3_encode_array(v)
    ref = nearest_code_bruteforce(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (shift, v[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_ties_go_to_even(orc):
    # midpoints between consecutive positive codes are exact ties
    mids = (POS_VALS[:-1] + POS_VALS[1:]) / 2
    got = orc.e4m3_encode_array(mids)
    lo, hi = POS_CODES[:-1], POS_CODES[1:]
    want = np.where((lo & 1) == 0, lo, hi)
    assert np.array_equal(got, want.astype(np.uint8))
    # the 448/480 midpoint saturates to 448
    assert orc.e4m3_encode(464.0) == 0x7E


# ------------------------------------------------------------- E8M0 scale
def test_e8m0_exhaustive_bf16(orc):
    pos = FINITE_BF16[(FINITE_BF16 < 0x8000) & (FINITE_BF16 != 0)]
    a = f32_from_bf16_bits(pos).astype(np.float64)
    got = orc.e8m0_exponent_array(a)
    want = np.clip(floor_log2_bf16_bits(pos) - 8, -127, 127)
    assert np.array_equal(got, want)
    # defining property when not clamped: amax * 2^-s lies in [256, 512)
    ok = want > -127
    v = a[ok] * np.ldexp(1.0, -want[ok])
    assert np.all((v >= 256) & (v < 512))
    assert orc.e8m0_exponent(0.0) == -127


# ------------------------------------------------------------- bf16 round
def test_bf16_round_is_nearest_even(orc):
    rng = np.random.default_rng(1)
    v = rng.standard_normal(20000) * np.exp2(rng.integers(-140, 120, 20000))
    got = orc.bf16_round_array(v)
    gv = f32_from_bf16_bits(got).astype(np.float64)
    # neighbours of the result
    up = f32_from_bf16_bits((got.astype(np.int64) + 1).astype(np.uint16)).astype(np.float64)
    dn = f32_from_bf16_bits((got.astype(np.int64) - 1).astype(np.uint16)).astype(np.float64)
    err = np.abs(gv - v)
    nz = (got & 0x7FFF) != 0
    assert np.all(err[nz] <= np.abs(up[nz] - v[nz]))
    assert np.all(err[nz] <= np.abs(dn[nz] - v[nz]) + 0.0)
    # single-precision inputs: agree with torch's float32 -> bfloat16 (RNE)
    f = v.astype(np.float32)
    t = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_round_array(f.astype(np.float64)), t)


# ---------------------------------------------------------- block quantize
def _round_trip_bound(v):
    """Error bound in units of the block scale: half an E4M3 ulp up to 464,
    the saturation gap (< 64) above."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -20)))
    ulp = np.exp2(np.maximum(e, -6) - 3)
    return np.where(a <= 464, ulp / 2, 64.0)


def test_block_quantize_bruteforce_tiny_blocks(orc):
    rng = np.random.default_rng(2)
    pool = np.array([0.0, -0.0, 1.0, -1.0, 1.5, -3.0, 0.375, 2.0 ** -10, 7.0, -448.0, 511.0, 1e-3, 96.5])
    for _ in range(300):
        x = rng.choice(pool, 32) * np.ldexp(1.0, int(rng.integers(-30, 30)))
        codes, sc = orc.quantize_block(x)
        amax = np.max(np.abs(x))
        if amax == 0:
            assert sc == 0
        else:
            s = sc - 127
            lead = int(np.floor(np.log2(amax)))
            assert s == max(-127, min(127, lead - 8))
            # no other shared exponent puts the block max in [256, 512)
            for s2 in range(s - 3, s + 4):
                inside = 256 <= amax * 2.0 ** -s2 < 512
                assert inside == (s2 == s) or s == -127
        s = sc - 127
        assert np.array_equal(codes, nearest_code_bruteforce(x * 2.0 ** -s))


def test_block_round_trip_bound_and_equivariance(orc):
    rng = np.random.default_rng(3)
    for _ in range(200):
        x = rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 3)
        x[rng.random(32) < 0.1] *= 1000
        codes, sc = orc.quantize_block(x)
        s = sc - 127
        deq = TABLE[codes] * 2.0 ** s
        v = x * 2.0 ** -s
        assert np.all(np.abs(deq - x) <= _round_trip_bound(v) * 2.0 ** s)
        k = int(rng.integers(-20, 20))
        c2, sc2 = orc.quantize_block(x * 2.0 ** k)
        assert np.array_equal(c2, codes) and sc2 == sc + k


# ---------------------------------------------------------------- swizzle
@pytest.mark.parametrize("R,C", [(128, 4), (256, 8), (384, 12), (128, 56)])
def test_swizzle_structure(orc, R, C):
    off = np.array([[orc.swizzle_offset(r, c, C) for c in range(C)] for r in range(R)])
    assert np.array_equal(np.sort(off.ravel()), np.arange(R * C))       # bijection
    r, c = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    assert np.array_equal(off // 512, (r // 128) * (C // 4) + c // 4)   # 128x4 atoms, row-major
    # the four scales of one row inside an atom are adjacent bytes
    assert np.all(np.diff(off.reshape(R, C // 4, 4), axis=2) == 1)
    # consecutive rows of the same 32-row slab are 16 bytes apart
    assert np.all((off[1:32] - off[:31]) == 16)
    # rows 32 apart share a 16-byte line, 4 bytes apart
    assert np.all(off[32:128] - off[0:96] == 4)
    S = np.arange(R * C, dtype=np.uint64).astype(np.uint8).reshape(R, C)
    sw = orc.swizzle(S)
    assert np.array_equal(sw[off.ravel()], S.ravel())


# ------------------------------------------------------- grouped quantize
def _tiny_inputs(M=512, K=256, seed=4, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(scale)
    x[rng.random((M, K)) < 0.01] *= 1000
    x[:32, :32] = 0.0
    return bf16_bits_from_f32(x)


def test_group_quantize_equals_blockwise_definition(orc):
    x = _tiny_inputs()
    ms = np.array([128, 0, 256, 128])
    r = orc.group_quantize(x, ms, swizzled=False)
    xf = f32_from_bf16_bits(x).astype(np.float64)
    M, K = x.shape
    for m in range(0, M, 7):
        for j in range(K // 32):
            c, s = orc.quantize_block(xf[m, 32 * j:32 * j + 32])
            assert np.array_equal(r["row_q"][m, 32 * j:32 * j + 32], c) and r["row_s"][m, j] == s
    for i in range(M // 32):
        for k in range(0, K, 5):
            c, s = orc.quantize_block(xf[32 * i:32 * i + 32, k])
            assert np.array_equal(r["col_q"][32 * i:32 * i + 32, k], c) and r["col_s"][i, k] == s
    assert r["row_s"][0, 0] == 0 and r["col_s"][0, 0] == 0   # all-zero blocks


def test_grouped_equals_dense_and_swizzle_bases(orc):
    x = _tiny_inputs()
    ms = np.array([128, 0, 256, 128])
    g = orc.group_quantize(x, ms, swizzled=False)
    d = orc.group_quantize(x, np.array([512]), swizzled=False)
    for k in ("row_q", "row_s", "col_q", "col_s"):
        assert np.array_equal(g[k], d[k])
    sw = orc.group_quantize(x, ms, swizzled=True)
    M, K = x.shape
    # rowwise: one dense (M, K/32) matrix
    for r_ in range(0, M, 3):
        for c in range(K // 32):
            assert sw["row_s"][orc.swizzle_offset(r_, c, K // 32)] == g["row_s"][r_, c]
    # colwise: per expert (K, m_e/32) at byte K*off_e/32
    off = 0
    for me in ms:
        for k in range(0, K, 3):
            for i in range(me // 32):
                b = K * off // 32 + orc.swizzle_offset(k, i, me // 32)
                assert sw["col_s"][b] == g["col_s"][off // 32 + i, k]
        off += me
    assert np.array_equal(sw["row_q"], g["row_q"]) and np.array_equal(sw["col_q"], g["col_q"])


def test_rowwise_and_colwise_bounds_against_source(orc):
    x = _tiny_inputs(seed=5)
    g = orc.group_quantize(x, np.array([256, 256]), swizzled=False)
    xf = f32_from_bf16_bits(x).astype(np.float64)
    M, K = x.shape
    srow = np.repeat(g["row_s"][:M, :K // 32].astype(np.int64) - 127, 32, axis=1)
    scol = np.repeat(g["col_s"][:M // 32, :K].astype(np.int64) - 127, 32, axis=0)
    drow = TABLE[g["row_q"]] * np.exp2(srow)
    dcol = TABLE[g["col_q"]] * np.exp2(scol)
    brow = _round_trip_bound(xf * np.exp2(-srow)) * np.exp2(srow)
    bcol = _round_trip_bound(xf * np.exp2(-scol)) * np.exp2(scol)
    assert np.all(np.abs(drow - xf) <= brow)
    assert np.all(np.abs(dcol - xf) <= bcol)
    assert np.all(np.abs(drow - dcol) <= brow + bcol)


def test_dequant_matches_independent_decode(orc):
    x = _tiny_inputs(seed=12)
    g = orc.group_quantize(x, np.array([384, 128]), swizzled=False)
    M, K = x.shape
    srow = np.repeat(g["row_s"][:M, :K // 32].astype(np.int64) - 127, 32, axis=1)
    scol = np.repeat(g["col_s"][:M // 32, :K].astype(np.int64) - 127, 32, axis=0)
    assert np.array_equal(orc.dequant_rowwise(g["row_q"], g["row_s"]), TABLE[g["row_q"]] * np.exp2(srow))
    assert np.array_equal(orc.dequant_colwise(g["col_q"], g["col_s"]), TABLE[g["col_q"]] * np.exp2(scol))


def test_invalid_splits_rejected(orc):
    x = _tiny_inputs(M=256, K=128)
    for bad in ([128, 64, 64], [256, -128, 128], [128, 0]):
        with pytest.raises(ValueError):
            orc.group_quantize(x, np.array(bad))


# ------------------------------------------------------------------ requant
def test_requant_is_colwise_quant_of_rowwise_dequant(orc):
    x = _tiny_inputs(seed=6)
    ms = np.array([128, 256, 0, 128])
    wire = orc.group_quantize(x, ms, rowwise=True, colwise=False, swizzled=False)
    rq = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=False, dbias=True, dequant=True)
    M, K = x.shape
    srow = np.repeat(wire["row_s"][:M, :K // 32].astype(np.int64) - 127, 32, axis=1)
    deq = TABLE[wire["row_q"]] * np.exp2(srow)          # independent decode
    for i in range(M // 32):
        for k in range(0, K, 3):
            c, s = orc.quantize_block(deq[32 * i:32 * i + 32, k])
            assert np.array_equal(rq["col_q"][32 * i:32 * i + 32, k], c) and rq["col_s"][i, k] == s
    # exact dequant fits bf16 here; the bf16 output is that value
    assert np.array_equal(f32_from_bf16_bits(rq["deq"]).astype(np.float64), deq)
    # dbias is reduced from the dequantized values, per expert; empty expert -> 0
    off = 0
    for e, me in enumerate(ms):
        np.testing.assert_allclose(rq["dbias"][e], deq[off:off + me].sum(axis=0), rtol=1e-12, atol=1e-9)
        off += me
    assert np.all(rq["dbias"][2] == 0)
    # swizzled rowwise scales are the swizzle of the compact ones
    assert np.array_equal(rq["row_s_swizzled"], orc.swizzle(wire["row_s"][:M, :K // 32]))
    # the double quantization differs from quantizing the source colwise
    direct = orc.group_quantize(x, ms, rowwise=False, colwise=True, swizzled=False)
    assert not np.array_equal(direct["col_q"], rq["col_q"])
    # and it stays within rowwise + colwise bounds of the source
    xf = f32_from_bf16_bits(x).astype(np.float64)
    scol = np.repeat(rq["col_s"][:M // 32, :K].astype(np.int64) - 127, 32, axis=0)
    dcol = TABLE[rq["col_q"]] * np.exp2(scol)
    brow = _round_trip_bound(xf * np.exp2(-srow)) * np.exp2(srow)
    bcol = _round_trip_bound(deq * np.exp2(-scol)) * np.exp2(scol)
    assert np.all(np.abs(dcol - xf) <= brow + bcol)


def test_requant_swizzled_matches_compact(orc):
    x = _tiny_inputs(seed=7)
    ms = np.array([256, 0, 256])
    wire = orc.group_quantize(x, ms, rowwise=True, colwise=False, swizzled=False)
    a = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=False)
    b = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=True)
    assert np.array_equal(a["col_q"], b["col_q"])
    M, K = x.shape
    off = 0
    for me in ms:
        for k in range(0, K, 5):
            for i in range(me // 32):
                assert b["col_s"][K * off // 32 + orc.swizzle_offset(k, i, me // 32)] == a["col_s"][off // 32 + i, k]
        off += me


# -------------------------------------------------------------------- dbias
def test_grouped_dbias(orc):
    rng = np.random.default_rng(8)
    dy = bf16_bits_from_f32(rng.standard_normal((512, 384)).astype(np.float32))
    ms = np.array([0, 256, 128, 0, 128])
    db = orc.grouped_dbias(dy, ms)
    f = f32_from_bf16_bits(dy).astype(np.float64)
    ref = np.stack([f[o:o + m].sum(axis=0) for o, m in zip(np.concatenate([[0], np.cumsum(ms)[:-1]]), ms)])
    np.testing.assert_allclose(db, ref, rtol=1e-12, atol=1e-10)
    assert np.all(db[0] == 0) and np.all(db[3] == 0)


# -------------------------------------------------------------------- GEMMs
def _int_operands(rng, shape):
    """E4M3 codes of small integers and unit scales: exact products."""
    vals = rng.integers(-4, 5, size=shape).astype(np.float64)
    codes = nearest_code_bruteforce(vals)
    assert np.array_equal(TABLE[codes], vals)
    return codes, vals


def test_gemms_exact_on_small_integers(orc):
    rng = np.random.default_rng(9)
    ms = np.array([128, 0, 256])
    M, N, K, E = 384, 256, 128, 3
    xq, xv = _int_operands(rng, (M, K))
    wq, wv = _int_operands(rng, (E, N, K))
    dyq, dyv = _int_operands(rng, (M, N))
    unit = lambda r, c: np.full((r, c), 127, np.uint8)
    xs, ws, dys = unit(M, K // 32), unit(E * N, K // 32), unit(M, N // 32)
    y, mag = orc.fprop(xq, xs, wq, ws, ms)
    e_of = np.repeat(np.arange(E), ms)
    ref = np.einsum("mk,mnk->mn", xv, wv[e_of])
    assert np.array_equal(y, ref) and np.all(mag >= np.abs(y))
    # dgrad reads the colwise weight copy: same integers, colwise unit scales
    wsc = np.full((E * N // 32, K), 127, np.uint8)
    dx, _ = orc.dgrad(dyq, dys, wq, wsc, ms)
    assert np.array_equal(dx, np.einsum("mn,mnk->mk", dyv, wv[e_of]))
    dysc = np.full((M // 32, N), 127, np.uint8)
    xsc = np.full((M // 32, K), 127, np.uint8)
    dw, _ = orc.wgrad(dyq, dysc, xq, xsc, ms)
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(E):
        assert np.array_equal(dw[e], dyv[off[e]:off[e + 1]].T @ xv[off[e]:off[e + 1]])
    assert np.all(dw[1] == 0)


def test_gemms_match_blas_on_quantized_operands(orc):
    rng = np.random.default_rng(10)
    ms = np.array([256, 128, 0, 128])
    E = len(ms)
    M, N, K = int(ms.sum()), 256, 384
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    w = bf16_bits_from_f32((0.02 * rng.standard_normal((E, N, K))).astype(np.float32))
    dy = bf16_bits_from_f32(rng.standard_normal((M, N)).astype(np.float32))
    b = bf16_bits_from_f32((0.02 * rng.standard_normal((E, N))).astype(np.float32))
    qx = orc.group_quantize(x, ms)
    qw = orc.quantize_weights(w)
    qdy = orc.group_quantize(dy, ms)

    def dec_row(q, s):
        return TABLE[q] * np.exp2(np.repeat(s[:q.shape[0], :q.shape[1] // 32].astype(np.int64) - 127, 32, axis=1))

    def dec_col(q, s):
        return TABLE[q] * np.exp2(np.repeat(s[:q.shape[0] // 32, :q.shape[1]].astype(np.int64) - 127, 32, axis=0))

    e_of = np.repeat(np.arange(E), ms)
    Xr, Wr = dec_row(qx["row_q"], qx["row_s"]), dec_row(qw["row_q"], qw["row_s"]).reshape(E, N, K)
    Wc = dec_col(qw["col_q"], qw["col_s"]).reshape(E, N, K)
    DYr, DYc, Xc = dec_row(qdy["row_q"], qdy["row_s"]), dec_col(qdy["col_q"], qdy["col_s"]), dec_col(qx["col_q"], qx["col_s"])
    bias = f32_from_bf16_bits(b).astype(np.float64)

    y, _ = orc.fprop(qx["row_q"], qx["row_s"], qw["row_q"].reshape(E, N, K), qw["row_s"], ms, bias=b)
    ref = np.stack([Xr[m] @ Wr[e_of[m]].T + bias[e_of[m]] for m in range(M)])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    dx, _ = orc.dgrad(qdy["row_q"], qdy["row_s"], qw["col_q"].reshape(E, N, K), qw["col_s"], ms)
    ref = np.stack([DYr[m] @ Wc[e_of[m]] for m in range(M)])
    np.testing.assert_allclose(dx, ref, rtol=1e-12, atol=1e-12)
    dw, _ = orc.wgrad(qdy["col_q"], qdy["col_s"], qx["col_q"], qx["col_s"], ms)
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(E):
        np.testing.assert_allclose(dw[e], DYc[off[e]:off[e + 1]].T @ Xc[off[e]:off[e + 1]], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- SwiGLU
def test_swiglu_against_closed_forms(orc):
    from scipy.special import expit

    rng = np.random.default_rng(11)
    M, F = 64, 96
    y = bf16_bits_from_f32((3 * rng.standard_normal((M, 2 * F))).astype(np.float32))
    dh = bf16_bits_from_f32(rng.standard_normal((M, F)).astype(np.float32))
    yf = f32_from_bf16_bits(y).astype(np.float64)
    g, u = yf[:, :F], yf[:, F:]
    h = f32_from_bf16_bits(orc.swiglu_fwd(y)).astype(np.float64)
    ref = g * expit(g) * u
    # within half a bf16 ulp of the exact value (single rounding)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -120))) - 7)
    assert np.all(np.abs(h - ref) <= ulp / 2 * (1 + 1e-9))
    d = orc.swiglu_bwd(dh, y)
    dg = f32_from_bf16_bits(d[:, :F]).astype(np.float64)
    du = f32_from_bf16_bits(d[:, F:]).astype(np.float64)
    dhf = f32_from_bf16_bits(dh).astype(np.float64)
    # derivative of silu by central finite differences (independent of the closed form)
    eps = 1e-6
    dsilu = ((g + eps) * expit(g + eps) - (g - eps) * expit(g - eps)) / (2 * eps)
    for got, want in ((dg, dhf * u * dsilu), (du, dhf * g * expit(g))):
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -120))) - 7)
        assert np.all(np.abs(got - want) <= ulp * 0.51 + 1e-8 * np.abs(dhf * u))


# ------------------------------------------- scaled bias / routing scales
def _scaled_bias_case(seed=31):
    rng = np.random.default_rng(seed)
    ms = np.array([128, 0, 256, 128], np.int64)  # one empty expert
    M, N, E = int(ms.sum()), 256, len(ms)
    dy_bits = bf16_bits_from_f32(rng.standard_normal((M, N)).astype(np.float32))
    probs = rng.random(M).astype(np.float32)
    bias = bf16_bits_from_f32((0.02 * rng.standard_normal((E, N))).astype(np.float32))
    return dy_bits, ms, probs, bias


def test_scaled_bias_grads_are_gradients_of_the_scaled_bias_term(orc):
    # L(s, b) = sum_m sum_n dY[m,n] * s_m * b_e(m)[n], the part of <dY, y> that the
    # scaled bias contributes, is linear in every s_m and b_e[n]: central differences
    # of this forward definition give both gradients up to rounding
    dy_bits, ms, probs, bias = _scaled_bias_case()
    dy = f32_from_bf16_bits(dy_bits).astype(np.float64)
    b = f32_from_bf16_bits(bias).astype(np.float64)
    e_of = np.repeat(np.arange(len(ms)), ms)

    def L(s, bb):
        return float(np.sum(dy * (s[:, None] * bb[e_of])))

    db, ds = orc.scaled_bias_grads(dy, ms, probs, bias)
    s0, h = probs.astype(np.float64), 0.5
    for m in [0, 127, 128, 300, 383, 384, 511]:
        sp, sm = s0.copy(), s0.copy()
        sp[m] += h
        sm[m] -= h
        fd = (L(sp, b) - L(sm, b)) / (2 * h)
        assert abs(ds[m] - fd) <= 1e-9 * (1 + abs(fd)), m
    for e, n in [(0, 0), (0, 255), (2, 17), (3, 128), (3, 255)]:
        bp, bm = b.copy(), b.copy()
        bp[e, n] += h
        bm[e, n] -= h
        fd = (L(s0, bp) - L(s0, bm)) / (2 * h)
        assert abs(db[e, n] - fd) <= 1e-9 * (1 + abs(fd)), (e, n)
    assert np.all(db[1] == 0)  # the empty expert
    # both sides of <dY, s*b> agree: sum_m s_m ds_m == sum_e <b_e, db_e> == L(s, b)
    tot = L(s0, b)
    assert abs(float(s0 @ ds) - tot) <= 1e-9 * (1 + abs(tot))
    assert abs(float(np.sum(b * db)) - tot) <= 1e-9 * (1 + abs(tot))


def test_scaled_bias_with_unit_scales_is_the_plain_dbias(orc):
    dy_bits, ms, _, bias = _scaled_bias_case(seed=32)
    dy = f32_from_bf16_bits(dy_bits).astype(np.float64)
    db, ds = orc.scaled_bias_grads(dy, ms, np.ones(len(dy), np.float32), bias, dprobs=False)
    assert ds is None
    assert np.array_equal(db, orc.grouped_dbias(dy_bits, ms))
    zero = np.zeros_like(bias)
    _, ds0 = orc.scaled_bias_grads(dy, ms, np.ones(len(dy), np.float32), zero, dbias=False)
    assert np.all(ds0 == 0)


# ------------------------------------------- experts not aligned to 128 rows
def test_padded_grouping_reduces_to_the_aligned_one(orc):
    rng = np.random.default_rng(71)
    ms = np.array([128, 0, 256, 128], np.int64)
    x = bf16_bits_from_f32(rng.standard_normal((512, 256)).astype(np.float32))
    for sw in (False, True):
        a = orc.group_quantize(x, ms, swizzled=sw)
        b = orc.group_quantize_padded(x, ms, swizzled=sw)
        for k in a:
            assert np.array_equal(a[k], b[k]), (sw, k)
    wire = orc.group_quantize(x, ms, rowwise=True, colwise=False)
    a = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, dbias=True, dequant=True)
    b = orc.requant_colwise_padded(wire["row_q"], wire["row_s"], ms, dbias=True, dequant=True)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_padded_partial_colwise_block_by_brute_force(orc):
    # expert 0 has 40 rows: one full 32-row block and a partial block of 8 real rows;
    # expert 1 has 3 rows. Each partial block's scale and codes come from its real rows
    # alone, through the pinned block quantizer
    rng = np.random.default_rng(72)
    ms = np.array([40, 3], np.int64)
    M, K = 43, 128
    x = bf16_bits_from_f32((rng.standard_normal((M, K)) * np.exp2(rng.integers(-3, 3, (M, 1)))).astype(np.float32))
    o = orc.group_quantize_padded(x, ms, rowwise=False, colwise=True, swizzled=False)
    xv = f32_from_bf16_bits(x).astype(np.float64)
    P, _ = orc.padded_offsets(ms)
    assert o["col_s"].shape == (int(P[-1]) // 32, K)
    blocks = [(0, 0, 32, 0), (0, 32, 40, 1), (1, 40, 43, P[1] // 32)]  # (expert, first row, end, scale row)
    for _, r0, r1, srow in blocks:
        for k in range(K):
            codes = np.zeros(r1 - r0, np.uint8)
            code = np.zeros(1, np.uint8)
            orc.lib().orc_quantize_block(orc._p(np.ascontiguousarray(xv[r0:r1, k])), r1 - r0, orc._p(codes),
                                         orc._p(code))
            assert o["col_s"][srow, k] == code[0], (r0, k)
            assert np.array_equal(o["col_q"][r0:r1, k], codes), (r0, k)
    # pad scale rows are zero: rows 2..3 of expert 0 (block rows 2, 3) and 5..7 of expert 1
    used = {0, 1, P[1] // 32}
    for r in range(o["col_s"].shape[0]):
        if r not in used:
            assert np.all(o["col_s"][r] == 0), r


def test_padded_swizzled_layouts_hold_every_scale_once(orc):
    rng = np.random.default_rng(73)
    ms = np.array([200, 0, 57, 128], np.int64)
    M, K = int(ms.sum()), 256
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    c = orc.group_quantize_padded(x, ms, swizzled=False)
    s = orc.group_quantize_padded(x, ms, swizzled=True)
    P, mp = orc.padded_offsets(ms)
    R = int(P[-1])
    # rowwise: the swizzle of the padded (R, K/32) matrix whose real rows are the dense compact scales
    Sp = orc.pad_rows(c["row_s"][:M, :K // 32], ms)
    assert np.array_equal(s["row_s"], orc.swizzle(Sp))
    # colwise: expert e's (K, mp_e/32) matrix at byte K * P_e / 32
    for e in range(len(ms)):
        if mp[e] == 0:
            continue
        Se = c["col_s"][P[e] // 32:(P[e] + mp[e]) // 32].T
        base = K * P[e] // 32
        assert np.array_equal(s["col_s"][base:base + Se.size], orc.swizzle(Se)), e
    assert s["col_s"].size == K * R // 32 and s["row_s"].size == R * K // 32
    # and the codes are the padded ones gathered back
    assert np.array_equal(s["row_q"], c["row_q"]) and np.array_equal(s["col_q"], c["col_q"])


def test_padded_dbias_is_the_plain_column_sum(orc):
    rng = np.random.default_rng(74)
    ms = np.array([33, 0, 95], np.int64)
    dy = bf16_bits_from_f32(rng.standard_normal((128, 256)).astype(np.float32))
    db = orc.grouped_dbias_padded(dy, ms)
    v = f32_from_bf16_bits(dy).astype(np.float64)
    assert np.allclose(db[0], v[:33].sum(axis=0), rtol=0, atol=1e-12)
    assert np.all(db[1] == 0)
    assert np.allclose(db[2], v[33:].sum(axis=0), rtol=0, atol=1e-12)
