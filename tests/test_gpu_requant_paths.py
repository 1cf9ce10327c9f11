"""Requant's two code paths, through the C ABI, against the oracle.

The requant kernel takes a warp's 32 rows x 128 columns in f16x2 steps when
the block row scales and the resulting column scales lie within the ranges in
which those steps are exact, and in fp32 otherwise; both must give the
oracle's codes and scales bit for bit. The wire format here is built directly
(random non-NaN E4M3 codes, chosen E8M0 row scales) so that each 32-row x
128-column warp tile sits on one side of a boundary of the fast path: row
scale spreads 0, 5 (pass 1's limit), 6, 14 (pass 2's lower limit), 15 and
40; spreads that reach scale code 0; columns whose largest code is 0x01 /
0x03 / 0x07 (a column scale 17 / 16 / 15 below the block's largest row
scale: pass 2's upper limit is 15); all-zero columns and all-zero blocks.
Every requant variant runs on it (swizzled and compact scales, dbias, bf16
dequant, colwise only, scaled bias, padded grouping). Bars: codes, scales and
the dequantized bf16 bit-exact; dbias within 1e-5 of the column's sum of
|value|."""
import numpy as np
import pytest

import oracle as orc
from tests._gpu import bf16_to_f64, dev_i64, dev_u8, first_diff, host, lib, require_gpu
from tests._layouts import random_codes

pytestmark = pytest.mark.gpu

M, K = 1536, 512
MS = np.array([512, 256, 0, 768], np.int64)
SPREADS = [0, 5, 6, 14, 15, 40]
N_CASES = len(SPREADS) + 6


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def wire(seed):
    """Rowwise E4M3 codes (M, K) and compact scales (M, K/32), one boundary case per warp tile."""
    rng = np.random.default_rng([41, seed])
    q = random_codes(rng, M * K).reshape(M, K)
    s = np.zeros((M, K // 32), np.uint8)
    for g in range(M // 32):
        for t in range(K // 128):
            case = (g * (K // 128) + t + seed) % N_CASES
            rows, cols = slice(32 * g, 32 * g + 32), slice(128 * t, 128 * t + 128)
            spread = SPREADS[case] if case < len(SPREADS) else int(rng.integers(0, 4))
            for b in range(4):
                base = int(rng.integers(0, 6)) if case == len(SPREADS) else int(rng.integers(60, 190))
                off = rng.integers(0, spread + 1, 32)
                off[rng.permutation(32)[:2]] = [0, spread]  # the spread is reached exactly
                s[rows, 4 * t + b] = np.minimum(base + off, 254)
            blk = q[rows, cols]
            if case == len(SPREADS) + 1:    # tiny columns: largest code 0x01
                c = rng.choice(128, 6, replace=False)
                blk[:, c] = (blk[:, c] & 0x80) | 0x01
            elif case == len(SPREADS) + 2:  # largest code 0x03
                c = rng.choice(128, 6, replace=False)
                blk[:, c] = (blk[:, c] & 0x80) | rng.integers(0, 4, (32, 6)).astype(np.uint8)
            elif case == len(SPREADS) + 3:  # largest code 0x07
                c = rng.choice(128, 6, replace=False)
                blk[:, c] = (blk[:, c] & 0x80) | rng.integers(0, 8, (32, 6)).astype(np.uint8)
            elif case == len(SPREADS) + 4:  # all-zero columns (either sign of zero)
                c = rng.choice(128, 9, replace=False)
                blk[:, c] = rng.choice(np.array([0x00, 0x80], np.uint8), (32, 9))
            elif case == len(SPREADS) + 5:  # an all-zero block, scale code 0
                b = int(rng.integers(0, 4))
                blk[:, 32 * b:32 * b + 32] = 0
                s[rows, 4 * t + b] = 0
            q[rows, cols] = blk
    return q, s


def _dbias_ok(got, ref, deq_bits, ms):
    deq = bf16_to_f64(deq_bits)
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(len(ms)):
        a = np.abs(deq[off[e]:off[e + 1]]).sum(axis=0)
        assert np.all(np.abs(got[e].astype(np.float64) - ref[e]) <= 1e-5 * a + 1e-30), e


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("swz,dbias,deq,rowsw", [(True, False, False, True), (False, False, False, True),
                                                 (True, True, False, True), (True, False, True, True),
                                                 (False, True, True, False), (True, False, False, False)])
def test_requant_paths_match_the_oracle(mxq, seed, swz, dbias, deq, rowsw):
    q, s = wire(seed)
    r = mxq.requant_colwise(dev_u8(q), dev_u8(s), dev_i64(MS), swizzle=swz, row_scale_swizzled=rowsw, dbias=dbias,
                            dequant=deq)
    o = orc.requant_colwise(q, s, MS, swizzled=swz, dbias=True, dequant=True)
    got = host(r["col_data"])
    assert np.array_equal(got, o["col_q"]), first_diff(got, o["col_q"])
    got = host(r["col_scale"]).reshape(o["col_s"].shape)
    assert np.array_equal(got, o["col_s"]), first_diff(got, o["col_s"])
    if rowsw:
        assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])
    if deq:
        assert np.array_equal(host(r["dequant"]), o["deq"])
    if dbias:
        _dbias_ok(host(r["dbias"]), o["dbias"], o["deq"], MS)


def test_scaled_bias_requant_codes_match_the_oracle(mxq):
    import torch
    q, s = wire(2)
    rng = np.random.default_rng(43)
    probs = torch.from_numpy(rng.random(M).astype(np.float32)).cuda()
    bias = torch.from_numpy(rng.integers(0, 1 << 14, (len(MS), K)).astype(np.int16)).cuda().view(torch.bfloat16)
    r = mxq.requant_colwise_scaled_bias(dev_u8(q), dev_u8(s), dev_i64(MS), probs, bias)
    o = orc.requant_colwise(q, s, MS, swizzled=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    assert np.array_equal(host(r["col_scale"]), o["col_s"])


def test_padded_requant_paths_match_the_oracle(mxq):
    q, s = wire(3)
    ms = np.array([300, 0, 1, 900, 335], np.int64)  # 1536 rows, counts not multiples of 128
    r = mxq.requant_colwise(dev_u8(q), dev_u8(s), dev_i64(ms), dbias=True, pad_experts=True)
    o = orc.requant_colwise_padded(q, s, ms, swizzled=True, dbias=True, dequant=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    ref = np.asarray(o["col_s"]).reshape(-1)
    got = host(r["col_scale"]).reshape(-1)[:ref.size]
    assert np.array_equal(got, ref), first_diff(got, ref)
    _dbias_ok(host(r["dbias"]), o["dbias"], o["deq"], ms)
