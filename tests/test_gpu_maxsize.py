"""GPU parity at sizes whose byte offsets pass 2^31 and 2^32: a grouped
tensor of 262,144 x 8,448 (2.2 G elements: its E4M3 codes span 2.2 GB and
its bf16 form 4.4 GB) through group_quantize (+ dbias), requant and the three
grouped GEMMs, through the C ABI, sampled against the oracle around the
2^31-byte row (254,200) and at the ends of both experts.

The GEMM and requant operands are random valid E4M3 codes and E8M0 scales
drawn on the host (tests/_layouts.py; the swizzled scales are the oracle's
swizzle of the compact ones). The bf16 input of group_quantize is a seeded
2,048-row block repeated 128 times, copy j multiplied by 2^s_j (exact in
bf16); the oracle quantizes the same rows on the host. Bar: codes and scales
bit-exact; GEMM entries |C - C*| / (|A|.|B|) <= 8e-3 (bf16 out) or 1e-3
(fp32 dW); dbias within 1e-5 of the column's sum of |x|."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import bf16_bits_from_f32, f32_from_bf16_bits
from tests._gpu import dev_i64, dev_u8, host, lib, require_gpu, scaled_error
from tests._layouts import random_codes, random_scales, swizzle_colwise_grouped, swizzle_rowwise

pytestmark = pytest.mark.gpu

M, K, N, E = 262144, 8448, 256, 2
MS = np.array([131072, 131072], np.int64)
ROW_2_31 = (1 << 31) // K  # first row whose E4M3 codes start past 2^31 bytes
BLOCK = 2048
TOL_BF16, TOL_F32 = 8e-3, 1e-3


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def sample_rows(rng, n_rand=48):
    fixed = [0, 1, 127, 131071, 131072, 131073, ROW_2_31 - 1, ROW_2_31, ROW_2_31 + 1, M - 2, M - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, M, n_rand)])).astype(np.int64)


@pytest.fixture(scope="module")
def ops():
    """Random operands of one grouped linear at the maximum size."""
    rng = np.random.default_rng([11, 2026])
    o = {"xq": random_codes(rng, M * K).reshape(M, K),  # X codes: rowwise for fprop, colwise for wgrad
         "xs_row": random_scales(rng, (M, K // 32)), "xs_col": random_scales(rng, (M // 32, K)),
         "wq_row": random_codes(rng, E * N * K).reshape(E, N, K), "ws_row": random_scales(rng, (E * N, K // 32)),
         "wq_col": random_codes(rng, E * N * K).reshape(E, N, K), "ws_col": random_scales(rng, (E * N // 32, K)),
         "dyq_row": random_codes(rng, M * N).reshape(M, N), "dys_row": random_scales(rng, (M, N // 32)),
         "dyq_col": random_codes(rng, M * N).reshape(M, N), "dys_col": random_scales(rng, (M // 32, N))}
    return o


@pytest.fixture(scope="module")
def xq_dev(ops):
    t = dev_u8(ops["xq"])
    yield t
    del t
    torch.cuda.empty_cache()


def test_fprop_max_size(mxq, ops, xq_dev):
    y = mxq.grouped_gemm_fprop(xq_dev, dev_u8(swizzle_rowwise(ops["xs_row"])), dev_u8(ops["wq_row"]),
                               dev_u8(swizzle_rowwise(ops["ws_row"])), dev_i64(MS))
    rng = np.random.default_rng(1)
    rows = sample_rows(rng)
    cols = np.arange(N)
    got = host(y[torch.from_numpy(rows).cuda()])
    got = f32_from_bf16_bits(got).astype(np.float64)
    r, c = np.meshgrid(rows, cols, indexing="ij")
    ref, mag = orc.fprop_entries(ops["xq"], ops["xs_row"], ops["wq_row"], ops["ws_row"], MS, r.ravel(), c.ravel())
    assert scaled_error(got.ravel(), ref, mag) <= TOL_BF16


def test_dgrad_max_size_output_past_2_32_bytes(mxq, ops):
    dx = mxq.grouped_gemm_dgrad(dev_u8(ops["dyq_row"]), dev_u8(swizzle_rowwise(ops["dys_row"])),
                                dev_u8(ops["wq_col"]), dev_u8(swizzle_colwise_grouped(ops["ws_col"], [N] * E, K)),
                                dev_i64(MS))
    assert dx.shape == (M, K) and dx.numel() * 2 > (1 << 32)
    rng = np.random.default_rng(2)
    rows = sample_rows(rng)
    cols = np.unique(np.concatenate([[0, 1, K - 2, K - 1], rng.integers(0, K, 60)]))
    got = host(dx[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    got = f32_from_bf16_bits(got).astype(np.float64)
    del dx
    torch.cuda.empty_cache()
    r, c = np.meshgrid(rows, cols, indexing="ij")
    ref, mag = orc.dgrad_entries(ops["dyq_row"], ops["dys_row"], ops["wq_col"], ops["ws_col"], MS, r.ravel(),
                                 c.ravel())
    assert scaled_error(got.ravel(), ref, mag) <= TOL_BF16


def test_wgrad_max_size(mxq, ops, xq_dev):
    dw = mxq.grouped_gemm_wgrad(dev_u8(ops["dyq_col"]), dev_u8(swizzle_colwise_grouped(ops["dys_col"], MS, N)),
                                xq_dev, dev_u8(swizzle_colwise_grouped(ops["xs_col"], MS, K)), dev_i64(MS))
    rng = np.random.default_rng(3)
    nn = rng.integers(0, N, 12)
    kk = np.unique(np.concatenate([[0, K - 1], rng.integers(0, K, 30)]))
    e, n, k = np.meshgrid(np.arange(E), nn, kk, indexing="ij")
    got = host(dw)[e.ravel(), n.ravel(), k.ravel()].astype(np.float64)
    ref, mag = orc.wgrad_entries(ops["dyq_col"], ops["dys_col"], ops["xq"], ops["xs_col"], MS, e.ravel(), n.ravel(),
                                 k.ravel())
    assert scaled_error(got, ref, mag) <= TOL_F32


def windows():
    """128-row windows (one tile row) at both ends of each expert and around the 2^31-byte row."""
    return [0, 131072 - 128, 131072, ROW_2_31 // 128 * 128, M - 128]


def test_requant_max_size(mxq, ops, xq_dev):
    r = mxq.requant_colwise(xq_dev, dev_u8(ops["xs_row"]), dev_i64(MS), swizzle=False)
    row_sw = host(r["row_scale_swizzled"])
    for r0 in windows():
        sl = slice(r0, r0 + 128)
        o = orc.requant_colwise(ops["xq"][sl], ops["xs_row"][sl], np.array([128]), swizzled=False)
        assert np.array_equal(host(r["col_data"][r0:r0 + 128]), o["col_q"]), r0
        assert np.array_equal(host(r["col_scale"].view(M // 32, K)[r0 // 32:r0 // 32 + 4]), o["col_s"]), r0
        atoms = (K // 32) // 4 * 512  # one 128-row stripe of the swizzled rowwise scales
        assert np.array_equal(row_sw[r0 // 128 * atoms:(r0 // 128 + 1) * atoms], o["row_s_swizzled"]), r0


def test_group_quantize_and_dbias_max_size(mxq):
    rng = np.random.default_rng(12)
    block = bf16_bits_from_f32(rng.standard_normal((BLOCK, K)).astype(np.float32))
    shifts = [(j * 5) % 9 - 4 for j in range(M // BLOCK)]
    blk = torch.from_numpy(block.view(np.int16)).cuda().view(torch.bfloat16)
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    for j, s in enumerate(shifts):
        x[j * BLOCK:(j + 1) * BLOCK] = blk * (2.0 ** s)  # exact: a power-of-two scaling of bf16
    assert x.numel() * 2 > (1 << 32)
    q = mxq.group_quantize(x, dev_i64(MS), swizzle=False, dbias=True)
    del x
    torch.cuda.empty_cache()
    bf = f32_from_bf16_bits(block)
    for r0 in windows():
        j = r0 // BLOCK
        rows = bf16_bits_from_f32((bf[r0 % BLOCK:r0 % BLOCK + 128] * np.float32(2.0 ** shifts[j])))
        o = orc.group_quantize(rows, np.array([128]))
        assert np.array_equal(host(q["row_data"][r0:r0 + 128]), o["row_q"]), r0
        assert np.array_equal(host(q["row_scale"].view(M, K // 32)[r0:r0 + 128]), o["row_s"]), r0
        assert np.array_equal(host(q["col_data"][r0:r0 + 128]), o["col_q"]), r0
        assert np.array_equal(host(q["col_scale"].view(M // 32, K)[r0 // 32:r0 // 32 + 4]), o["col_s"]), r0
    # dbias of expert e: sum over its copies j of 2^s_j times the block's column sums (fp64)
    colsum = orc.grouped_dbias(block, np.array([BLOCK]))[0]
    colabs = np.abs(bf.astype(np.float64)).sum(axis=0)
    got = host(q["dbias"]).astype(np.float64)
    per = int(MS[0]) // BLOCK
    for e in range(E):
        w = sum(2.0 ** shifts[j] for j in range(e * per, (e + 1) * per))
        assert np.all(np.abs(got[e] - w * colsum) <= 1e-5 * w * colabs + 1e-30), e
