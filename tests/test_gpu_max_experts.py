"""GPU parity at the expert-count limits, through the C ABI, against the
oracle: 1024 experts (MXQ_MAX_EXPERTS, 128-aligned, most of them empty)
through group_quantize + dbias, requant and the three GEMMs; 512 experts
(the padded-grouping GEMM's limit) with expert counts that are not multiples
of 128 through the padded quantizer and the padded GEMMs; one expert more
than each limit is rejected before any launch. Bars as in the other parity
tests: codes and scales bit-exact, GEMM entries |C - C*| / (|A|.|B|) <= 8e-3
(bf16) or 1e-3 (fp32 dW), empty experts' dW exactly 0, dbias within 1e-5 of
the column's sum of |x|."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import bf16_bits_from_f32
from tests._gpu import bf16_to_f64, dev_bf16, dev_i64, dev_u8, first_diff, host, lib, require_gpu, scaled_error
from tests.test_gpu_gemm import TOL_BF16, TOL_F32, Operands, f64
from tests.test_gpu_padded import PaddedOps, _check_padded_gemms

pytestmark = pytest.mark.gpu

E_MAX, E_MAX_PADDED = 1024, 512


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def _aligned_splits(seed, busy=40):
    rng = np.random.default_rng(seed)
    ms = np.zeros(E_MAX, np.int64)
    hot = np.unique(np.concatenate([[0, E_MAX - 1], rng.choice(E_MAX, busy, replace=False)]))
    ms[hot] = 128
    return ms


@pytest.fixture(scope="module")
def aligned():
    ms = _aligned_splits(7)
    M, N, K = int(ms.sum()), 256, 256
    rng = np.random.default_rng(8)
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    w = bf16_bits_from_f32((0.02 * rng.standard_normal((E_MAX, N, K))).astype(np.float32))
    dy = bf16_bits_from_f32(rng.standard_normal((M, N)).astype(np.float32))
    return Operands(x, w, dy, ms), x


def test_quantize_requant_dbias_at_1024_experts(mxq, aligned):
    op, x = aligned
    ms = op.ms
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), dbias=True)
    for dk, ok in (("row_data", "row_q"), ("row_scale", "row_s"), ("col_data", "col_q"), ("col_scale", "col_s")):
        got = host(q[dk]).reshape(op.sx[ok].shape)
        assert np.array_equal(got, op.sx[ok]), (dk, first_diff(got, op.sx[ok]))
    db = orc.grouped_dbias(x, ms)
    got = host(q["dbias"]).astype(np.float64)
    off = np.concatenate([[0], np.cumsum(ms)])
    xa = np.abs(bf16_to_f64(x))
    for e in range(E_MAX):
        tol = 1e-5 * xa[off[e]:off[e + 1]].sum(axis=0) + 1e-30
        assert np.all(np.abs(got[e] - db[e]) <= tol), e
    wire = orc.group_quantize(x, ms, rowwise=True, colwise=False)
    r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms))
    o = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    assert np.array_equal(host(r["col_scale"]), o["col_s"])
    assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])


def test_gemms_at_1024_experts(mxq, aligned):
    op, _ = aligned
    M, N, K, E = op.M, op.N, op.K, op.E
    r, c = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, mag = op.ref_fprop(r.ravel(), c.ravel())
    assert scaled_error(f64(op.gpu_fprop(mxq)).ravel(), ref, mag) <= TOL_BF16
    r, c = np.meshgrid(np.arange(M), np.arange(K), indexing="ij")
    ref, mag = op.ref_dgrad(r.ravel(), c.ravel())
    assert scaled_error(f64(op.gpu_dgrad(mxq)).ravel(), ref, mag) <= TOL_BF16
    dw = op.gpu_wgrad(mxq)
    busy = np.flatnonzero(op.ms)
    empty = torch.from_numpy(op.ms == 0).cuda()
    assert float(dw[empty].abs().max()) == 0.0  # every empty expert's dW is written as zeros
    got = f64(dw[torch.from_numpy(busy).cuda()])
    e, n, k = (a.ravel() for a in np.meshgrid(busy, np.arange(N), np.arange(K), indexing="ij"))
    ref, mag = op.ref_wgrad(e, n, k)
    pos = np.searchsorted(busy, e)
    assert scaled_error(got[pos, n, k], ref, mag) <= TOL_F32


def test_padded_grouping_at_512_experts(mxq):
    rng = np.random.default_rng(17)
    ms = rng.integers(0, 25, E_MAX_PADDED)
    ms[[0, 5, E_MAX_PADDED - 1]] = [0, 130, 1]
    op = PaddedOps(ms, 256, 256, 18)
    x = bf16_bits_from_f32(np.random.default_rng(19).standard_normal((op.M, 256)).astype(np.float32))
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), dbias=True, pad_experts=True)
    o = orc.group_quantize_padded(x, ms, swizzled=True)
    assert np.array_equal(host(q["row_data"]), o["row_q"])
    assert np.array_equal(host(q["col_data"]), o["col_q"])
    for dk, ok in (("row_scale", "row_s"), ("col_scale", "col_s")):
        ref = np.asarray(o[ok]).reshape(-1)
        got = host(q[dk]).reshape(-1)[:ref.size]
        assert np.array_equal(got, ref), (dk, first_diff(got, ref))
    _check_padded_gemms(mxq, op, nk_samples=20000)


def test_one_expert_past_each_limit_is_rejected(mxq):
    x = dev_bf16(np.zeros((128, 128), np.uint16))
    with pytest.raises(mxq.MXQError):
        mxq.group_quantize(x, dev_i64(np.r_[128, np.zeros(E_MAX, np.int64)]))
    ms = dev_i64(np.r_[128, np.zeros(E_MAX_PADDED, np.int64)])
    E = E_MAX_PADDED + 1
    a = dev_u8(np.zeros((128, 256), np.uint8))
    with pytest.raises(mxq.MXQError):
        mxq.grouped_gemm_fprop(a, dev_u8(np.zeros(128 * 8, np.uint8)), dev_u8(np.zeros((E, 256, 256), np.uint8)),
                               dev_u8(np.zeros(E * 256 * 8, np.uint8)), ms, pad_experts=True)
