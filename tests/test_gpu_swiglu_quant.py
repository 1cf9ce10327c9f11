"""GPU parity: SwiGLU fused with group quantization, forward and backward.

Two checks together fix every output (the fused kernels write their bf16 h or
dY1 on request, as well as its codes):
  (i)  every bf16 h / dY1 value the kernel produced is within one bf16 step of
       the oracle's fp64 SwiGLU (or its backward) on the same inputs, or within
       the bound of the fp32 sigmoid flush below g = -86 (tests/_gpu.py);
  (ii) the codes and scales equal, byte for byte, the oracle's group_quantize
       of the kernel's own bf16 values, and dbias is within 1e-5 * sum|x| per
       column of the oracle's fp64 per-expert sums of them.
Quantization is exactly defined, so (i) and (ii) leave nothing unchecked."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import (assert_swiglu_close, bf16_to_f64, dev_bf16, dev_i64, first_diff, host, lib, require_gpu,
                        swiglu_bwd_slack, swiglu_fwd_slack)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def _inputs(M, F, seed):
    rng = np.random.default_rng(seed)
    y = (3 * rng.standard_normal((M, 2 * F))).astype(np.float32)
    y[rng.random((M, 2 * F)) < 0.002] *= 100.0       # saturated gates (some below -86) and big ups
    y[:32, :32] = 0.0                                 # all-zero blocks
    y[32:64, F:F + 32] = np.float32(1e-39)            # bf16 subnormal ups
    dh = rng.standard_normal((M, F)).astype(np.float32)
    dh[64:96, :32] = 0.0
    return bf16_bits_from_f32(y), bf16_bits_from_f32(dh)


def _cmp(q, o, what):
    for k, dk in (("row_q", "row_data"), ("row_s", "row_scale"), ("col_q", "col_data"), ("col_s", "col_scale")):
        if o[k] is None or dk not in q:
            continue
        got = host(q[dk]).reshape(o[k].shape)
        assert np.array_equal(got, o[k]), (what, k, first_diff(got, o[k]))


def check_forward(q, y, ms, swizzled, rowwise=True, colwise=True, what="fwd"):
    """(i) q["h"] against the fp64 definition; (ii) codes == group_quantize(q["h"])."""
    h = host(q["h"])
    assert_swiglu_close(h, orc.swiglu_fwd(y), swiglu_fwd_slack(y), what + " h")
    _cmp(q, orc.group_quantize(h, np.asarray(ms), rowwise=rowwise, colwise=colwise, swizzled=swizzled), what)


def check_backward(q, dh, y, ms, swizzled, rowwise=True, colwise=True, dbias=True, what="bwd"):
    """(i) q["dy"] against the fp64 backward; (ii) codes == group_quantize(q["dy"]), dbias of q["dy"]."""
    ms = np.asarray(ms)
    dy = host(q["dy"])
    assert_swiglu_close(dy, orc.swiglu_bwd(dh, y), swiglu_bwd_slack(dh, y), what + " dY1")
    _cmp(q, orc.group_quantize(dy, ms, rowwise=rowwise, colwise=colwise, swizzled=swizzled), what)
    if dbias:
        ref = orc.grouped_dbias(dy, ms)
        got = host(q["dbias"]).astype(np.float64)
        f = np.abs(bf16_to_f64(dy))
        off = np.concatenate([[0], np.cumsum(ms)])
        for e in range(len(ms)):
            assert np.all(np.abs(got[e] - ref[e]) <= 1e-5 * f[off[e]:off[e + 1]].sum(axis=0) + 1e-30), (what, e)


CASES = [(512, 256, [128, 256, 0, 128]), (384, 128, [384]), (640, 384, [0, 256, 128, 0, 256])]


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[f"{m}x{f}_E{len(s)}" for m, f, s in CASES])
def test_swiglu_quantize_forward(mxq, case, swz):
    M, F, ms = case
    y, _ = _inputs(M, F, M + F)
    assert (bf16_to_f64(y)[:, :F] < -86).any()        # the flush branch is exercised
    q = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms), swizzle=swz, h_out=True)
    check_forward(q, y, ms, swz)


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[f"{m}x{f}_E{len(s)}" for m, f, s in CASES])
def test_swiglu_quantize_backward(mxq, case, swz):
    M, F, ms = case
    y, dh = _inputs(M, F, 7 * M + F)
    q = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), swizzle=swz, dbias=True, dy_out=True)
    check_backward(q, dh, y, ms, swz)


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_swiglu_quantize_single_direction(mxq, rowwise, colwise):
    M, F, ms = 512, 256, [256, 256]
    y, dh = _inputs(M, F, 3)
    q = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms), rowwise=rowwise, colwise=colwise, h_out=True)
    check_forward(q, y, ms, True, rowwise=rowwise, colwise=colwise, what="fwd1")
    q = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), rowwise=rowwise, colwise=colwise,
                                dbias=False, dy_out=True)
    check_backward(q, dh, y, ms, True, rowwise=rowwise, colwise=colwise, dbias=False, what="bwd1")


def test_unfused_swiglu_equals_fused(mxq):
    """The unfused kernels run the same fp32 steps: their outputs equal the fused kernels' bf16
    side outputs bit for bit, and both are within the tolerance of the fp64 definition."""
    M, F = 512, 384
    y, dh = _inputs(M, F, 5)
    ms = [M]
    h = host(mxq.swiglu_fwd(dev_bf16(y)))
    dy = host(mxq.swiglu_bwd(dev_bf16(dh), dev_bf16(y)))
    assert_swiglu_close(h, orc.swiglu_fwd(y), swiglu_fwd_slack(y), "h")
    assert_swiglu_close(dy, orc.swiglu_bwd(dh, y), swiglu_bwd_slack(dh, y), "dY1")
    qf = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms), h_out=True)
    qb = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), dbias=False, dy_out=True)
    assert np.array_equal(h, host(qf["h"]))
    assert np.array_equal(dy, host(qb["dy"]))


def test_noop_and_bad_splits(mxq):
    M, F = 256, 128
    y, dh = _inputs(M, F, 9)
    out = {"row_data": torch.full((M, F), 0x11, dtype=torch.uint8, device="cuda"),
           "row_scale": torch.full((mxq.scale_bytes(M, F, False),), 0x11, dtype=torch.uint8, device="cuda"),
           "col_data": torch.full((M, F), 0x11, dtype=torch.uint8, device="cuda"),
           "col_scale": torch.full((mxq.scale_bytes(M, F, True),), 0x11, dtype=torch.uint8, device="cuda")}
    noop = torch.ones(1, dtype=torch.int32, device="cuda")
    mxq.swiglu_quantize(dev_bf16(y), dev_i64([M]), noop=noop, out=out)
    status = mxq.new_status()
    mxq.swiglu_quantize(dev_bf16(y), dev_i64([128, 64, 64]), status=status, out=out)
    assert mxq.status_read(status) & 1
    assert all(bool((v == 0x11).all()) for v in out.values())


@pytest.mark.parametrize("name", ["e64_h3072_f1024_t84k_prequant", "e32_h4096_f1536_t64k_swiglu"])
def test_full_size(mxq, name):
    """FC1 output of the SwiGLU workloads: (M, 2F) with F = 1024 or 1536."""
    w = WORKLOADS[name]
    ms = make_inputs(w, which=())["m_splits"]
    rng = np.random.default_rng(w.wid)
    y = bf16_bits_from_f32((2 * rng.standard_normal((w.M, 2 * w.F))).astype(np.float32))
    dh = bf16_bits_from_f32(rng.standard_normal((w.M, w.F)).astype(np.float32))
    q = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms), h_out=True)
    check_forward(q, y, ms, True, what=name + " fwd")
    del q
    q = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), dbias=True, dy_out=True)
    check_backward(q, dh, y, ms, True, what=name + " bwd")
