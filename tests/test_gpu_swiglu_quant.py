"""GPU parity: SwiGLU fused with group quantization, forward and backward.

The oracle computes SwiGLU in the kernels' fp32 precision (the rounding of h
to bf16 decides the E4M3 codes, so both sides take it in the same precision),
then quantizes with its own group_quantize and reduces dbias in fp64. Codes
and scales must be bit-exact, the optional bf16 outputs equal, dbias within
1e-5 * sum|x| per column."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import bf16_to_f64, dev_bf16, dev_i64, first_diff, host, lib, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def _inputs(M, F, seed):
    rng = np.random.default_rng(seed)
    y = (3 * rng.standard_normal((M, 2 * F))).astype(np.float32)
    y[rng.random((M, 2 * F)) < 0.002] *= 100.0       # saturated gates and big ups
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


CASES = [(512, 256, [128, 256, 0, 128]), (384, 128, [384]), (640, 384, [0, 256, 128, 0, 256])]


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[f"{m}x{f}_E{len(s)}" for m, f, s in CASES])
def test_swiglu_quantize_forward(mxq, case, swz):
    M, F, ms = case
    y, _ = _inputs(M, F, M + F)
    q = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms), swizzle=swz, h_out=True)
    h = orc.swiglu_fwd_f32(y)
    assert np.array_equal(host(q["h"]), h), first_diff(host(q["h"]), h)
    _cmp(q, orc.group_quantize(h, np.array(ms), swizzled=swz), "fwd")


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[f"{m}x{f}_E{len(s)}" for m, f, s in CASES])
def test_swiglu_quantize_backward(mxq, case, swz):
    M, F, ms = case
    y, dh = _inputs(M, F, 7 * M + F)
    q = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), swizzle=swz, dbias=True, dy_out=True)
    dy = orc.swiglu_bwd_f32(dh, y)
    assert np.array_equal(host(q["dy"]), dy), first_diff(host(q["dy"]), dy)
    _cmp(q, orc.group_quantize(dy, np.array(ms), swizzled=swz), "bwd")
    ref = orc.grouped_dbias(dy, np.array(ms))
    got = host(q["dbias"]).astype(np.float64)
    f = np.abs(bf16_to_f64(dy))
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(len(ms)):
        assert np.all(np.abs(got[e] - ref[e]) <= 1e-5 * f[off[e]:off[e + 1]].sum(axis=0) + 1e-30), e


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_swiglu_quantize_single_direction(mxq, rowwise, colwise):
    M, F, ms = 512, 256, [256, 256]
    y, dh = _inputs(M, F, 3)
    q = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms), rowwise=rowwise, colwise=colwise)
    _cmp(q, orc.group_quantize(orc.swiglu_fwd_f32(y), np.array(ms), rowwise=rowwise, colwise=colwise,
                               swizzled=True), "fwd1")
    q = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), rowwise=rowwise, colwise=colwise)
    _cmp(q, orc.group_quantize(orc.swiglu_bwd_f32(dh, y), np.array(ms), rowwise=rowwise, colwise=colwise,
                               swizzled=True), "bwd1")


def test_unfused_swiglu_equals_kernel_precision_definition(mxq):
    M, F = 512, 384
    y, dh = _inputs(M, F, 5)
    assert np.array_equal(host(mxq.swiglu_fwd(dev_bf16(y))), orc.swiglu_fwd_f32(y))
    assert np.array_equal(host(mxq.swiglu_bwd(dev_bf16(dh), dev_bf16(y))), orc.swiglu_bwd_f32(dh, y))


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
    q = mxq.swiglu_quantize(dev_bf16(y), dev_i64(ms))
    _cmp(q, orc.group_quantize(orc.swiglu_fwd_f32(y), ms, swizzled=True), name + " fwd")
    del q
    q = mxq.swiglu_bwd_quantize(dev_bf16(dh), dev_bf16(y), dev_i64(ms), dbias=True)
    dy = orc.swiglu_bwd_f32(dh, y)
    _cmp(q, orc.group_quantize(dy, ms, swizzled=True), name + " bwd")
    ref = orc.grouped_dbias(dy, ms)
    got = host(q["dbias"]).astype(np.float64)
    f = np.abs(bf16_to_f64(dy))
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(w.E):
        assert np.all(np.abs(got[e] - ref[e]) <= 1e-5 * f[off[e]:off[e + 1]].sum(axis=0) + 1e-30), e
