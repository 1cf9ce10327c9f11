"""GPU parity: FC1 fprop with SwiGLU and the MXFP8 quantization of h in the
GEMM epilogue, and FC2 dgrad with the SwiGLU backward and the quantization of
dY1 in the epilogue (the fused grouped MLP's FC1 -> activation -> FC2,
TransformerEngine PR #3545; quantization as group_quantize, PR #3244 / #3224).

Stage-wise, through the C ABI: y1 (the saved FC1 output) must be bit-identical
to the plain grouped fprop and within the GEMM tolerance of the oracle's fp64
product of the oracle-quantized operands. The epilogues also write the bf16
h / dY1 they quantize (on request); those values must be within one bf16 step
of the oracle's fp64 SwiGLU (or its backward, on the plain dgrad's dh) or
within the fp32 sigmoid-flush bound, and the codes, scales and dbias must equal
the oracle's group_quantize and per-expert sums of those same values. The
fused results must also equal the standalone fused SwiGLU -> quantize kernels
bit for bit. A last test runs the MLP backward from the saved state the pages
keep (colwise copies, y1) after the rowwise copies were freed."""
import numpy as np
import pytest

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import (assert_swiglu_close, bf16_to_f64, dev_bf16, dev_i64, dev_u8, first_diff, host, lib,
                        require_gpu, scaled_error, swiglu_bwd_slack, swiglu_fwd_slack)

pytestmark = pytest.mark.gpu

TOL_BF16 = 8e-3


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def _operands(ms, F, K, seed, bias=True):
    rng = np.random.default_rng(seed)
    ms = np.asarray(ms, np.int64)
    M, E = int(ms.sum()), len(ms)
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    w1 = bf16_bits_from_f32((0.05 * rng.standard_normal((E, 2 * F, K))).astype(np.float32))
    b1 = bf16_bits_from_f32((0.05 * rng.standard_normal((E, 2 * F))).astype(np.float32)) if bias else None
    return x, w1, b1, ms


def _run(mxq, x, w1, b1, ms, swizzle):
    E, N2, K = w1.shape
    sx = orc.group_quantize(x, ms, rowwise=True, colwise=False, swizzled=True)
    sw = orc.quantize_weights(w1, swizzled=True)
    args = (dev_u8(sx["row_q"]), dev_u8(sx["row_s"]), dev_u8(sw["row_q"]).view(E, N2, K), dev_u8(sw["row_s"]),
            dev_i64(ms))
    b = None if b1 is None else dev_bf16(b1)
    fused = mxq.grouped_gemm_fprop_swiglu(*args, bias=b, swizzle=swizzle, h_out=True)
    plain = mxq.grouped_gemm_fprop(*args, bias=b)
    return fused, plain


def _check_h(mxq, fused, ms, swizzle):
    y1 = host(fused["y1"])
    h = host(fused["h"])
    # (i) the epilogue's h against the fp64 definition on the same y1
    assert_swiglu_close(h, orc.swiglu_fwd(y1), swiglu_fwd_slack(y1), "h")
    # (ii) its codes: the oracle's quantization of that h
    o = orc.group_quantize(h, ms, swizzled=swizzle)
    for dk, ok in (("row_data", "row_q"), ("row_scale", "row_s"), ("col_data", "col_q"), ("col_scale", "col_s")):
        got = host(fused[dk]).reshape(o[ok].shape)
        assert np.array_equal(got, o[ok]), (dk, first_diff(got, o[ok]))
    # the standalone fused kernel on the same y1 gives the same bits
    ref = mxq.swiglu_quantize(fused["y1"], dev_i64(ms), swizzle=swizzle, h_out=True)
    for k in ("h", "row_data", "row_scale", "col_data", "col_scale"):
        assert np.array_equal(host(fused[k]), host(ref[k])), k


CASES = [
    ([128, 256, 0, 128], 256, 512),
    ([384], 128, 256),
    ([128] * 4, 384, 384),
    ([0, 256, 0, 128], 512, 1152),
]


@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[f"E{len(s)}_F{f}_K{k}" for s, f, k in CASES])
def test_fprop_swiglu_stagewise(mxq, case, swizzle):
    splits, F, K = case
    x, w1, b1, ms = _operands(splits, F, K, 61)
    fused, plain = _run(mxq, x, w1, b1, ms, swizzle)
    assert np.array_equal(host(fused["y1"]), host(plain)), "y1 differs from the plain fprop"
    # y1 against the oracle's fp64 product (every entry)
    M, E = int(ms.sum()), len(ms)
    cx = orc.group_quantize(x, ms)
    cw = orc.quantize_weights(w1)
    r, c = np.meshgrid(np.arange(M), np.arange(2 * F), indexing="ij")
    ref, mag = orc.fprop_entries(cx["row_q"], cx["row_s"], cw["row_q"].reshape(E, 2 * F, K), cw["row_s"], ms,
                                 r.ravel(), c.ravel(), bias=b1)
    y1 = (host(fused["y1"]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert scaled_error(y1.ravel(), ref, mag) <= TOL_BF16
    _check_h(mxq, fused, ms, swizzle)


def test_fprop_swiglu_without_bias(mxq):
    x, w1, _, ms = _operands([256, 128], 256, 256, 62, bias=False)
    fused, plain = _run(mxq, x, w1, None, ms, True)
    assert np.array_equal(host(fused["y1"]), host(plain))
    _check_h(mxq, fused, ms, True)


def test_full_size_fprop_swiglu(mxq):
    """64 experts, 83968 routed rows, hidden 3072, F = 1024, with the FC1 bias."""
    w = WORKLOADS["e64_h3072_f1024_t84k_prequant"]
    d = make_inputs(w, which=("x", "w", "b1"))
    ms = d["m_splits"]
    fused, plain = _run(mxq, d["x"], d["w"], d["b1"], ms, True)
    assert np.array_equal(host(fused["y1"]), host(plain))
    del plain
    _check_h(mxq, fused, ms, True)


# ------------------------------------------------ FC2 dgrad + SwiGLU backward
def _bwd_operands(ms, F, H, seed):
    rng = np.random.default_rng(seed)
    ms = np.asarray(ms, np.int64)
    M, E = int(ms.sum()), len(ms)
    dy2 = bf16_bits_from_f32(rng.standard_normal((M, H)).astype(np.float32))
    w2 = bf16_bits_from_f32((0.05 * rng.standard_normal((E, H, F))).astype(np.float32))
    y1 = bf16_bits_from_f32((2.0 * rng.standard_normal((M, 2 * F))).astype(np.float32))
    return dy2, w2, y1, ms


def _run_bwd(mxq, dy2, w2, y1, ms, swizzle):
    E, H, F = w2.shape
    sdy = orc.group_quantize(dy2, ms, rowwise=True, colwise=False, swizzled=True)
    sw = orc.quantize_weights(w2, swizzled=True)
    args = (dev_u8(sdy["row_q"]), dev_u8(sdy["row_s"]), dev_u8(sw["col_q"]).view(E, H, F), dev_u8(sw["col_s"]))
    y1d = dev_bf16(y1)
    fused = mxq.grouped_gemm_dgrad_swiglu(*args, y1d, dev_i64(ms), swizzle=swizzle, dy_out=True)
    dh = mxq.grouped_gemm_dgrad(*args, dev_i64(ms))
    ref = mxq.swiglu_bwd_quantize(dh, y1d, dev_i64(ms), swizzle=swizzle, dbias=True, dy_out=True)
    return fused, dh, ref


def _check_bwd(fused, dh, ref, y1, ms, swizzle):
    dy1 = host(fused["dy"])
    dhh = host(dh)
    # (i) the epilogue's dY1 against the fp64 backward on the plain dgrad's dh and y1
    assert_swiglu_close(dy1, orc.swiglu_bwd(dhh, y1), swiglu_bwd_slack(dhh, y1), "dY1")
    # (ii) its codes and dbias: the oracle's quantization and per-expert sums of that dY1
    o = orc.group_quantize(dy1, ms, swizzled=swizzle)
    for dk, ok in (("row_data", "row_q"), ("row_scale", "row_s"), ("col_data", "col_q"), ("col_scale", "col_s")):
        got = host(fused[dk]).reshape(o[ok].shape)
        assert np.array_equal(got, o[ok]), (dk, first_diff(got, o[ok]))
        assert np.array_equal(host(fused[dk]), host(ref[dk])), dk
    assert np.array_equal(dy1, host(ref["dy"]))
    db = orc.grouped_dbias(dy1, ms)
    a = np.abs(bf16_to_f64(dy1))
    off = np.concatenate([[0], np.cumsum(ms)])
    got = host(fused["dbias"]).astype(np.float64)
    for e in range(len(ms)):
        tol = 1e-5 * a[off[e]:off[e + 1]].sum(axis=0) + 1e-30
        assert np.all(np.abs(got[e] - db[e]) <= tol), e


BWD_CASES = [
    ([128, 256, 0, 128], 256, 512),
    ([384], 512, 256),
    ([128] * 4, 256, 384),
]


@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("case", BWD_CASES, ids=[f"E{len(s)}_F{f}_H{h}" for s, f, h in BWD_CASES])
def test_dgrad_swiglu_stagewise(mxq, case, swizzle):
    splits, F, H = case
    dy2, w2, y1, ms = _bwd_operands(splits, F, H, 63)
    fused, dh, ref = _run_bwd(mxq, dy2, w2, y1, ms, swizzle)
    _check_bwd(fused, dh, ref, y1, ms, swizzle)


def test_full_size_dgrad_swiglu(mxq):
    """64 experts, 83968 routed rows: FC2 dgrad (hidden 3072 -> F = 1024) with the SwiGLU
    backward of a synthetic saved FC1 output."""
    w = WORKLOADS["e64_h3072_f1024_t84k_prequant"]
    d = make_inputs(w, which=("dy2", "w2"))
    ms = d["m_splits"]
    y1 = bf16_bits_from_f32((2.0 * np.random.default_rng([0, w.wid, 9]).standard_normal((w.M, 2 * w.F)))
                            .astype(np.float32))
    fused, dh, ref = _run_bwd(mxq, d["dy2"], d["w2"], y1, ms, True)
    _check_bwd(fused, dh, ref, y1, ms, True)


# ------------------------------------------------ saved state of the fused MLP
def _mlp_forward(mxq, x, w1q, w2q, ms, E, F, H):
    """Forward of FC1 -> SwiGLU -> FC2 from bf16 X: X quantized row + col, FC1 with the SwiGLU
    epilogue (h row + col), FC2 on h's rowwise copy."""
    qx = mxq.group_quantize(x, ms)
    fc1 = mxq.grouped_gemm_fprop_swiglu(qx["row_data"], qx["row_scale"], w1q["row_data"].view(E, 2 * F, H),
                                        w1q["row_scale"], ms)
    y2 = mxq.grouped_gemm_fprop(fc1["row_data"], fc1["row_scale"], w2q["row_data"].view(E, H, F), w2q["row_scale"],
                                ms)
    return qx, fc1, y2


def _mlp_backward(mxq, saved, dy2, w1q, w2q, ms, E, F, H):
    """Backward from the saved state only: X's and h's colwise copies and y1 (plus the weights'
    colwise copies and the incoming gradient)."""
    qd = mxq.group_quantize(dy2, ms)
    dh = mxq.grouped_gemm_dgrad(qd["row_data"], qd["row_scale"], w2q["col_data"].view(E, H, F), w2q["col_scale"], ms)
    dw2 = mxq.grouped_gemm_wgrad(qd["col_data"], qd["col_scale"], saved["h_col"], saved["h_col_s"], ms)
    q1 = mxq.swiglu_bwd_quantize(dh, saved["y1"], ms, dbias=True)
    dx = mxq.grouped_gemm_dgrad(q1["row_data"], q1["row_scale"], w1q["col_data"].view(E, 2 * F, H), w1q["col_scale"],
                                ms)
    dw1 = mxq.grouped_gemm_wgrad(q1["col_data"], q1["col_scale"], saved["x_col"], saved["x_col_s"], ms)
    return {"dx": dx, "dw1": dw1, "dw2": dw2, "db1": q1["dbias"]}


def test_backward_from_colwise_saved_state(mxq):
    """[FM]'s saved-state trim: every wgrad reads only colwise tiles and every dgrad only rowwise
    gradients, so after the forward the rowwise copies of X and h can be freed. Backward from the
    colwise copies and y1 alone, with the freed memory overwritten, must give the same dX, dW1,
    dW2 and dbias bits as backward with every forward tensor kept."""
    import torch

    ms_list = [256, 0, 384, 128, 256]
    E, F, H = len(ms_list), 256, 512
    ms = dev_i64(ms_list)
    M = sum(ms_list)
    rng = np.random.default_rng(77)
    x = dev_bf16(bf16_bits_from_f32(rng.standard_normal((M, H)).astype(np.float32)))
    dy2 = dev_bf16(bf16_bits_from_f32(rng.standard_normal((M, H)).astype(np.float32)))
    w1 = dev_bf16(bf16_bits_from_f32((0.05 * rng.standard_normal((E * 2 * F, H))).astype(np.float32)))
    w2 = dev_bf16(bf16_bits_from_f32((0.05 * rng.standard_normal((E * H, F))).astype(np.float32)))
    w1q = mxq.group_quantize(w1, None, E=E)
    w2q = mxq.group_quantize(w2, None, E=E)

    # reference: everything from the forward kept alive
    qx, fc1, y2 = _mlp_forward(mxq, x, w1q, w2q, ms, E, F, H)
    full = _mlp_backward(mxq, {"h_col": fc1["col_data"], "h_col_s": fc1["col_scale"], "y1": fc1["y1"],
                               "x_col": qx["col_data"], "x_col_s": qx["col_scale"]}, dy2, w1q, w2q, ms, E, F, H)
    full = {k: v.clone() for k, v in full.items()}
    del qx, fc1, y2

    # trimmed: keep the colwise copies and y1, free the rest, scribble over the freed memory
    qx, fc1, y2 = _mlp_forward(mxq, x, w1q, w2q, ms, E, F, H)
    saved = {"h_col": fc1["col_data"], "h_col_s": fc1["col_scale"], "y1": fc1["y1"], "x_col": qx["col_data"],
             "x_col_s": qx["col_scale"]}
    freed = [qx["row_data"], qx["row_scale"], fc1["row_data"], fc1["row_scale"], y2]
    sizes = [t.numel() * t.element_size() for t in freed]
    del qx, fc1, y2, freed
    # same-sized blocks: the caching allocator hands the freed ones back
    junk = [torch.full((n,), 0x7E, dtype=torch.uint8, device="cuda") for n in sizes]
    trimmed = _mlp_backward(mxq, saved, dy2, w1q, w2q, ms, E, F, H)
    torch.cuda.synchronize()
    del junk
    for k in full:
        a, b = full[k], trimmed[k]
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), k
