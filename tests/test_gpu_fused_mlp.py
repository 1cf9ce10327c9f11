"""GPU parity: FC1 fprop with SwiGLU and the MXFP8 quantization of h in the
GEMM epilogue (the fused grouped MLP's FC1 -> activation, TransformerEngine
PR #3545; quantization as group_quantize, PR #3244 / #3224).

Stage-wise, through the C ABI: y1 (the saved FC1 output) must be bit-identical
to the plain grouped fprop and within the GEMM tolerance of the oracle's fp64
product of the oracle-quantized operands; h's codes and scales must equal,
bit for bit, the oracle's fp32 SwiGLU of the GPU's y1 followed by its
group_quantize, and the standalone fused SwiGLU->quantize kernel on that y1."""
import numpy as np
import pytest

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import dev_bf16, dev_i64, dev_u8, first_diff, host, lib, require_gpu, scaled_error

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
    fused = mxq.grouped_gemm_fprop_swiglu(*args, bias=b, swizzle=swizzle)
    plain = mxq.grouped_gemm_fprop(*args, bias=b)
    return fused, plain


def _check_h(mxq, fused, ms, swizzle):
    y1 = host(fused["y1"])
    h = orc.swiglu_fwd_f32(y1)
    o = orc.group_quantize(h, ms, swizzled=swizzle)
    for dk, ok in (("row_data", "row_q"), ("row_scale", "row_s"), ("col_data", "col_q"), ("col_scale", "col_s")):
        got = host(fused[dk]).reshape(o[ok].shape)
        assert np.array_equal(got, o[ok]), (dk, first_diff(got, o[ok]))
    ref = mxq.swiglu_quantize(fused["y1"], dev_i64(ms), swizzle=swizzle)
    for k in ("row_data", "row_scale", "col_data", "col_scale"):
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
