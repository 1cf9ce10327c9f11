"""GPU parity: scaled-bias and routing-scale gradients fused into
group_quantize (bf16 gradient) and requant (rowwise E4M3 wire format),
through the C ABI, against the CPU oracle (TransformerEngine PR #3244: bias
and routing-scale reductions from the dequantized gradient; reading
y = X W_e^T + s_m b_e). Quantized bytes and scales bit-exact; dbias within
1e-5 * sum_m |s_m dY[m,n]| per column; dprobs within 1e-5 * sum_n |dY[m,n] b[n]|
per row (fp32 sums in a fixed order against the oracle's fp64)."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, f32_from_bf16_bits, make_inputs
from tests._gpu import bf16_to_f64, dev_bf16, dev_i64, dev_u8, first_diff, host, lib, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def _probs_bias(M, K, E, seed):
    rng = np.random.default_rng(seed)
    probs = rng.random(M).astype(np.float32)  # routing scales in [0, 1)
    bias = bf16_bits_from_f32((0.02 * rng.standard_normal((E, K))).astype(np.float32))
    return probs, bias


def _dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _check_reductions(got_db, got_ds, vals, ms, probs, bias):
    """vals: the exact gradient values (M, K) in float64."""
    db, ds = orc.scaled_bias_grads(vals, ms, probs, bias, dbias=got_db is not None, dprobs=got_ds is not None)
    off = np.concatenate([[0], np.cumsum(ms)])
    if got_db is not None:
        got = host(got_db).astype(np.float64)
        sv = np.abs(vals) * probs.astype(np.float64)[:, None]
        for e in range(len(ms)):
            tol = 1e-5 * sv[off[e]:off[e + 1]].sum(axis=0) + 1e-30
            assert np.all(np.abs(got[e] - db[e]) <= tol), (e, np.max(np.abs(got[e] - db[e]) - tol))
    if got_ds is not None:
        got = host(got_ds).astype(np.float64)
        b = f32_from_bf16_bits(bias).astype(np.float64)
        for e in range(len(ms)):
            rows = slice(off[e], off[e + 1])
            tol = 1e-5 * (np.abs(vals[rows]) * np.abs(b[e])).sum(axis=1) + 1e-30
            assert np.all(np.abs(got[rows] - ds[rows]) <= tol), e


SHAPES = [
    (512, 512, [128, 256, 0, 128]),
    (384, 1152, [384]),
    (1024, 896, [128] * 8),
    (640, 256, [0, 0, 256, 128, 0, 256]),
]


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{m}x{k}_E{len(s)}" for m, k, s in SHAPES])
def test_quantize_scaled_bias(mxq, shape, swz):
    M, K, ms = shape
    rng = np.random.default_rng(41)
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    probs, bias = _probs_bias(M, K, len(ms), 42)
    q = mxq.group_quantize_scaled_bias(dev_bf16(x), dev_i64(ms), _dev_f32(probs), dev_bf16(bias), swizzle=swz)
    o = orc.group_quantize(x, np.array(ms), swizzled=swz)
    for dk, ok in (("row_data", "row_q"), ("row_scale", "row_s"), ("col_data", "col_q"), ("col_scale", "col_s")):
        got = host(q[dk]).reshape(o[ok].shape)
        assert np.array_equal(got, o[ok]), (dk, first_diff(got, o[ok]))
    _check_reductions(q["dbias"], q["dprobs"], bf16_to_f64(x), np.array(ms), probs, bias)


@pytest.mark.parametrize("dbias,dprobs", [(True, True), (True, False), (False, True)])
def test_scaled_bias_reductions_only(mxq, dbias, dprobs):
    M, K, ms = 768, 640, [256, 0, 384, 128]
    rng = np.random.default_rng(43)
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    probs, bias = _probs_bias(M, K, len(ms), 44)
    q = mxq.group_quantize_scaled_bias(dev_bf16(x), dev_i64(ms), _dev_f32(probs), dev_bf16(bias), rowwise=False,
                                       colwise=False, dbias=dbias, dprobs=dprobs)
    assert set(q) == {k for k, on in (("dbias", dbias), ("dprobs", dprobs)) if on}
    _check_reductions(q.get("dbias"), q.get("dprobs"), bf16_to_f64(x), np.array(ms), probs, bias)


def test_unit_scales_reproduce_the_plain_dbias_bit_for_bit(mxq):
    # s_m = 1: every fused multiply-add s*v + acc rounds exactly like v + acc
    M, K, ms = 1024, 768, [128, 512, 0, 384]
    rng = np.random.default_rng(45)
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    _, bias = _probs_bias(M, K, len(ms), 46)
    q = mxq.group_quantize_scaled_bias(dev_bf16(x), dev_i64(ms), _dev_f32(np.ones(M)), dev_bf16(bias), dprobs=False)
    plain = mxq.group_quantize(dev_bf16(x), dev_i64(ms), dbias=True)
    assert torch.equal(q["dbias"], plain["dbias"])


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("shape", SHAPES[:3], ids=[f"{m}x{k}" for m, k, _ in SHAPES[:3]])
def test_requant_scaled_bias(mxq, shape, swz):
    M, K, ms = shape
    rng = np.random.default_rng(47)
    x = bf16_bits_from_f32((rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, (M, 1)))).astype(np.float32))
    wire = orc.group_quantize(x, np.array(ms), rowwise=True, colwise=False, swizzled=False)
    probs, bias = _probs_bias(M, K, len(ms), 48)
    r = mxq.requant_colwise_scaled_bias(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), _dev_f32(probs),
                                        dev_bf16(bias), swizzle=swz, dequant=True)
    o = orc.requant_colwise(wire["row_q"], wire["row_s"], np.array(ms), swizzled=swz, dequant=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    assert np.array_equal(host(r["col_scale"]).reshape(o["col_s"].shape), o["col_s"])
    assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])
    assert np.array_equal(host(r["dequant"]), o["deq"])
    deq = orc.dequant_rowwise(wire["row_q"], wire["row_s"])
    _check_reductions(r["dbias"], r["dprobs"], deq, np.array(ms), probs, bias)


def test_noop_and_bad_splits_leave_outputs_untouched(mxq):
    M, K, ms = 256, 256, [128, 128]
    rng = np.random.default_rng(49)
    x = dev_bf16(bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32)))
    probs, bias = _probs_bias(M, K, 2, 50)
    out = {"dbias": torch.full((2, K), 7.0, device="cuda"), "dprobs": torch.full((M,), 7.0, device="cuda")}
    noop = torch.ones(1, dtype=torch.int32, device="cuda")
    mxq.group_quantize_scaled_bias(x, dev_i64(ms), _dev_f32(probs), dev_bf16(bias), rowwise=False, colwise=False,
                                   noop=noop, out=out)
    torch.cuda.synchronize()
    assert torch.all(out["dbias"] == 7.0) and torch.all(out["dprobs"] == 7.0)
    status = mxq.new_status()
    mxq.group_quantize_scaled_bias(x, dev_i64([128, 64]), _dev_f32(probs), dev_bf16(bias), rowwise=False,
                                   colwise=False, status=status, out=out)
    assert mxq.status_read(status) & (mxq.mxq.STATUS_SPLIT_UNALIGNED | mxq.mxq.STATUS_SPLIT_SUM)
    assert torch.all(out["dbias"] == 7.0) and torch.all(out["dprobs"] == 7.0)


def test_deterministic(mxq):
    M, K, ms = 1024, 1024, [256, 512, 256]
    rng = np.random.default_rng(51)
    x = dev_bf16(bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32)))
    probs, bias = _probs_bias(M, K, 3, 52)
    p, b = _dev_f32(probs), dev_bf16(bias)
    a = mxq.group_quantize_scaled_bias(x, dev_i64(ms), p, b)
    c = mxq.group_quantize_scaled_bias(x, dev_i64(ms), p, b)
    assert torch.equal(a["dbias"], c["dbias"]) and torch.equal(a["dprobs"], c["dprobs"])


def test_full_size_requant_scaled_bias(mxq):
    """64 experts, 83968 routed rows: the FC2 gradient (3072 wide) arrives
    rowwise-quantized; requant with the scaled-bias reductions of its
    dequantized values, the FC2 bias b2 and seeded routing scales."""
    w = WORKLOADS["e64_h3072_f1024_t84k_prequant"]
    d = make_inputs(w, which=("dy2", "b2"))
    ms = d["m_splits"]
    probs = np.random.default_rng([0, w.wid, 8]).random(w.M).astype(np.float32)
    wire = orc.group_quantize(d["dy2"], ms, rowwise=True, colwise=False, swizzled=False)
    r = mxq.requant_colwise_scaled_bias(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), _dev_f32(probs),
                                        dev_bf16(d["b2"]))
    o = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    assert np.array_equal(host(r["col_scale"]), o["col_s"])
    assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])
    deq = orc.dequant_rowwise(wire["row_q"], wire["row_s"])
    _check_reductions(r["dbias"], r["dprobs"], deq, ms, probs, d["b2"])
