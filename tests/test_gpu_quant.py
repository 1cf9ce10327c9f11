"""GPU parity: group_quantize, requant_colwise, grouped_dbias and SwiGLU
against the CPU oracle, through the C ABI. Quantized bytes and scales must be
bit-exact; dbias within 1e-5 * sum|x| per column; SwiGLU within one bf16 step
of the oracle's fp64 definition (fp32 math on the GPU, one final rounding each;
the fp32 sigmoid flush below g = -86 has its own bound, tests/_gpu.py)."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import (assert_swiglu_close, bf16_to_f64, dev_bf16, dev_i64, dev_u8, first_diff, host, lib, require_gpu,
                        swiglu_bwd_slack, swiglu_fwd_slack)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def stress_bits(M, K, seed, kind):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        x = rng.standard_normal((M, K)).astype(np.float32)
    else:
        x = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-20, 20, (M, K)))).astype(np.float32)
        x[rng.random((M, K)) < 0.002] *= 1000.0
        x[rng.random((M, K)) < 0.01] = -0.0
        # exact RNE ties of the E4M3 cast: 1 + 1/16 (and odd multiples) times 2^k
        ties = rng.random((M, K)) < 0.05
        x[ties] = (np.float32(1.0625) * rng.choice([1, 3, 5, -1, -3], ties.sum())).astype(np.float32)
        x[:32, :32] = 0.0                                # all-zero row and column blocks
        x[32:64, 32:64] = np.float32(1e-40)              # bf16 subnormals
        x[64:96, 64:96] = np.float32(3e38)               # near the top of bf16
        x[96:128, :32] = rng.standard_normal((32, 32)).astype(np.float32) * np.float32(1e-38)
    return bf16_bits_from_f32(x)


SMALL = [
    (512, 512, [128, 256, 0, 128]),
    (384, 384, [384]),
    (256, 128, [0, 256, 0]),
    (1024, 896, [128] * 8),
    (128, 128, [128]),
    (640, 1152, [0, 0, 256, 128, 0, 256]),
]


def _compare_quant(q, o, what=""):
    for k in ("row_q", "row_s", "col_q", "col_s"):
        dk = {"row_q": "row_data", "row_s": "row_scale", "col_q": "col_data", "col_s": "col_scale"}[k]
        if o[k] is None:
            continue
        got = host(q[dk]).reshape(o[k].shape)
        assert np.array_equal(got, o[k]), (what, k, first_diff(got, o[k]))


@pytest.mark.parametrize("kind", ["normal", "stress"])
@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("shape", SMALL, ids=[f"{m}x{k}_E{len(s)}" for m, k, s in SMALL])
def test_group_quantize_bit_exact(mxq, shape, swz, kind):
    M, K, ms = shape
    x = stress_bits(M, K, M + K, kind)
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), swizzle=swz)
    o = orc.group_quantize(x, np.array(ms), swizzled=swz)
    _compare_quant(q, o, shape)


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_group_quantize_single_direction(mxq, rowwise, colwise):
    x = stress_bits(512, 256, 3, "stress")
    ms = [256, 0, 256]
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), rowwise=rowwise, colwise=colwise)
    o = orc.group_quantize(x, np.array(ms), rowwise=rowwise, colwise=colwise, swizzled=True)
    assert set(q) == ({"row_data", "row_scale"} if rowwise else {"col_data", "col_scale"})
    _compare_quant(q, o)


def test_uniform_members_weights(mxq):
    E, N, K = 4, 256, 384
    w = bf16_bits_from_f32((0.02 * np.random.default_rng(5).standard_normal((E, N, K))).astype(np.float32))
    q = mxq.group_quantize(dev_bf16(w).view(E * N, K), None, E=E)
    o = orc.quantize_weights(w, swizzled=True)
    _compare_quant(q, o)


@pytest.mark.parametrize("shape", SMALL[:4], ids=[f"{m}x{k}" for m, k, _ in SMALL[:4]])
def test_fused_dbias(mxq, shape):
    M, K, ms = shape
    x = stress_bits(M, K, 7, "normal")
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), dbias=True)
    ref = orc.grouped_dbias(x, np.array(ms))
    got = host(q["dbias"]).astype(np.float64)
    f = np.abs(bf16_to_f64(x))
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(len(ms)):
        tol = 1e-5 * f[off[e]:off[e + 1]].sum(axis=0) + 1e-30
        assert np.all(np.abs(got[e] - ref[e]) <= tol), e
        if ms[e] == 0:
            assert np.all(got[e] == 0)
    _compare_quant(q, orc.group_quantize(x, np.array(ms), swizzled=True))


def test_standalone_dbias(mxq):
    M, N, ms = 1024, 640, [256, 0, 512, 256]
    dy = stress_bits(M, N, 9, "normal")
    got = host(mxq.grouped_dbias(dev_bf16(dy), dev_i64(ms))).astype(np.float64)
    ref = orc.grouped_dbias(dy, np.array(ms))
    f = np.abs(bf16_to_f64(dy))
    off = np.concatenate([[0], np.cumsum(ms)])
    for e in range(len(ms)):
        assert np.all(np.abs(got[e] - ref[e]) <= 1e-5 * f[off[e]:off[e + 1]].sum(axis=0) + 1e-30)
    assert np.all(got[1] == 0)


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("shape", SMALL[:4], ids=[f"{m}x{k}" for m, k, _ in SMALL[:4]])
def test_requant_bit_exact(mxq, shape, swz):
    M, K, ms = shape
    x = stress_bits(M, K, 11, "stress")
    wire = orc.group_quantize(x, np.array(ms), rowwise=True, colwise=False, swizzled=False)
    r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), swizzle=swz, dbias=True,
                            dequant=True)
    o = orc.requant_colwise(wire["row_q"], wire["row_s"], np.array(ms), swizzled=swz, dbias=True, dequant=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    assert np.array_equal(host(r["col_scale"]).reshape(o["col_s"].shape), o["col_s"])
    assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])
    assert np.array_equal(host(r["dequant"]), o["deq"])
    deq = bf16_to_f64(o["deq"])
    off = np.concatenate([[0], np.cumsum(ms)])
    got = host(r["dbias"]).astype(np.float64)
    for e in range(len(ms)):
        a = np.abs(deq[off[e]:off[e + 1]]).sum(axis=0)
        fits = a < 1e37          # the stress input's ~3e38 block overflows an fp32 dbias by design
        tol = 1e-5 * a + 1e-30
        assert np.all(np.abs(got[e] - o["dbias"][e])[fits] <= tol[fits])


def test_requant_colwise_only(mxq):
    M, K, ms = 512, 256, [128, 384]
    x = stress_bits(M, K, 12, "normal")
    wire = orc.group_quantize(x, np.array(ms), rowwise=True, colwise=False, swizzled=False)
    r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), row_scale_swizzled=False)
    o = orc.requant_colwise(wire["row_q"], wire["row_s"], np.array(ms), swizzled=True)
    assert set(r) == {"col_data", "col_scale"}
    assert np.array_equal(host(r["col_data"]), o["col_q"]) and np.array_equal(host(r["col_scale"]), o["col_s"])


def test_noop_flag_writes_nothing(mxq):
    x = stress_bits(256, 256, 13, "normal")
    ms = dev_i64([256])
    out = {k: torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda") for k, n in
           (("row_data", 256 * 256), ("col_data", 256 * 256), ("row_scale", 2048), ("col_scale", 2048))}
    out["row_data"] = out["row_data"].view(256, 256)
    out["col_data"] = out["col_data"].view(256, 256)
    noop = torch.ones(1, dtype=torch.int32, device="cuda")
    mxq.group_quantize(dev_bf16(x), ms, noop=noop, out=out)
    torch.cuda.synchronize()
    assert all(bool((v == 0xA5).all()) for v in out.values())
    noop.zero_()
    mxq.group_quantize(dev_bf16(x), ms, noop=noop, out=out)
    _compare_quant(out, orc.group_quantize(x, np.array([256]), swizzled=True))


@pytest.mark.parametrize("bad,bits", [([128, 64, 64], 1), ([384, -128], 2), ([128, 0], 4)])
def test_invalid_splits_set_status_and_skip(mxq, bad, bits):
    x = stress_bits(256, 128, 14, "normal")
    status = mxq.new_status()
    out = {"row_data": torch.full((256, 128), 0x5A, dtype=torch.uint8, device="cuda"),
           "row_scale": torch.full((1024,), 0x5A, dtype=torch.uint8, device="cuda"),
           "col_data": torch.full((256, 128), 0x5A, dtype=torch.uint8, device="cuda"),
           "col_scale": torch.full((1024,), 0x5A, dtype=torch.uint8, device="cuda")}
    mxq.group_quantize(dev_bf16(x), dev_i64(bad), status=status, out=out)
    got = mxq.status_read(status)
    assert got & bits == bits, got
    assert all(bool((v == 0x5A).all()) for v in out.values())


def test_host_m_splits_rejected_at_the_abi(mxq):
    import ctypes

    L = mxq.mxq.lib()
    x = dev_bf16(stress_bits(256, 128, 15, "normal"))
    host_splits = np.array([256], np.int64)
    rq = torch.empty((256, 128), dtype=torch.uint8, device="cuda")
    rs = torch.empty(1024, dtype=torch.uint8, device="cuda")
    rc = L.mxq_group_quantize(x.data_ptr(), 256, 128, 1, host_splits.ctypes.data_as(ctypes.c_void_p), 1 | 4,
                              rq.data_ptr(), rs.data_ptr(), None, None, None, None, None, None, 0,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == -3
    rc = L.mxq_group_quantize(x.data_ptr(), 256, 100, 1, None, 1, rq.data_ptr(), rs.data_ptr(), None, None, None,
                              None, None, None, 0, None)
    assert rc == -2


def test_empty_input(mxq):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q = mxq.group_quantize(x, dev_i64([0, 0]))
    torch.cuda.synchronize()
    assert q["row_data"].numel() == 0


def test_deterministic(mxq):
    x = dev_bf16(stress_bits(1024, 512, 16, "normal"))
    ms = dev_i64([512, 512])
    a = mxq.group_quantize(x, ms, dbias=True)
    b = mxq.group_quantize(x, ms, dbias=True)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_swiglu(mxq):
    rng = np.random.default_rng(17)
    M, F = 384, 1536
    y = bf16_bits_from_f32((3 * rng.standard_normal((M, 2 * F))).astype(np.float32))
    dh = bf16_bits_from_f32(rng.standard_normal((M, F)).astype(np.float32))
    h = host(mxq.swiglu_fwd(dev_bf16(y)))
    dy = host(mxq.swiglu_bwd(dev_bf16(dh), dev_bf16(y)))
    assert_swiglu_close(h, orc.swiglu_fwd(y), swiglu_fwd_slack(y), "h")
    assert_swiglu_close(dy, orc.swiglu_bwd(dh, y), swiglu_bwd_slack(dh, y), "dY1")


# ---------------------------------------------------------------- full size
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_quantize_activation(mxq, name):
    """The first grouped linear's activation X of every workload, full size."""
    w = WORKLOADS[name]
    d = make_inputs(w, which=("x",))
    x, ms = d["x"], d["m_splits"]
    if w.prequant_x:
        wire = orc.group_quantize(x, ms, rowwise=True, colwise=False, swizzled=False)
        r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms))
        o = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=True)
        assert np.array_equal(host(r["col_data"]), o["col_q"])
        assert np.array_equal(host(r["col_scale"]), o["col_s"])
        assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])
    else:
        q = mxq.group_quantize(dev_bf16(x), dev_i64(ms))
        _compare_quant(q, orc.group_quantize(x, ms, swizzled=True), name)


def _dbias_ok(got, ref, src_abs_colsum):
    return np.all(np.abs(got - ref) <= 1e-5 * src_abs_colsum + 1e-30)


def test_full_size_mlp_backward_quantizers(mxq):
    """64 experts, 83968 routed rows: requant of the rowwise-prequantized FC2
    gradient (3072 wide) with fused dbias, and group_quantize of the FC1
    gradient (2048 wide, synthetic) with fused dbias."""
    w = WORKLOADS["e64_h3072_f1024_t84k_prequant"]
    d = make_inputs(w, which=("dy", "dy2"))
    ms = d["m_splits"]
    off = np.concatenate([[0], np.cumsum(ms)])
    # FC2 grad arrives rowwise-quantized (the combine's backward)
    wire = orc.group_quantize(d["dy2"], ms, rowwise=True, colwise=False, swizzled=False)
    r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), dbias=True)
    o = orc.requant_colwise(wire["row_q"], wire["row_s"], ms, swizzled=True, dbias=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    assert np.array_equal(host(r["col_scale"]), o["col_s"])
    assert np.array_equal(host(r["row_scale_swizzled"]), o["row_s_swizzled"])
    deq = orc.dequant_rowwise(wire["row_q"], wire["row_s"])
    got = host(r["dbias"]).astype(np.float64)
    for e in range(w.E):
        assert _dbias_ok(got[e], o["dbias"][e], np.abs(deq[off[e]:off[e + 1]]).sum(axis=0)), e
    del deq
    # FC1 grad (M, 2F) quantized row+col with fused dbias
    q = mxq.group_quantize(dev_bf16(d["dy"]), dev_i64(ms), dbias=True)
    _compare_quant(q, orc.group_quantize(d["dy"], ms, swizzled=True), "dY1")
    ref = orc.grouped_dbias(d["dy"], ms)
    got = host(q["dbias"]).astype(np.float64)
    f = np.abs(bf16_to_f64(d["dy"]))
    for e in range(w.E):
        assert _dbias_ok(got[e], ref[e], f[off[e]:off[e + 1]].sum(axis=0)), e


def test_full_size_swiglu(mxq):
    """SwiGLU fwd/bwd at 83968 x (2 x 1024)."""
    rng = np.random.default_rng(18)
    M, F = 83968, 1024
    y = bf16_bits_from_f32((2 * rng.standard_normal((M, 2 * F))).astype(np.float32))
    dh = bf16_bits_from_f32(rng.standard_normal((M, F)).astype(np.float32))
    h = host(mxq.swiglu_fwd(dev_bf16(y)))
    dy = host(mxq.swiglu_bwd(dev_bf16(dh), dev_bf16(y)))
    assert_swiglu_close(h, orc.swiglu_fwd(y), swiglu_fwd_slack(y), "h")
    assert_swiglu_close(dy, orc.swiglu_bwd(dh, y), swiglu_bwd_slack(dh, y), "dY1")
