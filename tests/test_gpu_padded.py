"""GPU parity: grouped quantization, requant and dbias with expert counts
that are not multiples of 128 (flag MXQ_PAD_EXPERTS: per-expert padded scale
layouts, after TransformerEngine PR #3244's review of the grouped swizzle),
against the oracle's padded grouping, through the C ABI. Codes and scales
bit-exact (scale buffers are compared over the padded row space the splits
actually use); dbias within 1e-5 * sum|x| per column."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import bf16_to_f64, dev_bf16, dev_i64, dev_u8, first_diff, host, lib, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


SPLITS = [
    [40, 3],                      # M = 43: partial blocks, M not a multiple of 128
    [128, 256, 0, 128],           # aligned (must equal the unflagged call)
    [200, 0, 57, 128, 1],         # empty and one-row experts
    [96, 160, 32, 224],           # multiples of 32, not of 128
    [0, 0, 300],
    [17] * 11,                    # many small experts inside one 128-row slice
]


def _x(M, K, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-4, 4, (M, 1)))).astype(np.float32)
    x[rng.random((M, K)) < 0.001] *= 1000.0
    return bf16_bits_from_f32(x)


def _cmp_scales(got, ref, what):
    ref = np.asarray(ref).reshape(-1)
    got = host(got).reshape(-1)[:ref.size]
    assert np.array_equal(got, ref), (what, first_diff(got, ref))


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("splits", SPLITS, ids=["_".join(map(str, s[:5])) for s in SPLITS])
def test_padded_group_quantize(mxq, splits, swz):
    ms = np.array(splits, np.int64)
    M, K = int(ms.sum()), 384
    x = _x(M, K, 81)
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), swizzle=swz, dbias=True, pad_experts=True)
    o = orc.group_quantize_padded(x, ms, swizzled=swz)
    assert np.array_equal(host(q["row_data"]), o["row_q"])
    assert np.array_equal(host(q["col_data"]), o["col_q"])
    if swz:
        _cmp_scales(q["row_scale"], o["row_s"], "row_s")
    else:  # dense compact rowwise scales: the rows the tensor has
        got = host(q["row_scale"]).reshape(o["row_s"].shape)[:M]
        assert np.array_equal(got, o["row_s"][:M])
    _cmp_scales(q["col_scale"], o["col_s"], "col_s")
    db = orc.grouped_dbias_padded(x, ms)
    a = np.abs(bf16_to_f64(x))
    off = np.concatenate([[0], np.cumsum(ms)])
    got = host(q["dbias"]).astype(np.float64)
    for e in range(len(ms)):
        tol = 1e-5 * a[off[e]:off[e + 1]].sum(axis=0) + 1e-30
        assert np.all(np.abs(got[e] - db[e]) <= tol), e


def test_padded_flag_with_aligned_splits_changes_nothing(mxq):
    ms = np.array([256, 0, 128, 384], np.int64)
    M, K = int(ms.sum()), 512
    x = dev_bf16(_x(M, K, 82))
    for swz in (True, False):
        a = mxq.group_quantize(x, dev_i64(ms), swizzle=swz, dbias=True)
        b = mxq.group_quantize(x, dev_i64(ms), swizzle=swz, dbias=True, pad_experts=True)
        for k in a:
            assert torch.equal(a[k], b[k].view(-1)[:a[k].numel()].view(a[k].shape)), (swz, k)


@pytest.mark.parametrize("swz", [True, False])
@pytest.mark.parametrize("splits", SPLITS[2:5], ids=["_".join(map(str, s[:5])) for s in SPLITS[2:5]])
def test_padded_requant(mxq, splits, swz):
    ms = np.array(splits, np.int64)
    M, K = int(ms.sum()), 256
    x = _x(M, K, 83)
    # the wire format: dense rowwise codes and dense compact scales (rowwise blocks ignore the grouping)
    wire = orc.group_quantize_padded(x, ms, rowwise=True, colwise=False, swizzled=False)
    r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), swizzle=swz, dbias=True,
                            dequant=True, pad_experts=True)
    o = orc.requant_colwise_padded(wire["row_q"], wire["row_s"], ms, swizzled=swz, dbias=True, dequant=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    _cmp_scales(r["col_scale"], o["col_s"], "col_s")
    _cmp_scales(r["row_scale_swizzled"], o["row_s_swizzled"], "row_s_swizzled")
    assert np.array_equal(host(r["dequant"]), o["deq"])
    deq = orc.dequant_rowwise(wire["row_q"], wire["row_s"])
    off = np.concatenate([[0], np.cumsum(ms)])
    got = host(r["dbias"]).astype(np.float64)
    for e in range(len(ms)):
        tol = 1e-5 * np.abs(deq[off[e]:off[e + 1]]).sum(axis=0) + 1e-30
        assert np.all(np.abs(got[e] - o["dbias"][e]) <= tol), e


def test_padded_status_bits(mxq):
    M, K = 300, 128
    x = dev_bf16(_x(M, K, 84))
    for bad, bit in (([100, -50, 250], 2), ([100, 150], 4)):
        status = mxq.new_status()
        out = {"row_data": torch.full((M, K), 7, dtype=torch.uint8, device="cuda")}
        mxq.group_quantize(x, dev_i64(bad), colwise=False, status=status, out=out, pad_experts=True)
        assert mxq.status_read(status) & bit
        assert torch.all(out["row_data"] == 7)
    status = mxq.new_status()
    mxq.group_quantize(x, dev_i64([100, 200]), status=status, pad_experts=True)
    assert mxq.status_read(status) == 0  # unaligned counts are valid with the flag


def test_full_size_padded_unaligned_routing(mxq):
    """The 64-expert workload's 83968 routed rows with counts NOT rounded to 128: seeded
    moves of rows between experts (sum kept), quantize with dbias and requant of the
    same rows as a wire format."""
    w = WORKLOADS["e64_h3072_f1024_t84k_prequant"]
    d = make_inputs(w, which=("dy2",))
    rng = np.random.default_rng([0, w.wid, 10])
    ms = d["m_splits"].copy()
    for _ in range(256):
        a, b = rng.integers(0, w.E, 2)
        mv = int(min(ms[a], rng.integers(1, 200)))
        ms[a] -= mv
        ms[b] += mv
    assert ms.sum() == w.M and np.any(ms % 128)
    x = d["dy2"]
    q = mxq.group_quantize(dev_bf16(x), dev_i64(ms), dbias=True, pad_experts=True)
    o = orc.group_quantize_padded(x, ms, swizzled=True)
    assert np.array_equal(host(q["row_data"]), o["row_q"])
    assert np.array_equal(host(q["col_data"]), o["col_q"])
    _cmp_scales(q["row_scale"], o["row_s"], "row_s")
    _cmp_scales(q["col_scale"], o["col_s"], "col_s")
    db = orc.grouped_dbias_padded(x, ms)
    a = np.abs(bf16_to_f64(x))
    off = np.concatenate([[0], np.cumsum(ms)])
    got = host(q["dbias"]).astype(np.float64)
    for e in range(w.E):
        assert np.all(np.abs(got[e] - db[e]) <= 1e-5 * a[off[e]:off[e + 1]].sum(axis=0) + 1e-30), e
    del q, o, a
    wire = orc.group_quantize_padded(x, ms, rowwise=True, colwise=False, swizzled=False)
    r = mxq.requant_colwise(dev_u8(wire["row_q"]), dev_u8(wire["row_s"]), dev_i64(ms), pad_experts=True)
    o = orc.requant_colwise_padded(wire["row_q"], wire["row_s"], ms, swizzled=True)
    assert np.array_equal(host(r["col_data"]), o["col_q"])
    _cmp_scales(r["col_scale"], o["col_s"], "col_s")
    _cmp_scales(r["row_scale_swizzled"], o["row_s_swizzled"], "row_s_swizzled")


# ------------------------------------------------ GEMMs on padded layouts
from tests._gpu import scaled_error  # noqa: E402

TOL_BF16, TOL_F32 = 8e-3, 1e-3


class PaddedOps:
    """Operands of one grouped linear with any expert counts: GPU inputs from the oracle's
    padded grouping (dense codes, padded swizzled scales); references from the aligned oracle
    applied to the zero-padded rows (pad rows add nothing to any product)."""

    def __init__(self, ms, N, K, seed):
        rng = np.random.default_rng(seed)
        self.ms = np.asarray(ms, np.int64)
        self.M, self.N, self.K, self.E = int(self.ms.sum()), N, K, len(ms)
        x = bf16_bits_from_f32(rng.standard_normal((self.M, K)).astype(np.float32))
        w = bf16_bits_from_f32((0.02 * rng.standard_normal((self.E, N, K))).astype(np.float32))
        dy = bf16_bits_from_f32(rng.standard_normal((self.M, N)).astype(np.float32))
        self.sx = orc.group_quantize_padded(x, self.ms, swizzled=True)
        self.sdy = orc.group_quantize_padded(dy, self.ms, swizzled=True)
        self.sw = orc.quantize_weights(w, swizzled=True)
        self.P, self.mp = orc.padded_offsets(self.ms)
        self.cx = orc.group_quantize(orc.pad_rows(x, self.ms), self.mp)
        self.cdy = orc.group_quantize(orc.pad_rows(dy, self.ms), self.mp)
        self.cw = orc.quantize_weights(w)
        off = np.concatenate([[0], np.cumsum(self.ms)])
        self.prow = np.concatenate([self.P[e] + np.arange(self.ms[e]) for e in range(self.E)]).astype(np.int64)
        assert self.prow.size == self.M and off[-1] == self.M

    def gpu(self, mxq):
        E, N, K = self.E, self.N, self.K
        ms = dev_i64(self.ms)
        y = mxq.grouped_gemm_fprop(dev_u8(self.sx["row_q"]), dev_u8(self.sx["row_s"]),
                                   dev_u8(self.sw["row_q"]).view(E, N, K), dev_u8(self.sw["row_s"]), ms,
                                   pad_experts=True)
        dx = mxq.grouped_gemm_dgrad(dev_u8(self.sdy["row_q"]), dev_u8(self.sdy["row_s"]),
                                    dev_u8(self.sw["col_q"]).view(E, N, K), dev_u8(self.sw["col_s"]), ms,
                                    pad_experts=True)
        dw = mxq.grouped_gemm_wgrad(dev_u8(self.sdy["col_q"]), dev_u8(self.sdy["col_s"]), dev_u8(self.sx["col_q"]),
                                    dev_u8(self.sx["col_s"]), ms, pad_experts=True)
        return y, dx, dw


def _f64(t):
    a = host(t)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _check_padded_gemms(mxq, op, rows=None, nk_samples=None):
    E, N, K = op.E, op.N, op.K
    y, dx, dw = op.gpu(mxq)
    rows = np.arange(op.M) if rows is None else rows
    r, c = np.meshgrid(rows, np.arange(N), indexing="ij")
    ref, mag = orc.fprop_entries(op.cx["row_q"], op.cx["row_s"], op.cw["row_q"].reshape(E, N, K), op.cw["row_s"],
                                 op.mp, op.prow[r.ravel()], c.ravel())
    assert scaled_error(_f64(y)[r.ravel(), c.ravel()], ref, mag) <= TOL_BF16
    r, c = np.meshgrid(rows, np.arange(K), indexing="ij")
    ref, mag = orc.dgrad_entries(op.cdy["row_q"], op.cdy["row_s"], op.cw["col_q"].reshape(E, N, K), op.cw["col_s"],
                                 op.mp, op.prow[r.ravel()], c.ravel())
    assert scaled_error(_f64(dx)[r.ravel(), c.ravel()], ref, mag) <= TOL_BF16
    if nk_samples is None:
        e, n, k = (a.ravel() for a in np.meshgrid(np.arange(E), np.arange(N), np.arange(K), indexing="ij"))
    else:
        rng = np.random.default_rng(91)
        e, n, k = rng.integers(0, E, nk_samples), rng.integers(0, N, nk_samples), rng.integers(0, K, nk_samples)
    ref, mag = orc.wgrad_entries(op.cdy["col_q"], op.cdy["col_s"], op.cx["col_q"], op.cx["col_s"], op.mp, e, n, k)
    assert scaled_error(_f64(dw)[e, n, k], ref, mag) <= TOL_F32
    dwh = host(dw)
    for ee in range(E):  # empty experts: dW = 0 exactly
        if op.ms[ee] == 0:
            assert np.all(dwh[ee] == 0)


@pytest.mark.parametrize("splits", [[40, 3, 0, 200, 57], [1, 127, 129, 0], [300]],
                         ids=["mixed", "edges", "one_expert"])
def test_padded_gemms_every_entry(mxq, splits):
    _check_padded_gemms(mxq, PaddedOps(splits, 256, 256, 92))


def test_padded_gemms_sampled(mxq):
    rng = np.random.default_rng(93)
    ms = rng.integers(0, 700, 12)
    ms[3] = 0
    op = PaddedOps(ms, 512, 768, 94)
    rows = np.unique(np.concatenate([np.cumsum(ms)[:-1], np.cumsum(ms) - 1, rng.integers(0, op.M, 200)]))
    rows = rows[(rows >= 0) & (rows < op.M)]
    _check_padded_gemms(mxq, op, rows=rows, nk_samples=20000)


def test_padded_gemms_with_aligned_splits_match_the_plain_calls(mxq):
    ms = [256, 0, 128, 384]
    op = PaddedOps(ms, 256, 512, 95)
    y, dx, dw = op.gpu(mxq)
    E, N, K = op.E, op.N, op.K
    d = dev_i64(np.asarray(ms, np.int64))
    y0 = mxq.grouped_gemm_fprop(dev_u8(op.sx["row_q"]), dev_u8(op.sx["row_s"]), dev_u8(op.sw["row_q"]).view(E, N, K),
                                dev_u8(op.sw["row_s"]), d)
    dx0 = mxq.grouped_gemm_dgrad(dev_u8(op.sdy["row_q"]), dev_u8(op.sdy["row_s"]),
                                 dev_u8(op.sw["col_q"]).view(E, N, K), dev_u8(op.sw["col_s"]), d)
    dw0 = mxq.grouped_gemm_wgrad(dev_u8(op.sdy["col_q"]), dev_u8(op.sdy["col_s"]), dev_u8(op.sx["col_q"]),
                                 dev_u8(op.sx["col_s"]), d)
    assert torch.equal(y, y0) and torch.equal(dx, dx0) and torch.equal(dw, dw0)


def test_padded_fprop_with_bias(mxq):
    """The bias on padded operands: full 32-row boxes leave through TMA stores, the rows of a box that
    reaches past its expert row by row; both add b_e in fp32 before the bf16 rounding."""
    ms = [40, 3, 0, 200, 57]
    op = PaddedOps(ms, 256, 256, 96)
    E, N, K = op.E, op.N, op.K
    bias = bf16_bits_from_f32((0.5 * np.random.default_rng(97).standard_normal((E, N))).astype(np.float32))
    y = mxq.grouped_gemm_fprop(dev_u8(op.sx["row_q"]), dev_u8(op.sx["row_s"]), dev_u8(op.sw["row_q"]).view(E, N, K),
                               dev_u8(op.sw["row_s"]), dev_i64(op.ms), bias=dev_bf16(bias), pad_experts=True)
    r, c = np.meshgrid(np.arange(op.M), np.arange(N), indexing="ij")
    ref, mag = orc.fprop_entries(op.cx["row_q"], op.cx["row_s"], op.cw["row_q"].reshape(E, N, K), op.cw["row_s"],
                                 op.mp, op.prow[r.ravel()], c.ravel(), bias=bias)
    assert scaled_error(_f64(y)[r.ravel(), c.ravel()], ref, mag) <= TOL_BF16


def test_padded_wgrad_bf16_out_and_accumulate(mxq):
    ms = [40, 3, 0, 200, 57]
    op = PaddedOps(ms, 256, 256, 98)
    E, N, K = op.E, op.N, op.K
    args = (dev_u8(op.sdy["col_q"]), dev_u8(op.sdy["col_s"]), dev_u8(op.sx["col_q"]), dev_u8(op.sx["col_s"]),
            dev_i64(op.ms))
    e, n, k = (a.ravel() for a in np.meshgrid(np.arange(E), np.arange(N), np.arange(K), indexing="ij"))
    ref, mag = orc.wgrad_entries(op.cdy["col_q"], op.cdy["col_s"], op.cx["col_q"], op.cx["col_s"], op.mp, e, n, k)
    dwb = mxq.grouped_gemm_wgrad(*args, out_bf16=True, pad_experts=True)
    assert scaled_error(_f64(dwb)[e, n, k], ref, mag) <= TOL_BF16
    prefill = np.random.default_rng(99).standard_normal((E, N, K)).astype(np.float32)
    acc = torch.from_numpy(prefill.copy()).cuda()
    mxq.grouped_gemm_wgrad(*args, accumulate=True, out=acc, pad_experts=True)
    got = host(acc).astype(np.float64) - prefill.astype(np.float64)
    # the fp32 read-modify-write adds one rounding of the sum's size on top of the product's tolerance
    tol = TOL_F32 * mag + 2.0 ** -23 * (np.abs(prefill.astype(np.float64))[e, n, k] + np.abs(ref))
    assert np.all(np.abs(got[e, n, k] - ref) <= tol + 1e-30)
    assert np.array_equal(host(acc)[2], prefill[2])  # the empty expert is left as it was
