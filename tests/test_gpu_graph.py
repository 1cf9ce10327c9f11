"""CUDA graph capture and replay of one grouped-linear step through the C ABI
(no call syncs or allocates once outputs are preallocated), including the
device noop flag: a replay with the flag set must leave every quantized
output untouched, a replay with it cleared must reproduce eager results
bit for bit."""
import numpy as np
import pytest
import torch

from synth import WORKLOADS, bf16_bits_from_f32, make_inputs
from tests._gpu import dev_bf16, dev_i64, lib, require_gpu

pytestmark = pytest.mark.gpu


def test_graph_capture_replay_with_noop():
    require_gpu()
    mxq = lib()
    w = WORKLOADS["e4_h512_n1024_t512"]
    d = make_inputs(w)
    E, N, K, M = w.E, w.N, w.K, w.M
    ms = dev_i64(d["m_splits"])
    x, wt, dy = dev_bf16(d["x"]), dev_bf16(d["w"]).view(E * N, K), dev_bf16(d["dy"])
    u8 = lambda n: torch.zeros(n, dtype=torch.uint8, device="cuda")
    qx = {"row_data": u8((M, K)), "row_scale": u8(mxq.scale_bytes(M, K, False)),
          "col_data": u8((M, K)), "col_scale": u8(mxq.scale_bytes(M, K, True))}
    qw = {"row_data": u8((E * N, K)), "row_scale": u8(mxq.scale_bytes(E * N, K, False)),
          "col_data": u8((E * N, K)), "col_scale": u8(mxq.scale_bytes(E * N, K, True))}
    qdy = {"row_data": u8((M, N)), "row_scale": u8(mxq.scale_bytes(M, N, False)),
           "col_data": u8((M, N)), "col_scale": u8(mxq.scale_bytes(M, N, True)), }
    dbias = torch.zeros((E, N), dtype=torch.float32, device="cuda")
    ws = u8(mxq.workspace_bytes(1, M, 0, N, E))
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.zeros((E, N, K), dtype=torch.float32, device="cuda")
    noop = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        mxq.group_quantize(x, ms, noop=noop, out=qx)
        mxq.group_quantize(wt, None, E=E, noop=noop, out=qw)
        qdy["dbias"] = dbias
        mxq.group_quantize(dy, ms, dbias=True, noop=noop, out=qdy, workspace=ws)
        mxq.grouped_gemm_fprop(qx["row_data"], qx["row_scale"], qw["row_data"].view(E, N, K), qw["row_scale"], ms,
                               out=y)
        mxq.grouped_gemm_dgrad(qdy["row_data"], qdy["row_scale"], qw["col_data"].view(E, N, K), qw["col_scale"],
                               ms, out=dx)
        mxq.grouped_gemm_wgrad(qdy["col_data"], qdy["col_scale"], qx["col_data"], qx["col_scale"], ms, out=dw)

    step()  # eager (also performs any first-call set-up before capture)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in [("y", y), ("dx", dx), ("dw", dw), ("db", dbias)]}
    eager_q = {k: v.clone() for k, v in {**{"x" + k: v for k, v in qx.items()},
                                          **{"w" + k: v for k, v in qw.items()}}.items()}

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)

    # replay with the noop flag set: quantized outputs untouched
    for t in list(qx.values()) + list(qw.values()):
        t.fill_(0x3C)
    noop.fill_(1)
    g.replay()
    torch.cuda.synchronize()
    assert all(bool((t == 0x3C).all()) for t in list(qx.values()) + list(qw.values()))

    # replay with the flag cleared: bit-identical to the eager step
    noop.zero_()
    y.zero_(); dx.zero_(); dw.zero_(); dbias.zero_()
    g.replay()
    torch.cuda.synchronize()
    for k, v in [("y", y), ("dx", dx), ("dw", dw), ("db", dbias)]:
        assert torch.equal(v, eager[k]), k
    for k, v in {**{"x" + k: v for k, v in qx.items()}, **{"w" + k: v for k, v in qw.items()}}.items():
        assert torch.equal(v, eager_q[k]), k


def test_graph_capture_of_the_fused_and_padded_entry_points():
    """The SwiGLU-fused FC1 fprop and FC2 dgrad, the scaled-bias requant and the padded-grouping
    quantize and fprop, captured in one graph and replayed: every output equals the eager one bit
    for bit (dbias and the routing-scale gradients included: their sums have a fixed order)."""
    require_gpu()
    mxq = lib()
    rng = np.random.default_rng(101)
    ms_a = np.array([128, 256, 0, 128], np.int64)
    ms_u = np.array([100, 3, 0, 409], np.int64)
    M, E, H, F = 512, 4, 256, 256
    bf = lambda *sh: dev_bf16(bf16_bits_from_f32((0.5 * rng.standard_normal(sh)).astype(np.float32)))
    x, w1, w2, dy2, b1, b2 = bf(M, H), bf(E, 2 * F, H), bf(E, H, F), bf(M, H), bf(E, 2 * F), bf(E, H)
    probs = torch.from_numpy(rng.random(M).astype(np.float32)).cuda()
    msa, msu = dev_i64(ms_a), dev_i64(ms_u)
    qx = mxq.group_quantize(x, msa)
    qw1 = mxq.group_quantize(w1.view(E * 2 * F, H), None, E=E, colwise=False)
    qw2 = mxq.group_quantize(w2.view(E * H, F), None, E=E, rowwise=False)
    wire = mxq.group_quantize(dy2, msa, rowwise=True, colwise=False, swizzle=False)
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device="cuda")
    ws = {"req": u8(mxq.workspace_bytes(mxq.mxq.OP_SCALED_BIAS, M, 0, H, E)),
          "bwd": u8(mxq.workspace_bytes(mxq.mxq.OP_GEMM_DGRAD_SWIGLU, M, H, F, E)),
          "pq": u8(mxq.workspace_bytes(mxq.mxq.OP_GROUP_QUANTIZE, M, 0, H, E, mxq.mxq.PAD_EXPERTS))}
    outs = {}

    def step():
        outs["fc1"] = mxq.grouped_gemm_fprop_swiglu(qx["row_data"], qx["row_scale"], qw1["row_data"].view(E, 2 * F, H),
                                                    qw1["row_scale"], msa, bias=b1, out=outs.get("fc1"))
        outs["req"] = mxq.requant_colwise_scaled_bias(wire["row_data"], wire["row_scale"], msa, probs, b2,
                                                      out=outs.get("req"), workspace=ws["req"])
        outs["bwd"] = mxq.grouped_gemm_dgrad_swiglu(wire["row_data"], outs["req"]["row_scale_swizzled"],
                                                    qw2["col_data"].view(E, H, F), qw2["col_scale"], outs["fc1"]["y1"],
                                                    msa, out=outs.get("bwd"), workspace=ws["bwd"])
        outs["pq"] = mxq.group_quantize(x, msu, dbias=True, pad_experts=True, out=outs.get("pq"), workspace=ws["pq"])
        outs["py"] = {"y": mxq.grouped_gemm_fprop(outs["pq"]["row_data"], outs["pq"]["row_scale"],
                                                  qw1["row_data"].view(E, 2 * F, H), qw1["row_scale"], msu,
                                                  pad_experts=True, out=(outs.get("py") or {}).get("y"))}

    def zero_all():
        for v in outs.values():
            for t in v.values():
                t.zero_()

    def snapshot():
        return {f"{k}.{kk}": t.clone() for k, v in outs.items() for kk, t in v.items()}

    step()  # allocates every output (and performs first-call set-up)
    zero_all()
    step()  # eager reference on zeroed outputs (scale-buffer tails past the used rows stay 0)
    torch.cuda.synchronize()
    eager = snapshot()
    zero_all()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    g.replay()
    torch.cuda.synchronize()
    got = snapshot()
    assert set(got) == set(eager)
    for k in eager:
        assert torch.equal(got[k], eager[k]), k
