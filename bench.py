"""Benchmark: one grouped MXFP8 linear training step of an MoE expert layer.

Headline workload: 128 experts (32 of them empty, the rest with Pareto(1.2)
loads rounded to 128-token multiples), hidden 7168, out 2048, 131072 routed
tokens, bf16 activations with x1000 outliers and all-zero 32x32 tiles. One
step is the whole hot path over one batch:

    group_quantize X (rowwise + colwise)      | group_quantize W (rowwise +
                                              | colwise, uniform members)
                                              [two streams, joined]
    grouped fprop  Y  = X W_e^T
    group_quantize dY (rowwise + colwise)
    grouped dgrad  dX = dY W_e
    grouped wgrad  dW = dY_e^T X_e (fp32)

(On a workload whose X arrives rowwise-quantized, as an expert-parallel FP8
dispatch delivers it, the first call is requant_colwise instead.)

value = GEMM flops of the step (6*M*N*K) / step time (whole step), in
TFLOP/s. L2 is flushed (256 MiB write) before every pass; the flush is outside
the per-pass CUDA-event brackets. The timed region runs K steps, each as R
back-to-back passes (R chosen so the region lasts over a second; ms_per_step
is one pass). Per-kernel times come from events on the stream that runs each
kernel; a serial pass of the same step times each quantize kernel alone. The
line also carries one grouped-linear step of every other synthetic workload
("configs"), the full SwiGLU MLP step on the 64-expert workload ("mlp_step"),
an end-to-end leg through pinned host buffers ("e2e") and the CPU oracle on a
bounded fraction of the step ("cpu_baseline"). `--impl reference` times the
CPU oracle alone.

Multi-GPU (torchrun): every rank runs an independent replica of the
workload (the grouped path has no exchange step of its own); rank 0 prints
the aggregate (weak scaling, max time over ranks).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "e128_h7168_n2048_t128k_skew"
TIMED_REGION_S = 1.2    # the timed region lasts at least this long (inner repeat of each step)
METRIC = "grouped MXFP8 GEMM TFLOPS (fprop+dgrad+wgrad); group_quantize HBM GB/s"
UNIT = "TFLOP/s"
MXFP8_OVER_BF16 = 2.0   # nominal dense MXFP8 / BF16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--repeat", type=int, default=0,
                   help="passes per timed step (0: enough for a timed region of at least TIMED_REGION_S)")
    p.add_argument("--no-configs", action="store_true", help="skip the other workloads' grouped-linear steps")
    p.add_argument("--workload", default=None,
                   help="run the timed step on this workload instead of the headline one (a small footprint for "
                        "profilers)")
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-mlp", action="store_true", help="skip the full-MLP step measurement")
    p.add_argument("--only", choices=["swiglu_quantize", "scaled_bias", "fused_mlp", "padded", "configs", "mma_peak",
                                      "mlp_e32"],
                   help="time only one fused kernel family on the MLP workload's shapes and print its line (a "
                        "small footprint for profilers): the SwiGLU->quantize kernels (forward and backward), "
                        "requant of the FC2 gradient with plain dbias vs with the scaled-bias reductions, the "
                        "SwiGLU-fused FC1 fprop and FC2 dgrad vs their unfused pairs, group_quantize with "
                        "expert counts that are not multiples of 128, one grouped-linear step on every "
                        "synthetic workload, the tensor-pipe ceiling probe (back-to-back block-scaled MMAs), or "
                        "the full SwiGLU MLP step (fwd+bwd) on the 32-expert bf16-input workload")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), d.get("hbm_gbs", FALLBACK_HBM_GBS), "measured"
    return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# --------------------------------------------------------------- workload
def make_host_workload(name=None):
    from synth import WORKLOADS, make_inputs

    w = WORKLOADS[name or WORKLOAD]
    d = make_inputs(w, which=("x", "w", "dy"))
    return w, d


def x_kernel(w) -> str:
    return "requant_x" if w.prequant_x else "quantize_x"


def workload_config(w, d, world):
    """The workload both arms run, as named in their JSON lines."""
    first = ("requant X (rowwise wire format -> colwise copy + swizzled rowwise scales)" if w.prequant_x
             else "quantize X (row+col)")
    return {"workload": w.name, "experts": w.E, "hidden": w.K, "out": w.N, "tokens": w.M,
            "m_splits": [int(v) for v in d["m_splits"]],
            "step": f"{first} + quantize W (row+col), fprop, quantize dY (row+col), dgrad, wgrad (fp32 dW)",
            "parallelism": f"replicas x{world}",
            "l2": "GPU arm: a 256 MiB buffer written before every timed pass (outside the event brackets)"}


class NativeStep:
    """Device-resident inputs/outputs of one step and the calls that run it.

    In the order of a training step: the forward's two quantizations, fprop,
    then the backward's (quantize dY) and dgrad, wgrad. The forward's two are
    independent, so by default they run concurrently: the quantization of X
    (or its requant, when X arrives rowwise-quantized) on a side stream forked
    from the caller's stream, quantize W on it, joined before fprop. Each
    kernel's last partial wave of CTAs leaves SMs idle that the other fills.
    The outputs are bit-identical to the serial order."""

    def __init__(self, w, d, dev):
        import torch

        import moe_expert_grouped_group_gb300 as mxq

        self.torch, self.mxq, self.w, self.dev = torch, mxq, w, dev
        self.pre_x = w.prequant_x
        E, N, K, M = w.E, w.N, w.K, w.M
        tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        self.ms = torch.from_numpy(d["m_splits"]).to(dev)
        self.x_bf16 = tb(d["x"])
        self.wt = tb(d["w"]).view(E * N, K)
        self.dy = tb(d["dy"])
        u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
        if self.pre_x:
            # The dispatch wire format (rowwise E4M3 + compact scales), made once
            # by the library itself (setup, untimed).
            q = mxq.group_quantize(self.x_bf16, self.ms, rowwise=True, colwise=False, swizzle=False)
            self.x_row, self.x_row_scale = q["row_data"], q["row_scale"]
            self.qx = {"col_data": u8((M, K)), "col_scale": u8(mxq.scale_bytes(M, K, True)),
                       "row_scale_swizzled": u8(mxq.scale_bytes(M, K, False))}
            self.e2e_inputs = ("x_row", "x_row_scale", "wt", "dy", "ms")
        else:
            self.qx = {"row_data": u8((M, K)), "row_scale": u8(mxq.scale_bytes(M, K, False)),
                       "col_data": u8((M, K)), "col_scale": u8(mxq.scale_bytes(M, K, True))}
            self.e2e_inputs = ("x_bf16", "wt", "dy", "ms")
        self.qw = {"row_data": u8((E * N, K)), "row_scale": u8(mxq.scale_bytes(E * N, K, False)),
                   "col_data": u8((E * N, K)), "col_scale": u8(mxq.scale_bytes(E * N, K, True))}
        self.qdy = {"row_data": u8((M, N)), "row_scale": u8(mxq.scale_bytes(M, N, False)),
                    "col_data": u8((M, N)), "col_scale": u8(mxq.scale_bytes(M, N, True))}
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((E, N, K), dtype=torch.float32, device=dev)
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.launches_per_step = 6
        self.kernel_events = kernel_events(self.pre_x)
        self.s_x = torch.cuda.Stream(device=dev)
        self.ev_fork, self.ev_x = torch.cuda.Event(), torch.cuda.Event()

    def x_operands(self):
        """(rowwise codes, swizzled rowwise scales, colwise codes, colwise scales) of X."""
        if self.pre_x:
            return self.x_row, self.qx["row_scale_swizzled"], self.qx["col_data"], self.qx["col_scale"]
        return self.qx["row_data"], self.qx["row_scale"], self.qx["col_data"], self.qx["col_scale"]

    def run(self, events=None, concurrent=True):
        """One step on the current stream. events: STEP_EVENTS timing events, recorded on the stream
        that runs each kernel (see kernel_events)."""
        torch, mxq, w = self.torch, self.mxq, self.w
        E, N, K = w.E, w.N, w.K
        main = torch.cuda.current_stream()
        rec = (lambda i, st=None: events[i].record(st or main)) if events else (lambda i, st=None: None)

        def quant_x():
            if self.pre_x:
                mxq.requant_colwise(self.x_row, self.x_row_scale, self.ms, out=self.qx)
            else:
                mxq.group_quantize(self.x_bf16, self.ms, out=self.qx)

        rec(0)
        if concurrent:
            self.ev_fork.record(main)
            self.s_x.wait_event(self.ev_fork)
            with torch.cuda.stream(self.s_x):
                rec(1, self.s_x)
                quant_x()
                rec(2, self.s_x)
            self.ev_x.record(self.s_x)
            rec(3)
            mxq.group_quantize(self.wt, None, E=E, out=self.qw)
            rec(4)
            main.wait_event(self.ev_x)
        else:
            rec(1)
            quant_x()
            rec(2)
            rec(3)
            mxq.group_quantize(self.wt, None, E=E, out=self.qw)
            rec(4)
        rec(5)
        x_row, x_rs, x_col, x_cs = self.x_operands()
        mxq.grouped_gemm_fprop(x_row, x_rs, self.qw["row_data"].view(E, N, K), self.qw["row_scale"], self.ms,
                               out=self.y)
        rec(6)
        mxq.group_quantize(self.dy, self.ms, out=self.qdy)
        rec(7)
        mxq.grouped_gemm_dgrad(self.qdy["row_data"], self.qdy["row_scale"], self.qw["col_data"].view(E, N, K),
                               self.qw["col_scale"], self.ms, out=self.dx)
        rec(8)
        mxq.grouped_gemm_wgrad(self.qdy["col_data"], self.qdy["col_scale"], x_col, x_cs, self.ms, out=self.dw)
        rec(9)

    def flush(self):
        self.flush_buf.fill_(1)


MLP_WORKLOAD = "e64_h3072_f1024_t84k_prequant"
MLP_WORKLOAD_E32 = "e32_h4096_f1536_t64k_swiglu"


class MLPStep:
    """Forward + backward of a grouped MoE MLP (FC1 -> SwiGLU -> FC2). On the 64-expert workload X
    and the FC2 gradient arrive rowwise-quantized (the expert-parallel dispatch and the combine's
    backward) and both linears carry per-expert biases; on the 32-expert workload X and the FC2
    gradient arrive in bf16 and there are no biases. Covers every step of the path: requant or
    quantize (+fused dbias), weight quantize, the three grouped GEMMs of both linears, SwiGLU.
    The forward's input quantizations run concurrently (X on a side stream, W1 and W2 on the
    caller's stream) and join before FC1; the rest runs in order on the caller's stream."""

    def __init__(self, dev, workload=MLP_WORKLOAD, seed=0):
        import torch

        import moe_expert_grouped_group_gb300 as mxq
        from synth import WORKLOADS, make_inputs

        self.torch, self.mxq = torch, mxq
        w = self.w = WORKLOADS[workload]
        self.pre_x, self.pre_dy, self.has_bias = w.prequant_x, w.prequant_dy, w.bias
        which = ("x", "w", "w2", "dy2") + (("b1", "b2") if w.bias else ())
        d = make_inputs(w, seed=seed, which=which)
        E, H, F, M = w.E, w.K, w.F, w.M
        self.E, self.H, self.F, self.M = E, H, F, M
        tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        self.ms = torch.from_numpy(d["m_splits"]).to(dev)
        self.w1 = tb(d["w"]).view(E * 2 * F, H)
        self.w2 = tb(d["w2"]).view(E * H, F)
        self.b1, self.b2 = (tb(d["b1"]), tb(d["b2"])) if w.bias else (None, None)
        u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
        bf = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=dev)
        sb = mxq.scale_bytes

        def q(rows, cols):
            return {"row_data": u8((rows, cols)), "row_scale": u8(sb(rows, cols, False)),
                    "col_data": u8((rows, cols)), "col_scale": u8(sb(rows, cols, True))}

        def rq(rows, cols):
            return {"col_data": u8((rows, cols)), "col_scale": u8(sb(rows, cols, True)),
                    "row_scale_swizzled": u8(sb(rows, cols, False))}

        if self.pre_x:  # the dispatch wire format, made once by the library itself (setup, untimed)
            qx = mxq.group_quantize(tb(d["x"]), self.ms, rowwise=True, colwise=False, swizzle=False)
            self.x_row, self.x_rs = qx["row_data"], qx["row_scale"]
            self.qx = rq(M, H)
        else:
            self.x_bf16 = tb(d["x"])
            self.qx = q(M, H)
        if self.pre_dy:
            qd = mxq.group_quantize(tb(d["dy2"]), self.ms, rowwise=True, colwise=False, swizzle=False)
            self.dy2_row, self.dy2_rs = qd["row_data"], qd["row_scale"]
            self.qd = rq(M, H)
        else:
            self.dy2_bf16 = tb(d["dy2"])
            self.qd = q(M, H)
        if w.bias:
            self.qd["dbias"] = torch.empty((E, H), dtype=torch.float32, device=dev)
        self.qw1, self.qw2 = q(E * 2 * F, H), q(E * H, F)
        self.qh = q(M, F)
        self.qdy1 = q(M, 2 * F)
        if w.bias:
            self.qdy1["dbias"] = torch.empty((E, 2 * F), dtype=torch.float32, device=dev)
        self.ws = u8(max(mxq.workspace_bytes(mxq.mxq.OP_REQUANT_COLWISE, M, 0, H, E),
                         mxq.workspace_bytes(mxq.mxq.OP_GROUP_QUANTIZE, M, 0, H, E),
                         mxq.workspace_bytes(mxq.mxq.OP_SWIGLU_BWD_QUANTIZE, M, 0, F, E)))
        self.y1, self.y2 = bf(M, 2 * F), bf(M, H)
        self.fc1_out = dict(self.qh, y1=self.y1)  # FC1 output saved bf16 + h quantized in its epilogue
        self.dh, self.dx = bf(M, F), bf(M, H)
        self.dw1 = torch.empty((E, 2 * F, H), dtype=torch.float32, device=dev)
        self.dw2 = torch.empty((E, H, F), dtype=torch.float32, device=dev)
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.launches_per_step = 11 + (1 if w.bias else 0) * 2
        self.s_x = torch.cuda.Stream(device=dev)
        self.ev_fork, self.ev_x = torch.cuda.Event(), torch.cuda.Event()
        b = "_dbias" if w.bias else ""
        # stage name -> (start, end) timing events of run(); event 5 is the forward quantize phase's join
        names = [("requant_x" if self.pre_x else "quantize_x"), "quantize_w1_w2", "fc1_fprop_swiglu_quantize_h",
                 "fc2_fprop", ("requant_dy2" if self.pre_dy else "quantize_dy2") + b, "fc2_dgrad", "fc2_wgrad",
                 "swiglu_bwd_quantize_dy1" + b, "fc1_dgrad", "fc1_wgrad"]
        self.stages = dict(zip(names, [(1, 2), (3, 4)] + [(k, k + 1) for k in range(5, 13)]))
        self.n_events = 14

    def flops(self):
        return 6.0 * self.M * (2 * self.F * self.H + self.H * self.F)

    def run(self, ev=None, concurrent=True):
        torch, mxq, E, H, F = self.torch, self.mxq, self.E, self.H, self.F
        main = torch.cuda.current_stream()
        rec = (lambda i, st=None: ev[i].record(st or main)) if ev else (lambda i, st=None: None)
        side = self.s_x if concurrent else main
        rec(0)
        if concurrent:
            self.ev_fork.record(main)
            side.wait_event(self.ev_fork)
        with torch.cuda.stream(side):
            rec(1, side)
            if self.pre_x:
                mxq.requant_colwise(self.x_row, self.x_rs, self.ms, out=self.qx)
                x_row, x_rs = self.x_row, self.qx["row_scale_swizzled"]
            else:
                mxq.group_quantize(self.x_bf16, self.ms, out=self.qx)
                x_row, x_rs = self.qx["row_data"], self.qx["row_scale"]
            rec(2, side)
        if concurrent:
            self.ev_x.record(side)
        rec(3)
        mxq.group_quantize(self.w1, None, E=E, out=self.qw1)
        mxq.group_quantize(self.w2, None, E=E, out=self.qw2)
        rec(4)
        if concurrent:
            main.wait_event(self.ev_x)
        rec(5)
        mxq.grouped_gemm_fprop_swiglu(x_row, x_rs, self.qw1["row_data"].view(E, 2 * F, H), self.qw1["row_scale"],
                                      self.ms, bias=self.b1, out=self.fc1_out)
        rec(6)
        mxq.grouped_gemm_fprop(self.qh["row_data"], self.qh["row_scale"], self.qw2["row_data"].view(E, H, F),
                               self.qw2["row_scale"], self.ms, bias=self.b2, out=self.y2)
        rec(7)
        if self.pre_dy:
            mxq.requant_colwise(self.dy2_row, self.dy2_rs, self.ms, dbias=self.has_bias, out=self.qd,
                                workspace=self.ws)
            dy2_row, dy2_rs = self.dy2_row, self.qd["row_scale_swizzled"]
        else:
            mxq.group_quantize(self.dy2_bf16, self.ms, dbias=self.has_bias, out=self.qd, workspace=self.ws)
            dy2_row, dy2_rs = self.qd["row_data"], self.qd["row_scale"]
        rec(8)
        mxq.grouped_gemm_dgrad(dy2_row, dy2_rs, self.qw2["col_data"].view(E, H, F), self.qw2["col_scale"], self.ms,
                               out=self.dh)
        rec(9)
        mxq.grouped_gemm_wgrad(self.qd["col_data"], self.qd["col_scale"], self.qh["col_data"], self.qh["col_scale"],
                               self.ms, out=self.dw2)
        rec(10)
        mxq.swiglu_bwd_quantize(self.dh, self.y1, self.ms, dbias=self.has_bias, out=self.qdy1, workspace=self.ws)
        rec(11)
        mxq.grouped_gemm_dgrad(self.qdy1["row_data"], self.qdy1["row_scale"], self.qw1["col_data"].view(E, 2 * F, H),
                               self.qw1["col_scale"], self.ms, out=self.dx)
        rec(12)
        mxq.grouped_gemm_wgrad(self.qdy1["col_data"], self.qdy1["col_scale"], self.qx["col_data"],
                               self.qx["col_scale"], self.ms, out=self.dw1)
        rec(13)

    def flush(self):
        self.flush_buf.fill_(1)


def time_mlp(dev, steps=10, warmup=3, workload=MLP_WORKLOAD):
    import torch

    st = MLPStep(dev, workload)
    for _ in range(warmup):
        st.flush()
        st.run()
    torch.cuda.synchronize()
    n = st.n_events
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n)] for _ in range(steps)]
    for i in range(steps):
        st.flush()
        st.run(evs[i])
    torch.cuda.synchronize()
    ms = statistics.mean(evs[i][0].elapsed_time(evs[i][n - 1]) for i in range(steps))
    per = {k: statistics.mean(evs[i][a].elapsed_time(evs[i][b]) for i in range(steps))
           for k, (a, b) in st.stages.items()}
    fwd_quant_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][5]) for i in range(steps))
    gemm_ms = sum(v for k, v in per.items() if "prop" in k or "grad" in k)
    bias = " (bias)" if st.has_bias else ""
    arrive = ("X and dY2 rowwise-prequantized" if st.pre_x and st.pre_dy else
              "X and dY2 in bf16, quantized rowwise+colwise inside the step")
    return {"workload": workload, "steps": steps, "warmup": warmup, "ms_per_step": ms,
            "tflops_step": st.flops() / (ms * 1e-3) / 1e12, "gemm_tflops": st.flops() / (gemm_ms * 1e-3) / 1e12,
            "stage_ms": per, "fwd_quantize_phase_ms": fwd_quant_ms, "gpu_launches": st.launches_per_step * steps,
            "step": f"fwd+bwd of FC1{bias} -> SwiGLU -> FC2{bias}, {arrive}; SwiGLU and the quantization of h in "
                    "FC1's GEMM epilogue (forward); SwiGLU backward fused with the quantization of dY1"
                    + (" and its dbias" if st.has_bias else "") + " (backward)",
            "l2": "a 256 MiB buffer written before every step",
            "streams": "the quantization of X on a side stream concurrent with that of W1 and W2 (stage_ms of the "
                       "two overlap); the rest in order after the join",
            "gemm_note": "gemm_tflops counts the FC1 stage whole (its epilogue also runs SwiGLU and quantizes h)"}


def swiglu_quant_bytes(M, F):
    """Algorithmic HBM bytes of the fused SwiGLU->quantize kernels (row+col
    E4M3 codes and E8M0 scales written once, inputs read once; backward adds
    the fp32 per-128-row dbias partials)."""
    fwd = M * 2 * F * 2 + M * F * (2 + 2 / 32)
    bwd = M * F * 2 + M * 2 * F * 2 + M * 2 * F * (2 + 2 / 32) + (M // 128) * 2 * F * 4
    return fwd, bwd


def time_swiglu_quantize(dev, steps, warmup):
    """The fused SwiGLU->quantize kernels alone on the MLP workload's shapes:
    y1 (M, 2F) and dh (M, F) bf16 ~N(0,1), forward with h's row+col codes,
    backward with dY1's row+col codes and its dbias."""
    import torch

    import moe_expert_grouped_group_gb300 as mxq
    from synth import WORKLOADS, bf16_normal, make_m_splits

    w = WORKLOADS[MLP_WORKLOAD]
    M, F, E = w.M, w.F, w.E
    tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    ms = torch.from_numpy(make_m_splits(w, 0)).to(dev)
    y1 = tb(bf16_normal((M, 2 * F), 1.0, (0, w.wid, 11)))
    dh = tb(bf16_normal((M, F), 1.0, (0, w.wid, 12)))
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
    sb = mxq.scale_bytes

    def q(rows, cols):
        return {"row_data": u8((rows, cols)), "row_scale": u8(sb(rows, cols, False)),
                "col_data": u8((rows, cols)), "col_scale": u8(sb(rows, cols, True))}

    qh, qdy1 = q(M, F), q(M, 2 * F)
    qdy1["dbias"] = torch.empty((E, 2 * F), dtype=torch.float32, device=dev)
    ws = u8(mxq.workspace_bytes(7, M, 0, F, E))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(warmup + steps):
        flush.fill_(1)
        e = ev[i - warmup] if i >= warmup else None
        if e:
            e[0].record()
        mxq.swiglu_quantize(y1, ms, out=qh)
        if e:
            e[1].record()
        mxq.swiglu_bwd_quantize(dh, y1, ms, dbias=True, out=qdy1, workspace=ws)
        if e:
            e[2].record()
    torch.cuda.synchronize()
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    fb, bb = swiglu_quant_bytes(M, F)
    return {"workload": MLP_WORKLOAD, "rows": M, "F": F, "steps": steps, "warmup": warmup,
            "fwd_us": fwd_ms * 1e3, "bwd_us": bwd_ms * 1e3,
            "fwd_gbs": fb / (fwd_ms * 1e-3) / 1e9, "bwd_gbs": bb / (bwd_ms * 1e-3) / 1e9,
            "fwd_bytes": fb, "bwd_bytes": bb,
            "l2": "256 MiB buffer written before every forward+backward pair"}


def time_scaled_bias(dev, steps, warmup):
    """Requant of the rowwise-quantized FC2 gradient (83968 x 3072, 64 experts):
    with the plain fused dbias, and with the scaled-bias reductions (dbias
    weighted by seeded routing scales, and each row's dot product with its
    expert's bias)."""
    import torch

    import moe_expert_grouped_group_gb300 as mxq
    from synth import WORKLOADS, make_inputs

    w = WORKLOADS[MLP_WORKLOAD]
    d = make_inputs(w, which=("dy2", "b2"))
    M, K, E = w.M, w.K, w.E
    tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    ms = torch.from_numpy(d["m_splits"]).to(dev)
    wire = mxq.group_quantize(tb(d["dy2"]), ms, rowwise=True, colwise=False, swizzle=False)
    probs = torch.from_numpy(np.random.default_rng([0, w.wid, 8]).random(M).astype(np.float32)).to(dev)
    b2 = tb(d["b2"])
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
    sb = mxq.scale_bytes
    out = {"col_data": u8((M, K)), "col_scale": u8(sb(M, K, True)), "row_scale_swizzled": u8(sb(M, K, False)),
           "dbias": torch.empty((E, K), dtype=torch.float32, device=dev),
           "dprobs": torch.empty((M,), dtype=torch.float32, device=dev)}
    ws = u8(mxq.workspace_bytes(mxq.mxq.OP_SCALED_BIAS, M, 0, K, E))
    plain_out = {k: v for k, v in out.items() if k != "dprobs"}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    runs = {
        "requant_dbias": lambda: mxq.requant_colwise(wire["row_data"], wire["row_scale"], ms, dbias=True,
                                                     out=plain_out, workspace=ws),
        "requant_scaled_bias": lambda: mxq.requant_colwise_scaled_bias(wire["row_data"], wire["row_scale"], ms,
                                                                       probs, b2, out=out, workspace=ws),
    }
    res = {"workload": MLP_WORKLOAD, "rows": M, "cols": K, "steps": steps, "warmup": warmup,
           "l2": "256 MiB buffer written before every launch"}
    base = M * K * (2 + 3 / 32)  # E4M3 in + colwise out + three scale sets
    nbytes = {"requant_dbias": base, "requant_scaled_bias": base + M * 4 + E * K * 2}
    for name, fn in runs.items():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(warmup + steps):
            flush.fill_(1)
            if i >= warmup:
                ev[i - warmup][0].record()
            fn()
            if i >= warmup:
                ev[i - warmup][1].record()
        torch.cuda.synchronize()
        us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
        res[name + "_us"] = us
        res[name + "_gbs"] = nbytes[name] / (us * 1e-6) / 1e9
    return res


def time_fused_mlp(dev, steps, warmup):
    """The two SwiGLU-fused GEMMs of the MLP workload (64 experts, 83968 rows,
    hidden 3072, F 1024) against their unfused pairs: FC1 fprop + SwiGLU and
    quantization of h, and FC2 dgrad + SwiGLU backward and quantization of dY1
    with its dbias. Operands are quantized on the device."""
    import torch

    import moe_expert_grouped_group_gb300 as mxq
    from synth import WORKLOADS, make_inputs

    w = WORKLOADS[MLP_WORKLOAD]
    d = make_inputs(w, which=("x", "w", "w2", "dy2", "b1"))
    E, H, F, M = w.E, w.K, w.F, w.M
    tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    ms = torch.from_numpy(d["m_splits"]).to(dev)
    qx = mxq.group_quantize(tb(d["x"]), ms, rowwise=True, colwise=False)
    qd = mxq.group_quantize(tb(d["dy2"]), ms, rowwise=True, colwise=False)
    qw1 = mxq.group_quantize(tb(d["w"]).view(E * 2 * F, H), None, E=E, colwise=False)
    qw2 = mxq.group_quantize(tb(d["w2"]).view(E * H, F), None, E=E, rowwise=False)
    del d
    b1 = tb(make_inputs(w, which=("b1",))["b1"])
    w1v, w2v = qw1["row_data"].view(E, 2 * F, H), qw2["col_data"].view(E, H, F)
    fc1_out = mxq.grouped_gemm_fprop_swiglu(qx["row_data"], qx["row_scale"], w1v, qw1["row_scale"], ms, bias=b1)
    y1 = fc1_out["y1"]
    ws = torch.empty(mxq.workspace_bytes(mxq.mxq.OP_GEMM_DGRAD_SWIGLU, M, H, F, E), dtype=torch.uint8, device=dev)
    dy1 = mxq.grouped_gemm_dgrad_swiglu(qd["row_data"], qd["row_scale"], w2v, qw2["col_scale"], y1, ms,
                                        workspace=ws)
    dh = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
    qh = {k: torch.empty_like(v) for k, v in fc1_out.items() if k != "y1"}
    qdy1 = {k: torch.empty_like(v) for k, v in dy1.items()}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    runs = {
        "fc1_fused": [lambda: mxq.grouped_gemm_fprop_swiglu(qx["row_data"], qx["row_scale"], w1v, qw1["row_scale"],
                                                            ms, bias=b1, out=fc1_out)],
        "fc1_unfused": [lambda: mxq.grouped_gemm_fprop(qx["row_data"], qx["row_scale"], w1v, qw1["row_scale"], ms,
                                                       bias=b1, out=y1),
                        lambda: mxq.swiglu_quantize(y1, ms, out=qh)],
        "fc2_dgrad_fused": [lambda: mxq.grouped_gemm_dgrad_swiglu(qd["row_data"], qd["row_scale"], w2v,
                                                                  qw2["col_scale"], y1, ms, out=dy1, workspace=ws)],
        "fc2_dgrad_unfused": [lambda: mxq.grouped_gemm_dgrad(qd["row_data"], qd["row_scale"], w2v, qw2["col_scale"],
                                                             ms, out=dh),
                              lambda: mxq.swiglu_bwd_quantize(dh, y1, ms, dbias=True, out=qdy1, workspace=ws)],
    }
    res = {"workload": MLP_WORKLOAD, "steps": steps, "warmup": warmup,
           "l2": "256 MiB buffer written before every launch sequence"}
    for name, fns in runs.items():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(warmup + steps):
            flush.fill_(1)
            if i >= warmup:
                ev[i - warmup][0].record()
            for fn in fns:
                fn()
            if i >= warmup:
                ev[i - warmup][1].record()
        torch.cuda.synchronize()
        res[name + "_us"] = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    fl = 2.0 * M * 2 * F * H  # one GEMM of either linear: 2 M (2F) H = 2 M H F * 2
    res["fc1_fused_tflops"] = fl / (res["fc1_fused_us"] * 1e-6) / 1e12
    res["fc2_dgrad_fused_tflops"] = (2.0 * M * H * F) / (res["fc2_dgrad_fused_us"] * 1e-6) / 1e12
    return res


def unaligned_splits(w, ms):
    """The workload's routed rows with counts NOT rounded to 128: seeded moves of rows
    between experts, the total kept."""
    rng = np.random.default_rng([0, w.wid, 10])
    ms = ms.copy()
    for _ in range(256):
        a, b = rng.integers(0, w.E, 2)
        mv = int(min(ms[a], rng.integers(1, 200)))
        ms[a] -= mv
        ms[b] += mv
    return ms


def time_padded(dev, steps, warmup):
    """group_quantize (row + col + dbias, swizzled) of the 83968 x 3072 FC2 gradient: aligned
    counts, aligned counts through the padded-grouping path, and unaligned counts."""
    import torch

    import moe_expert_grouped_group_gb300 as mxq
    from synth import WORKLOADS, make_inputs

    w = WORKLOADS[MLP_WORKLOAD]
    d = make_inputs(w, which=("dy2",))
    M, K, E = w.M, w.K, w.E
    x = torch.from_numpy(np.ascontiguousarray(d["dy2"]).view(np.int16)).to(dev).view(torch.bfloat16)
    ms_a = torch.from_numpy(d["m_splits"]).to(dev)
    ms_u = torch.from_numpy(unaligned_splits(w, d["m_splits"])).to(dev)
    outs = {k: mxq.group_quantize(x, ms_a, dbias=True, pad_experts=(k != "aligned"))
            for k in ("aligned", "aligned_padded_path", "unaligned")}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    runs = {"aligned": lambda: mxq.group_quantize(x, ms_a, dbias=True, out=outs["aligned"]),
            "aligned_padded_path": lambda: mxq.group_quantize(x, ms_a, dbias=True, pad_experts=True,
                                                              out=outs["aligned_padded_path"]),
            "unaligned": lambda: mxq.group_quantize(x, ms_u, dbias=True, pad_experts=True, out=outs["unaligned"])}
    res = {"workload": MLP_WORKLOAD, "rows": M, "cols": K, "steps": steps, "warmup": warmup,
           "unaligned_experts": int((unaligned_splits(w, d["m_splits"]) % 128 != 0).sum()),
           "l2": "256 MiB buffer written before every launch"}
    nbytes = M * K * (2 + 2 + 2 / 32)
    _, hbm, _ = peaks()
    for name, fn in runs.items():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(warmup + steps):
            flush.fill_(1)
            if i >= warmup:
                ev[i - warmup][0].record()
            fn()
            if i >= warmup:
                ev[i - warmup][1].record()
        torch.cuda.synchronize()
        us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
        res[name + "_us"] = us
        res[name + "_frac"] = nbytes / (us * 1e-6) / 1e9 / hbm
    return res


def time_configs(dev, steps, warmup, skip=()):
    """One grouped-linear step (the first linear: FC1 for the SwiGLU MLPs) on every synthetic
    workload but those in `skip`: X quantized row+col (or, prequantized, requantized colwise), W and
    dY quantized row+col, fprop, dgrad, wgrad (fp32 dW), each call timed alone (CUDA events, L2
    flushed before each step); per-kernel times, GEMM TFLOP/s and quantize GB/s with their
    roofline fractions."""
    import torch

    import moe_expert_grouped_group_gb300 as mxq
    from synth import WORKLOADS, make_inputs

    bf16_peak, hbm, _ = peaks()
    mx_peak = bf16_peak * MXFP8_OVER_BF16
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    out = {}
    for name, w in WORKLOADS.items():
        if name in skip:
            continue
        d = make_inputs(w, which=("x", "w", "dy"))
        E, N, K, M = w.E, w.N, w.K, w.M
        ms = torch.from_numpy(d["m_splits"]).to(dev)
        x, wt, dy = tb(d["x"]), tb(d["w"]).view(E * N, K), tb(d["dy"])
        del d
        if w.prequant_x:
            wire = mxq.group_quantize(x, ms, rowwise=True, colwise=False, swizzle=False)
            qx = mxq.requant_colwise(wire["row_data"], wire["row_scale"], ms)
            qx["row_data"], qx["row_scale"] = wire["row_data"], qx["row_scale_swizzled"]
        else:
            qx = mxq.group_quantize(x, ms)
        qw = mxq.group_quantize(wt, None, E=E)
        qd = mxq.group_quantize(dy, ms)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((E, N, K), dtype=torch.float32, device=dev)
        if w.prequant_x:
            xq = lambda: mxq.requant_colwise(wire["row_data"], wire["row_scale"], ms, out={
                "col_data": qx["col_data"], "col_scale": qx["col_scale"], "row_scale_swizzled": qx["row_scale"]})
        else:
            xq = lambda: mxq.group_quantize(x, ms, out=qx)
        calls = [(x_kernel(w), xq), ("quantize_w", lambda: mxq.group_quantize(wt, None, E=E, out=qw)),
                 ("quantize_dy", lambda: mxq.group_quantize(dy, ms, out=qd)),
                 ("fprop", lambda: mxq.grouped_gemm_fprop(qx["row_data"], qx["row_scale"], qw["row_data"].view(E, N, K),
                                                          qw["row_scale"], ms, out=y)),
                 ("dgrad", lambda: mxq.grouped_gemm_dgrad(qd["row_data"], qd["row_scale"], qw["col_data"].view(E, N, K),
                                                          qw["col_scale"], ms, out=dx)),
                 ("wgrad", lambda: mxq.grouped_gemm_wgrad(qd["col_data"], qd["col_scale"], qx["col_data"],
                                                          qx["col_scale"], ms, out=dw))]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(steps)]
        for i in range(warmup + steps):
            flush.fill_(1)
            for j, (_, fn) in enumerate(calls):
                if i >= warmup:
                    ev[i - warmup][j].record()
                fn()
            if i >= warmup:
                ev[i - warmup][len(calls)].record()
        torch.cuda.synchronize()
        us = {k: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) * 1e3 for j, (k, _) in enumerate(calls)}
        wev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(steps):  # the three quantize calls again, no L2 flush in between
            for j in range(3):
                wev[i][j].record()
                calls[j][1]()
            wev[i][3].record()
        torch.cuda.synchronize()
        us_warm = {calls[j][0]: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in wev) * 1e3 for j in range(3)}
        out[name] = config_record(w, ms.cpu().numpy(), us, us_warm, mx_peak, hbm)
        del x, wt, dy, qx, qw, qd, y, dx, dw
        if w.prequant_x:
            del wire
        torch.cuda.empty_cache()
    return {"steps": steps, "warmup": warmup, "l2": "256 MiB buffer written before every step",
            "peak_tflops": mx_peak, "peak_gbs": hbm, "configs": out}


# NativeStep.run's timing events: 0 step start, (1, 2) quantize or requant X, (3, 4) quantize W, 5 forward
# quantize phase joined = fprop start, 6 fprop end, 7 quantize dY end, 8 dgrad end, 9 wgrad end (= step end)
STEP_EVENTS = 10


def kernel_events(pre_x: bool) -> dict:
    return {("requant_x" if pre_x else "quantize_x"): (1, 2), "quantize_w": (3, 4), "fprop": (5, 6),
            "quantize_dy": (6, 7), "dgrad": (7, 8), "wgrad": (8, 9)}


def step_event_times(evs, kev):
    """Mean ms per kernel (kev: kernel -> (start, end) event), of the forward quantize phase (X with
    quantize W) and of the step, over a list of STEP_EVENTS-event steps."""
    per = {k: statistics.mean(e[a].elapsed_time(e[b]) for e in evs) for k, (a, b) in kev.items()}
    per_step = [e[0].elapsed_time(e[STEP_EVENTS - 1]) for e in evs]
    phase = statistics.mean(e[0].elapsed_time(e[5]) for e in evs)
    return per, per_step, phase


def algorithmic(w):
    M, N, K, E = w.M, w.N, w.K, w.E
    flops = {"fprop": 2.0 * M * N * K, "dgrad": 2.0 * M * N * K, "wgrad": 2.0 * M * N * K}
    bytes_ = {x_kernel(w): (2.09375 if w.prequant_x else 4.0625) * M * K, "quantize_w": 4.0625 * E * N * K,
              "quantize_dy": 4.0625 * M * N}
    return flops, bytes_


def time_mma_stream(mmas_per_sm=8192, reps=5, random=False, warm=2):
    """TFLOP/s of the tensor-pipe ceiling probe (back-to-back block-scaled 128x256x32 MMAs on
    every SM from resident shared memory): the most the grouped GEMMs' instructions can reach.
    With zero operands and short launches it is the burst ceiling at the maximum clock; with
    random operands and about a second of launches (after `warm` untimed ones) the power limit
    holds the clock down, as it does for a GEMM on real data."""
    import torch

    import moe_expert_grouped_group_gb300 as mxq

    status = mxq.new_status()
    for _ in range(warm):
        mxq.probe_mma_stream(mmas_per_sm, status=status, random=random)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    flops = sum(mxq.probe_mma_stream(mmas_per_sm, status=status, random=random) for _ in range(reps))
    b.record()
    torch.cuda.synchronize()
    assert mxq.status_read(status) == 0, "the ceiling probe's wait timed out"
    return flops / (a.elapsed_time(b) * 1e-3) / 1e12


def gemm_bound_us(m_splits, N, K, mx_peak_tflops, hbm_gbs):
    """Per-expert roofline of the three grouped GEMMs: sum over experts of
    max(flops_e / tensor peak, bytes_e / HBM bandwidth), bytes_e being the
    algorithmic operand and output bytes of expert e (E4M3 codes + E8M0 scales
    in, bf16 Y / dX and fp32 dW out; an empty expert still writes its dW
    zeros). Equal to the dense bound when every expert is compute-bound."""
    q = 1 + 1 / 32  # one E4M3 byte + its share of an E8M0 scale
    tot = {"fprop": 0.0, "dgrad": 0.0, "wgrad": 0.0}
    for m in (int(v) for v in m_splits):
        f = 2.0 * m * N * K / (mx_peak_tflops * 1e12)
        b = {"fprop": m * K * q + N * K * q + m * N * 2, "dgrad": m * N * q + N * K * q + m * K * 2,
             "wgrad": m * N * q + m * K * q + N * K * 4}
        for k in tot:
            if m == 0 and k != "wgrad":
                continue
            tot[k] += max(f, b[k] / (hbm_gbs * 1e9))
    return {k: v * 1e6 for k, v in tot.items()}


def time_warm(st, steps):
    """Per-kernel times of the step with no L2 flush between steps (inputs
    that fit in the 129 MB L2 may then be served from it); kernels in order
    on one stream."""
    torch = st.torch
    for _ in range(3):
        st.run(concurrent=False)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(STEP_EVENTS)] for _ in range(steps)]
    for i in range(steps):
        st.run(evs[i], concurrent=False)
    torch.cuda.synchronize()
    return step_event_times(evs, st.kernel_events)[0]


def time_serial(st, steps):
    """The step with its kernels in order on one stream, L2 flushed before
    each step: every kernel timed alone (the quantize kernels' own HBM
    rates) and the serial step time."""
    torch = st.torch
    for _ in range(3):
        st.flush()
        st.run(concurrent=False)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(STEP_EVENTS)] for _ in range(steps)]
    for i in range(steps):
        st.flush()
        st.run(evs[i], concurrent=False)
    torch.cuda.synchronize()
    per, per_step, _ = step_event_times(evs, st.kernel_events)
    return per, statistics.mean(per_step)


def inner_repeat(st, steps, requested):
    """Passes per timed step: `requested` if > 0, else enough for a timed region of TIMED_REGION_S."""
    if requested > 0:
        return requested
    torch = st.torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        st.flush()
        st.run()
    b.record()
    torch.cuda.synchronize()
    pass_s = a.elapsed_time(b) * 1e-3 / 3
    return max(1, int(np.ceil(TIMED_REGION_S / (max(1, steps) * pass_s))))


def time_native(st, steps, warmup, sampler, repeat_requested):
    """K steps of R passes each (R = inner_repeat after the warm-up); every pass is one step of the hot
    path over the batch, preceded by its L2 flush (outside its event brackets)."""
    torch = st.torch
    for _ in range(warmup):
        st.flush()
        st.run()
    torch.cuda.synchronize()
    repeat = inner_repeat(st, steps, repeat_requested)
    n = steps * repeat
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(STEP_EVENTS)] for _ in range(n)]
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n):
        st.flush()
        st.run(evs[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    clocks = sampler.stop() if sampler else None
    per_kernel, per_step, phase = step_event_times(evs, st.kernel_events)
    return per_step, per_kernel, phase, wall, clocks, repeat


def time_e2e(st, steps, warmup, d):
    """Through the public API from pinned host memory: every step copies its
    inputs (X -- bf16, or the wire format and its scales --, W, dY, m_splits)
    host -> device, runs the six calls and copies its results (Y, dX, dW)
    device -> host.

    Pipelined: the copies run on their own streams, so step i+1's inputs go
    up and step i-1's results come down while step i's kernels run; inputs
    and outputs are double-buffered (two slots), the quantized intermediates
    are shared (the kernels of consecutive steps are ordered on one stream).
    Also returns the per-step time of the same work issued serially on one
    stream."""
    import copy

    torch = st.torch
    names_in, names_out = st.e2e_inputs, ("y", "dx", "dw")
    host_in = {k: getattr(st, k).cpu().pin_memory() for k in names_in}
    host_out = {k: torch.empty_like(getattr(st, k), device="cpu").pin_memory() for k in names_out}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    st2 = copy.copy(st)
    for k in names_in + names_out:
        setattr(st2, k, torch.empty_like(getattr(st, k)))
    slots = [st, st2]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in slots]    # the slot's inputs have landed
    ev_used = [torch.cuda.Event() for _ in slots]  # the slot's step has run
    ev_out = [torch.cuda.Event() for _ in slots]   # the slot's results are on the host

    def serial():
        for k in names_in:
            getattr(st, k).copy_(host_in[k], non_blocking=True)
        st.run()
        for k in names_out:
            host_out[k].copy_(getattr(st, k), non_blocking=True)

    def pipelined(i):
        j = i % 2
        s = slots[j]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_used[j])  # step i-2 has finished reading this slot's inputs
            for k in names_in:
                getattr(s, k).copy_(host_in[k], non_blocking=True)
            ev_in[j].record(s_in)
        comp.wait_event(ev_in[j])
        comp.wait_event(ev_out[j])  # step i-2's results have left this slot
        s.run()
        ev_used[j].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_used[j])
            for k in names_out:
                host_out[k].copy_(getattr(s, k), non_blocking=True)
            ev_out[j].record(s_out)

    def timed(body):
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        s_in.wait_stream(comp)
        for i in range(steps):
            body(i)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)
        b.record(comp)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    for _ in range(warmup):
        serial()
    ms_serial = timed(lambda i: serial())
    for i in range(warmup):
        pipelined(i)
    ms_pipe = timed(pipelined)
    return ms_pipe, ms_serial, h2d, d2h


def config_record(w, ms, us, us_warm, mx_peak, hbm):
    """One workload's row of the five-workload table: per-kernel times (us), GEMM TFLOP/s and quantize GB/s
    with their roofline fractions."""
    E, N, K, M = w.E, w.N, w.K, w.M
    bound = gemm_bound_us(ms, N, K, mx_peak, hbm)
    flops = 6.0 * M * N * K
    gemm_us = us["fprop"] + us["dgrad"] + us["wgrad"]
    _, qb = algorithmic(w)
    return {"us": {k: round(v, 1) for k, v in us.items()},
            "gemm_tflops": flops / (gemm_us * 1e-6) / 1e12,
            "gemm_frac": flops / (gemm_us * 1e-6) / 1e12 / mx_peak,
            "gemm_per_expert_bound_us": {k: round(v, 1) for k, v in bound.items()},
            "gemm_frac_of_per_expert_bound": sum(bound.values()) / gemm_us,
            "us_no_l2_flush": {k: round(v, 1) for k, v in us_warm.items()},
            "quant_gbs": {k: qb[k] / (us[k] * 1e-6) / 1e9 for k in qb},
            "quant_frac": {k: qb[k] / (us[k] * 1e-6) / 1e9 / hbm for k in qb},
            "x_path": "requant" if w.prequant_x else "quantize"}


# ------------------------------------------------------------- CPU oracle
class OracleSample:
    """The CPU oracle on a bounded fraction f of one step's GEMM work.

    The GEMMs: f*M*N fprop entries (full-length dot products over K), f*M*K
    dgrad entries (over N) and f*M*N*K/r wgrad entries, each reducing over r
    sampled tokens -- f of each GEMM's 2*M*N*K flops. The quantizations run on
    r rows of X and dY and on f of W's rows, rounded up to whole 128-row
    blocks (at least f of that work). The r sampled rows are treated as one
    expert's (so only one expert's weights are needed); the cost per entry does
    not depend on which expert it is. f * step flops / its measured time is
    therefore a lower bound of the oracle's rate in the step's metric."""

    def __init__(self, w, d, frac):
        import oracle as orc

        self.orc, self.w, self.d = orc, w, d
        M, N, K, E = w.M, w.N, w.K, w.E
        self.frac = frac
        self.rows = max(128, int(round(M * frac / 128)) * 128)
        self.wrows = max(128, int(round(E * N * frac / 128)) * 128)
        rows = self.rows
        self.wire = orc.group_quantize(d["x"][:rows], [rows], rowwise=True, colwise=False)
        self.cx = orc.group_quantize(d["x"][:rows], [rows])
        self.cdy = orc.group_quantize(d["dy"][:rows], [rows])
        self.cw = orc.quantize_weights(d["w"][:1])
        rng = np.random.default_rng(0)
        self.nf, self.nd = int(round(frac * M * N)), int(round(frac * M * K))
        self.nw = int(round(frac * M * N * K / rows))
        self.fr, self.fc = rng.integers(0, rows, self.nf), rng.integers(0, N, self.nf)
        self.dr, self.dc = rng.integers(0, rows, self.nd), rng.integers(0, K, self.nd)
        self.wn, self.wk = rng.integers(0, N, self.nw), rng.integers(0, K, self.nw)
        self.cores = orc.num_threads()
        first = "requant" if w.prequant_x else "quantize"
        self.sample = (f"f = {frac:.3g} of one step's GEMM work: {self.nf} fprop and {self.nd} dgrad entries "
                       f"(full-length dot products), {self.nw} wgrad entries over {rows} tokens; {first} X and "
                       f"quantize dY on {rows} rows, quantize W on {self.wrows}/{E * N} rows")

    def run(self):
        """Seconds per part of the sampled step."""
        orc, w, d = self.orc, self.w, self.d
        N, K = w.N, w.K
        rows, t = self.rows, {}
        t1 = time.perf_counter()
        if w.prequant_x:
            orc.requant_colwise(self.wire["row_q"], self.wire["row_s"], [rows], swizzled=True)
        else:
            orc.group_quantize(d["x"][:rows], [rows], swizzled=True)
        t[x_kernel(w)] = time.perf_counter() - t1
        t1 = time.perf_counter()
        orc.group_quantize(d["w"].reshape(-1, K)[:self.wrows], [self.wrows], swizzled=True)
        t["quantize_w"] = time.perf_counter() - t1
        t1 = time.perf_counter()
        orc.group_quantize(d["dy"][:rows], [rows], swizzled=True)
        t["quantize_dy"] = time.perf_counter() - t1
        cx, cdy, cw = self.cx, self.cdy, self.cw
        t1 = time.perf_counter()
        orc.fprop_entries(cx["row_q"], cx["row_s"], cw["row_q"].reshape(1, N, K), cw["row_s"], [rows],
                          self.fr, self.fc)
        t["fprop"] = time.perf_counter() - t1
        t1 = time.perf_counter()
        orc.dgrad_entries(cdy["row_q"], cdy["row_s"], cw["col_q"].reshape(1, N, K), cw["col_s"], [rows],
                          self.dr, self.dc)
        t["dgrad"] = time.perf_counter() - t1
        t1 = time.perf_counter()
        orc.wgrad_entries(cdy["col_q"], cdy["col_s"], cx["col_q"], cx["col_s"], [rows],
                          np.zeros(self.nw, np.int64), self.wn, self.wk)
        t["wgrad"] = time.perf_counter() - t1
        return t


# --------------------------------------------------------------- dist
_PG = None


def barrier():
    if _PG is not None:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float) -> float:
    if _PG is None:
        return v
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, world: int, t_max_s: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return per_rank_units * world / t_max_s


REFERENCE_FRAC = 1 / 8192   # fraction of a step's GEMM work the reference arm's oracle runs per timed step
CPU_BASELINE_FRAC = 1 / 2048  # fraction in the GPU line's cpu_baseline (10-30 s of CPU work)


def reference_arm(args, rank, world):
    """The CPU oracle as the reference implementation: each timed step is the oracle on a fixed
    fraction f of the workload's step; value = f * step flops / measured step time."""
    if rank != 0:
        return
    w, d = make_host_workload()
    flops, _ = algorithmic(w)
    step_flops = sum(flops.values())
    sample = OracleSample(w, d, REFERENCE_FRAC)
    for _ in range(args.warmup):
        sample.run()
    t0 = time.perf_counter()
    times = [sum(sample.run().values()) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    ms = statistics.mean(times) * 1e3
    value = sample.frac * step_flops / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(w, d, world),
            "step_fraction": sample.frac,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": sample.cores, "kind": "oracle",
                             "sample": sample.sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s_timed_region": wall}
    print(json.dumps(line), flush=True)


def main():
    global _PG
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        _PG = dist.group.WORLD
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    from __graft_entry__ import build

    build()
    if args.only == "swiglu_quantize":
        r = time_swiglu_quantize(dev, max(1, args.steps), max(1, args.warmup))
        _, hbm_peak, src = peaks()
        r.update(fwd_frac=r["fwd_gbs"] / hbm_peak, bwd_frac=r["bwd_gbs"] / hbm_peak, hbm_peak_gbs=hbm_peak,
                 peak_source=src)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    if args.only == "configs":
        r = time_configs(dev, max(1, args.steps), max(1, args.warmup))
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    if args.only == "padded":
        r = time_padded(dev, max(1, args.steps), max(1, args.warmup))
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    if args.only == "mma_peak":
        bf16_peak, _, src = peaks()
        t = time_mma_stream()
        sampler = ClockSampler(0)
        sampler.start()
        rnd = time_mma_stream(mmas_per_sm=1 << 22, reps=3, random=True, warm=2)
        rclk = sampler.stop()
        r = {"metric": "block-scaled MXFP8 tcgen05 MMA stream (128x256x32, one CTA per SM, resident operands)",
             "tflops": t, "unit": "TFLOP/s", "roofline_peak": bf16_peak * MXFP8_OVER_BF16,
             "ratio_to_roofline_peak": t / (bf16_peak * MXFP8_OVER_BF16), "peak_source": src,
             "operands": "zeros, 5 launches of 8192 MMAs per SM",
             "random_sustained_tflops": rnd,
             "random_sustained": "pseudo-random E4M3 operands, unit scales; 2 untimed then 3 timed launches of "
                                 "4194304 MMAs per SM (about a second)",
             "random_sustained_clocks": rclk}
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    if args.only == "mlp_e32":
        r = time_mlp(dev, max(1, args.steps), max(1, args.warmup), MLP_WORKLOAD_E32)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    if args.only == "fused_mlp":
        r = time_fused_mlp(dev, max(1, args.steps), max(1, args.warmup))
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    if args.only == "scaled_bias":
        r = time_scaled_bias(dev, max(1, args.steps), max(1, args.warmup))
        _, hbm_peak, src = peaks()
        r.update({k.replace("_gbs", "_frac"): v / hbm_peak for k, v in list(r.items()) if k.endswith("_gbs")})
        r.update(hbm_peak_gbs=hbm_peak, peak_source=src)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    bf16_peak, hbm_peak, src = peaks()
    mx_peak = bf16_peak * MXFP8_OVER_BF16
    w, d = make_host_workload(args.workload)
    st = NativeStep(w, d, dev)
    flops, bytes_ = algorithmic(w)
    step_flops = sum(flops.values())
    warmup = max(3, args.warmup)

    sampler = ClockSampler(local if world > 1 else 0) if rank == 0 else None
    per_step, per_kernel, phase_ms, wall, clocks, repeat = time_native(st, args.steps, warmup, sampler, args.repeat)
    ms_step = statistics.mean(per_step)
    ms_step_max = max_over_ranks(ms_step)
    value = aggregate(step_flops, world, ms_step_max * 1e-3) / 1e12

    gemm_ms = per_kernel["fprop"] + per_kernel["dgrad"] + per_kernel["wgrad"]
    gemm_tflops = step_flops / (gemm_ms * 1e-3) / 1e12
    serial_kernels, serial_ms = time_serial(st, max(10, args.steps // 2))
    quant_gbs = {k: bytes_[k] / (serial_kernels[k] * 1e-3) / 1e9 for k in bytes_}
    xk = x_kernel(w)
    phase_gbs = (bytes_[xk] + bytes_["quantize_w"]) / (phase_ms * 1e-3) / 1e9
    warm = time_warm(st, max(5, args.steps // 5))
    headline_record = config_record(w, d["m_splits"], {k: v * 1e3 for k, v in serial_kernels.items()},
                                    {k: warm[k] * 1e3 for k in bytes_}, mx_peak, hbm_peak)

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(10, args.steps // 2)
        ms_e2e, ms_serial, h2d, d2h = time_e2e(st, e2e_steps, max(3, args.warmup), d)
        ms_e2e, ms_serial = max_over_ranks(ms_e2e), max_over_ranks(ms_serial)
        e2e = {"value": aggregate(step_flops, world, ms_e2e * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "steps": e2e_steps,
               "issue": "copies on their own streams, overlapping the neighbouring steps' kernels; inputs and "
                        "outputs double-buffered",
               "serial_ms_per_step": ms_serial,
               "serial_value": aggregate(step_flops, world, ms_serial * 1e-3) / 1e12}
    del st
    torch.cuda.empty_cache()

    roofline = {"bound": "tensor", "achieved": gemm_tflops, "peak": mx_peak, "unit": "TFLOP/s",
                "frac": gemm_tflops / mx_peak, "traffic": None,
                "kernel": "grouped_gemm_kernel (fprop+dgrad+wgrad launches of one step)",
                "peak_source": f"{src} bf16 burst {bf16_peak} TFLOP/s x {MXFP8_OVER_BF16} (nominal MXFP8/BF16)"}
    sustained = None
    ppath = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(ppath):
        with open(ppath) as f:
            sustained = json.load(f).get("bf16_tflops_sustained")
    if sustained:
        # the GEMM launches are timed inside the step loop (about a second of back-to-back steps),
        # where the board's power limit holds the SM clock below its maximum: the sustained figure
        # is their peak, the burst one (a kernel timed alone) is kept beside it
        roofline["peak_burst"], roofline["frac_of_burst"] = mx_peak, gemm_tflops / mx_peak
        roofline["peak"] = sustained * MXFP8_OVER_BF16
        roofline["frac"] = gemm_tflops / roofline["peak"]
        roofline["peak_source"] = (f"{src} bf16 sustained {sustained} TFLOP/s x {MXFP8_OVER_BF16} (nominal "
                                   f"MXFP8/BF16): the GEMMs are timed inside a step loop of "
                                   f"{wall:.2f} s under the power limit")
    tpath = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if os.path.exists(tpath):
        from moe_expert_grouped_group_gb300.build import source_stamp

        with open(tpath) as f:
            tj = json.load(f)
        if tj.get("source_stamp") == source_stamp() and tj.get("workload") == w.name:
            roofline["traffic"] = tj.get("dram_bytes_per_step")
            roofline["traffic_per_launch"] = tj.get("dram_bytes_per_launch")
            roofline["traffic_note"] = tj.get("note")
    if rank == 0:
        try:
            stream_tflops = time_mma_stream()
            roofline["mma_stream_tflops"] = stream_tflops
            roofline["frac_of_mma_stream"] = gemm_tflops / stream_tflops
            # random operands for about a second: the ceiling under the power limit
            rnd = time_mma_stream(mmas_per_sm=1 << 22, reps=3, random=True, warm=2)
            roofline["mma_stream_random_sustained_tflops"] = rnd
            roofline["frac_of_mma_stream_random_sustained"] = gemm_tflops / rnd
        except Exception as ex:  # noqa: BLE001
            roofline["mma_stream_tflops"] = {"error": f"{type(ex).__name__}: {ex}"}
    bound = gemm_bound_us(d["m_splits"], w.N, w.K, mx_peak, hbm_peak)
    roofline["per_expert_bound_us"] = bound
    roofline["frac_of_per_expert_bound"] = sum(bound.values()) / (gemm_ms * 1e3)

    configs = None
    mlp = None
    if rank == 0:
        # secondary legs: a failure is reported in the line instead of losing the line
        if not args.no_configs:
            try:
                configs = time_configs(dev, min(10, max(1, args.steps)), 2, skip=(w.name,))
                configs["configs"][w.name] = dict(headline_record, note="from the headline run's serial pass")
            except Exception as ex:  # noqa: BLE001
                configs = {"error": f"{type(ex).__name__}: {ex}"}
            torch.cuda.empty_cache()
        if not args.no_mlp:
            try:
                mlp = time_mlp(dev)
            except Exception as ex:  # noqa: BLE001
                mlp = {"error": f"{type(ex).__name__}: {ex}"}
            torch.cuda.empty_cache()
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        t0 = time.perf_counter()
        try:
            sample = OracleSample(w, d, CPU_BASELINE_FRAC)
            t = sample.run()
            cpu_s = sum(t.values())
            cpu = {"value": sample.frac * step_flops / cpu_s / 1e12, "unit": UNIT, "cores": sample.cores,
                   "kind": "oracle", "sample": sample.sample, "step_fraction": sample.frac,
                   "sample_s": cpu_s, "per_part_s": t, "wall_s": time.perf_counter() - t0}
        except Exception as ex:  # noqa: BLE001
            cpu = {"error": f"{type(ex).__name__}: {ex}", "kind": "oracle"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": ms_step_max, "ms_per_step_median": statistics.median(per_step),
        "inner_repeat": repeat, "timed_passes": args.steps * repeat,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8_e4m3 (fp32 accumulate)", "data": "synthetic",
        "config": workload_config(w, d, world),
        "streams": "the quantization of X on a side stream concurrent with quantize W; the rest in order after "
                   "the join",
        "timing": f"{args.steps} timed steps of {repeat} back-to-back passes each; ms_per_step is the mean pass",
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 6 * args.steps * repeat,
        "clocks": clocks,
        "kernels_ms": per_kernel, "gemm_tflops": gemm_tflops,
        "fwd_quantize_phase_ms": phase_ms, "fwd_quantize_phase_gbs": phase_gbs,
        "fwd_quantize_phase_frac": phase_gbs / hbm_peak,
        "kernels_ms_serial": serial_kernels, "ms_per_step_serial": serial_ms,
        "group_quantize_gbs": quant_gbs, "hbm_peak_gbs": hbm_peak,
        "group_quantize_frac": {k: v / hbm_peak for k, v in quant_gbs.items()},
        "group_quantize_note": "each quantize kernel timed alone (serial pass, L2 flushed before each step); in "
                               "the timed step the quantizations of X and W overlap, and kernels_ms holds their "
                               "concurrent durations",
        "kernels_ms_no_l2_flush": warm,
        "wall_s_timed_region": wall,
        "configs": configs,
        "mlp_step": mlp,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
