"""Host-side arithmetic of bench.py: the per-expert GEMM roofline, the step layout, the source stamp."""
import pathlib

import pytest

import bench


def test_per_expert_bound_equals_the_dense_bound_when_every_expert_is_compute_bound():
    N, K, peak, bw = 4096, 2048, 3845.4, 6665.6
    ms = [2048] * 8
    b = bench.gemm_bound_us(ms, N, K, peak, bw)
    dense = 2.0 * sum(ms) * N * K / (peak * 1e12) * 1e6
    for k in ("fprop", "dgrad", "wgrad"):
        assert b[k] == pytest.approx(dense, rel=1e-12)


def test_small_and_empty_experts_are_bound_by_their_bytes():
    N, K, peak, bw = 2048, 7168, 3845.4, 6665.6
    q = 1 + 1 / 32
    b = bench.gemm_bound_us([0, 128], N, K, peak, bw)
    # expert 1 (128 rows) streams its weight: W bytes dominate its 2*128*N*K flops
    fprop = (128 * K * q + N * K * q + 128 * N * 2) / (bw * 1e9) * 1e6
    assert b["fprop"] == pytest.approx(fprop, rel=1e-12)
    # the empty expert still writes its fp32 dW zeros; expert 1 writes its fp32 dW
    wgrad = N * K * 4 / (bw * 1e9) * 1e6 + (128 * N * q + 128 * K * q + N * K * 4) / (bw * 1e9) * 1e6
    assert b["wgrad"] == pytest.approx(wgrad, rel=1e-12)
    assert b["dgrad"] == pytest.approx((128 * N * q + N * K * q + 128 * K * 2) / (bw * 1e9) * 1e6, rel=1e-12)


class _FakeEvent:
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_step_event_layout():
    # one step: quantize X 0.1-0.3 on the side stream and quantize W 0.0-0.5 on the main stream, joined at
    # 0.6, then fprop / quantize dY / dgrad / wgrad ending at 1.0 / 1.3 / 1.8 / 2.4
    t = [0.0, 0.1, 0.3, 0.0, 0.5, 0.6, 1.0, 1.3, 1.8, 2.4]
    assert len(t) == bench.STEP_EVENTS
    for pre_x, xk in ((False, "quantize_x"), (True, "requant_x")):
        kev = bench.kernel_events(pre_x)
        per, per_step, phase = bench.step_event_times([[_FakeEvent(v) for v in t]], kev)
        assert per == pytest.approx({xk: 0.2, "quantize_w": 0.5, "fprop": 0.4, "quantize_dy": 0.3,
                                     "dgrad": 0.5, "wgrad": 0.6})
        assert per_step == pytest.approx([2.4]) and phase == pytest.approx(0.6)


def test_both_arms_name_the_same_workload():
    from types import SimpleNamespace

    import numpy as np

    w = SimpleNamespace(name=bench.WORKLOAD, E=128, K=7168, N=2048, M=131072, prequant_x=False)
    d = {"m_splits": np.full(128, 1024, np.int64)}
    c = bench.workload_config(w, d, 1)
    assert c["workload"] == bench.WORKLOAD and c["m_splits"] == [1024] * 128 and c["parallelism"] == "replicas x1"
    assert (c["experts"], c["hidden"], c["out"], c["tokens"]) == (128, 7168, 2048, 131072)
    assert c["step"].startswith("quantize X (row+col)")


def test_headline_is_the_largest_workload():
    from synth import WORKLOADS

    w = WORKLOADS[bench.WORKLOAD]
    assert all(6 * v.M * v.N * v.K <= 6 * w.M * w.N * w.K for v in WORKLOADS.values())


def test_oracle_sample_is_the_stated_fraction_of_the_gemm_work():
    """The reference arm's step: f of each GEMM's flops, so f * step flops / time is its rate."""
    from types import SimpleNamespace

    import numpy as np

    w = SimpleNamespace(E=2, K=256, N=256, M=1024, prequant_x=False)
    rng = np.random.default_rng(0)
    bits = lambda *sh: (rng.standard_normal(sh).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    d = {"x": bits(1024, 256), "dy": bits(1024, 256), "w": bits(2, 256, 256)}
    f = 1 / 4
    s = bench.OracleSample(w, d, f)
    M, N, K = w.M, w.N, w.K
    gemm_flops = 2 * s.nf * K + 2 * s.nd * N + 2 * s.nw * s.rows
    assert gemm_flops == pytest.approx(f * 6 * M * N * K, rel=1e-9)
    t = s.run()
    assert set(t) == {"quantize_x", "quantize_w", "quantize_dy", "fprop", "dgrad", "wgrad"}


def test_inner_repeat_reaches_the_timed_region():
    class _St:
        pass

    assert bench.inner_repeat(_St(), 20, 7) == 7


def test_source_stamp_ignores_comments_but_not_code(tmp_path, monkeypatch):
    """The GEMM traffic record is matched to the code by a stamp of the kernel sources without their
    comments: editing a comment keeps it, editing code changes it, and string literals (PTX) stay whole."""
    from moe_expert_grouped_group_gb300 import build as B

    text = 'int a = 1;  // note\n/* block\n comment */ asm("mov.b32 %0, 1; // kept");\nchar c = \'"\';\n'
    code = B._code_only(text)
    assert "note" not in code and "block" not in code
    assert 'asm("mov.b32 %0, 1; // kept");' in code and "char c = '\"';" in code

    for n in ("mxq_gemm.cu", "mxq_common.cuh", "mxq_internal.h"):
        (tmp_path / n).write_text(pathlib.Path(B.CSRC, n).read_text())
    monkeypatch.setattr(B, "CSRC", str(tmp_path))
    base = B.source_stamp()
    gemm = tmp_path / "mxq_gemm.cu"
    src = gemm.read_text()
    gemm.write_text("// a new comment line\n" + src.replace("// One-SM kernel", "// The one-SM kernel", 1))
    assert B.source_stamp() == base
    gemm.write_text(src + "\nstatic int mxq_stamp_probe = 1;\n")
    assert B.source_stamp() != base
