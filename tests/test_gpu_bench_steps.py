"""The steps bench.py times, run through the C ABI: the concurrent schedule
of each (the forward's quantizations on two streams) gives outputs bit-
identical to the same calls in order on one stream, for the grouped-linear
training step of the headline workload (128 experts, hidden 7168) and the
64-expert SwiGLU MLP step. The calls
themselves are checked against the oracle by the other GPU tests; this pins
the streams and events of the timed steps."""
import numpy as np
import pytest
import torch

import bench
from tests._gpu import first_diff, require_gpu

pytestmark = pytest.mark.gpu


def _snap(tensors):
    torch.cuda.synchronize()
    return {k: v.clone() for k, v in tensors.items()}


def _same(a, b):
    for k in a:
        if not torch.equal(a[k], b[k]):
            x = a[k].view(torch.uint8).cpu().numpy().reshape(-1)
            y = b[k].view(torch.uint8).cpu().numpy().reshape(-1)
            raise AssertionError((k, first_diff(x, y)))


def test_grouped_linear_step_concurrent_equals_serial():
    require_gpu()
    dev = torch.device("cuda", 0)
    w, d = bench.make_host_workload()
    st = bench.NativeStep(w, d, dev)

    def outs():
        o = {"y": st.y, "dx": st.dx, "dw": st.dw}
        o.update({f"qx.{k}": v for k, v in st.qx.items()})
        o.update({f"qw.{k}": v for k, v in st.qw.items()})
        o.update({f"qdy.{k}": v for k, v in st.qdy.items()})
        return o

    st.run(concurrent=False)
    ref = _snap(outs())
    for v in outs().values():
        v.zero_()
    for _ in range(2):
        st.run()
        _same(ref, _snap(outs()))
    assert float(ref["y"].float().abs().max()) > 0 and float(ref["dw"].abs().max()) > 0
    del st
    torch.cuda.empty_cache()


def test_mlp_step_concurrent_equals_serial():
    require_gpu()
    dev = torch.device("cuda", 0)
    st = bench.MLPStep(dev)

    def outs():
        o = {"y1": st.y1, "y2": st.y2, "dh": st.dh, "dx": st.dx, "dw1": st.dw1, "dw2": st.dw2}
        for name, q in (("qx", st.qx), ("qd", st.qd), ("qh", st.qh), ("qdy1", st.qdy1), ("qw1", st.qw1)):
            o.update({f"{name}.{k}": v for k, v in q.items()})
        return o

    st.run(concurrent=False)
    ref = _snap(outs())
    for v in outs().values():
        v.zero_()
    st.run()
    _same(ref, _snap(outs()))
    assert float(ref["y2"].float().abs().max()) > 0 and float(ref["dw1"].abs().max()) > 0
    del st
    torch.cuda.empty_cache()
