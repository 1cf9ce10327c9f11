"""Concurrent calls on separate CUDA streams, through the C ABI: the
library keeps no device state between calls (every scratch buffer is the
caller's), so calls running at the same time on different streams give
exactly what they give one after another. A grouped-linear step with the
forward's requant of X on a side stream beside the quantization of W (as
bench.py runs it), plus a quantize with fused dbias and a GEMM on a third
stream, is compared byte for byte with the same calls in order on one
stream; the quantized codes and scales are also checked against the oracle
(bit-exact)."""
import numpy as np
import pytest
import torch

import oracle as orc
from synth import bf16_bits_from_f32
from tests._gpu import dev_bf16, dev_i64, dev_u8, first_diff, host, lib, require_gpu

pytestmark = pytest.mark.gpu

E, K, N = 8, 512, 768
MS = np.array([256, 0, 384, 128, 512, 128, 0, 640], np.int64)
M = int(MS.sum())


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


@pytest.fixture(scope="module")
def inputs():
    rng = np.random.default_rng([5, 7])
    x = bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))
    w = bf16_bits_from_f32((0.02 * rng.standard_normal((E * N, K))).astype(np.float32))
    dy = bf16_bits_from_f32(rng.standard_normal((M, N)).astype(np.float32))
    wire = orc.group_quantize(x, MS, rowwise=True, colwise=False)
    return x, w, dy, wire


def _step(mxq, d, concurrent):
    """requant X | quantize W, fprop, quantize dY (+dbias) | a second fprop; returns every output."""
    ms = d["ms"]
    main = torch.cuda.current_stream()
    side, third = torch.cuda.Stream(), torch.cuda.Stream()
    out = {}
    if concurrent:
        fork = torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            out["rq"] = mxq.requant_colwise(d["x_row"], d["x_rs"], ms)
        j = torch.cuda.Event()
        j.record(side)
        out["qw"] = mxq.group_quantize(d["w"], None, E=E)
        main.wait_event(j)
    else:
        out["rq"] = mxq.requant_colwise(d["x_row"], d["x_rs"], ms)
        out["qw"] = mxq.group_quantize(d["w"], None, E=E)
    wq = out["qw"]["row_data"].view(E, N, K)
    out["y"] = mxq.grouped_gemm_fprop(d["x_row"], out["rq"]["row_scale_swizzled"], wq, out["qw"]["row_scale"], ms)
    if concurrent:
        fork2 = torch.cuda.Event()
        fork2.record(main)
        third.wait_event(fork2)
        with torch.cuda.stream(third):
            out["y2"] = mxq.grouped_gemm_fprop(d["x_row"], out["rq"]["row_scale_swizzled"], wq,
                                               out["qw"]["row_scale"], ms)
        out["qdy"] = mxq.group_quantize(d["dy"], ms, dbias=True)
        j2 = torch.cuda.Event()
        j2.record(third)
        main.wait_event(j2)
    else:
        out["y2"] = mxq.grouped_gemm_fprop(d["x_row"], out["rq"]["row_scale_swizzled"], wq, out["qw"]["row_scale"],
                                           ms)
        out["qdy"] = mxq.group_quantize(d["dy"], ms, dbias=True)
    torch.cuda.synchronize()
    flat = {}
    for k, v in out.items():
        if isinstance(v, dict):
            flat.update({f"{k}.{kk}": host(vv) for kk, vv in v.items()})
        else:
            flat[k] = host(v)
    return flat


def test_concurrent_streams_match_serial_and_oracle(mxq, inputs):
    x, w, dy, wire = inputs
    d = {"ms": dev_i64(MS), "x_row": dev_u8(wire["row_q"]), "x_rs": dev_u8(wire["row_s"]), "w": dev_bf16(w),
         "dy": dev_bf16(dy)}
    serial = _step(mxq, d, False)
    for _ in range(3):  # several rounds: a race would not show every time
        conc = _step(mxq, d, True)
        assert serial.keys() == conc.keys()
        for k in serial:
            assert np.array_equal(serial[k], conc[k]), (k, first_diff(serial[k], conc[k]))
    # the codes and scales themselves, against the oracle
    rq = orc.requant_colwise(wire["row_q"], wire["row_s"], MS, swizzled=True)
    assert np.array_equal(serial["rq.col_data"].reshape(-1), np.asarray(rq["col_q"]).reshape(-1))
    assert np.array_equal(serial["rq.col_scale"].reshape(-1), np.asarray(rq["col_s"]).reshape(-1))
    qdy = orc.group_quantize(dy, MS, swizzled=True)
    assert np.array_equal(serial["qdy.row_data"].reshape(qdy["row_q"].shape), qdy["row_q"])
    assert np.array_equal(serial["qdy.col_scale"].reshape(-1), np.asarray(qdy["col_s"]).reshape(-1))
    assert np.array_equal(serial["y"], serial["y2"])
