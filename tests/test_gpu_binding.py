"""The Python binding checks every tensor it hands to the library as a raw
pointer: an output smaller than the bytes the call writes, an input smaller
than the bytes it reads, or a wrong element type raises MXQError before any
launch (the library itself cannot see tensor sizes)."""
import numpy as np
import pytest
import torch

from tests._gpu import dev_bf16, dev_i64, lib, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def test_undersized_outputs_are_rejected_and_left_untouched(mxq):
    x = dev_bf16(np.zeros((256, 256), np.uint16))
    ms = dev_i64([128, 128])
    small = torch.full((256 * 256 - 1,), 7, dtype=torch.uint8, device="cuda")
    with pytest.raises(mxq.MXQError, match="row_data"):
        mxq.group_quantize(x, ms, out={"row_data": small})
    with pytest.raises(mxq.MXQError, match="dbias"):
        mxq.group_quantize(x, ms, dbias=True, out={"dbias": torch.empty((2, 255), device="cuda")})
    torch.cuda.synchronize()
    assert torch.all(small == 7)
    q = mxq.group_quantize(x, ms)
    w = torch.zeros((2, 256, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(mxq.MXQError, match="out"):
        mxq.grouped_gemm_fprop(q["row_data"], q["row_scale"], w, q["row_scale"][:0].new_zeros(2 * 256 * 8), ms,
                               out=torch.empty((256, 255), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(mxq.MXQError, match="out"):
        mxq.grouped_gemm_wgrad(q["col_data"], q["col_scale"], q["col_data"], q["col_scale"], ms,
                               out=torch.empty((2, 256, 256), dtype=torch.bfloat16, device="cuda"))


def test_undersized_inputs_and_wrong_types_are_rejected(mxq):
    ms = dev_i64([128, 128])
    with pytest.raises(mxq.MXQError, match="x"):
        mxq.group_quantize(torch.zeros((256, 256), dtype=torch.float32, device="cuda"), ms)
    q = mxq.group_quantize(dev_bf16(np.zeros((256, 256), np.uint16)), ms)
    with pytest.raises(mxq.MXQError, match="w_scale"):
        mxq.grouped_gemm_fprop(q["row_data"], q["row_scale"], torch.zeros((2, 256, 256), dtype=torch.uint8,
                                                                          device="cuda"),
                               torch.zeros(100, dtype=torch.uint8, device="cuda"), ms)
    with pytest.raises(mxq.MXQError, match="status"):
        mxq.group_quantize(dev_bf16(np.zeros((256, 256), np.uint16)), ms,
                           status=torch.zeros(1, dtype=torch.int64, device="cuda"))
