"""The tensor-pipe ceiling probe (mxq_probe_mma_stream) runs to completion
through the C ABI without a wait timing out, and rejects bad counts."""
import pytest
import torch

from tests._gpu import lib, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    require_gpu()
    return lib()


def test_probe_runs_and_reports_no_timeout(mxq):
    status = mxq.new_status()
    for n in (0, 4, 1024):
        flops = mxq.probe_mma_stream(n, status=status)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert flops == 2.0 * 128 * 256 * 32 * n * sms
    assert mxq.status_read(status) == 0


def test_probe_rejects_bad_counts(mxq):
    with pytest.raises(mxq.MXQError):
        mxq.probe_mma_stream(-1)
    with pytest.raises(mxq.MXQError):
        mxq.probe_mma_stream(1 << 31)
