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


def test_probe_with_random_operands_runs_and_reports_no_timeout(mxq):
    status = mxq.new_status()
    for n in (0, 4, 1024):
        flops = mxq.probe_mma_stream(n, status=status, random=True)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert flops == 2.0 * 128 * 256 * 32 * n * sms
    torch.cuda.synchronize()
    assert mxq.status_read(status) == 0


def test_probe_rejects_an_unknown_operand_mode(mxq):
    rc = mxq.mxq.lib().mxq_probe_mma_stream_ex(4, 2, None, None)
    assert rc == -7  # MXQ_ERR_FLAGS


def test_probe_rejects_bad_counts(mxq):
    with pytest.raises(mxq.MXQError):
        mxq.probe_mma_stream(-1)
    with pytest.raises(mxq.MXQError):
        mxq.probe_mma_stream(1 << 31)


def test_an_expired_wait_reports_its_status_and_leaves_the_context_usable(mxq):
    """Failure detection without a fault: a bounded on-chip wait on an mbarrier
    that nothing arrives on expires, the kernel sets STATUS_WAIT_TIMEOUT and
    returns; the next calls on the same context run normally."""
    import time

    import numpy as np

    import oracle as orc
    from synth import bf16_bits_from_f32
    from tests._gpu import dev_bf16, dev_i64, host

    status = mxq.new_status()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mxq.selftest_wait_timeout(status, limit_ns=20_000_000)
    got = mxq.status_read(status)
    elapsed = time.perf_counter() - t0
    assert got & mxq.mxq.STATUS_WAIT_TIMEOUT
    assert 0.02 <= elapsed < 5.0
    fresh = mxq.new_status()
    x = bf16_bits_from_f32(np.random.default_rng(9).standard_normal((256, 256)).astype(np.float32))
    q = mxq.group_quantize(dev_bf16(x), dev_i64([128, 128]), status=fresh)
    assert mxq.status_read(fresh) == 0
    o = orc.group_quantize(x, np.array([128, 128]), swizzled=True)
    assert np.array_equal(host(q["row_data"]), o["row_q"])


def test_the_self_test_rejects_bad_limits(mxq):
    status = mxq.new_status()
    for bad in (0, 999, 10_000_000_001):
        with pytest.raises(mxq.MXQError):
            mxq.selftest_wait_timeout(status, limit_ns=bad)
    assert mxq.status_read(status) == 0
