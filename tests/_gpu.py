"""Helpers shared by the GPU parity tests (host <-> device marshalling and
the error measures the tolerances are stated in)."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip("needs an sm_103 (GB300) device")


def lib():
    from __graft_entry__ import build

    build()
    import moe_expert_grouped_group_gb300 as m

    return m


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_i64(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def scaled_error(got: np.ndarray, ref: np.ndarray, mag: np.ndarray) -> float:
    """max |C - C*| / (|A|.|B|), the dot-product error measure; entries whose
    magnitude sum is 0 must be exactly 0."""
    got = np.asarray(got, np.float64)
    zero = mag == 0
    assert np.all(got[zero] == 0), "an entry with no contributing products is not 0"
    if np.all(zero):
        return 0.0
    return float(np.max(np.abs(got[~zero] - ref[~zero]) / mag[~zero]))


def first_diff(a: np.ndarray, b: np.ndarray):
    idx = np.argwhere(a != b)
    return None if idx.size == 0 else (idx.shape[0], idx[:5].tolist(), a[tuple(idx[0])], b[tuple(idx[0])])


# ------------------------------------------------------------ SwiGLU tolerance
# The kernels evaluate SwiGLU in fp32; the oracle's definition is fp64 with one
# final rounding to bf16. Every fp32 step errs by far less than half a bf16 ulp
# (2^-9) relative, so after the final rounding the two may differ by one bf16
# step at most (a rounding boundary between them). The one exception is the
# sigmoid below g = -86: its exact value is under 2^-124 there, where fp32 has
# only subnormals to hold it, and the kernels' flush-to-zero approximations
# give 0 below g = -87.3 (and every fp32 sigmoid is 0 below g = -103.3). The
# results may then be off by up to the whole term, at most |g u| 2^-124 for h,
# |dh u| (1 + |g|) 2^-124 for dg and |dh g| 2^-124 for du, each allowed twice
# over to cover the final rounding of the fp64 result.
SIGMOID_FLUSH_G = -86.0
SIGMOID_FLUSH_BOUND = 2.0 ** -123


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Number of bf16 steps between two arrays of bf16 bit patterns (+0 and -0 coincide)."""
    def key(x):
        x = np.asarray(x).astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)

    return np.abs(key(a) - key(b))


def _gate_up(y_bits):
    y = bf16_to_f64(y_bits)
    F = y.shape[1] // 2
    return y[:, :F], y[:, F:]


def swiglu_fwd_slack(y_bits: np.ndarray) -> np.ndarray:
    g, u = _gate_up(y_bits)
    return np.where(g < SIGMOID_FLUSH_G, np.abs(g * u) * SIGMOID_FLUSH_BOUND, 0.0)


def swiglu_bwd_slack(dh_bits: np.ndarray, y_bits: np.ndarray) -> np.ndarray:
    g, u = _gate_up(y_bits)
    dh = np.abs(bf16_to_f64(dh_bits))
    flush = g < SIGMOID_FLUSH_G
    dg = np.where(flush, dh * np.abs(u) * (1 + np.abs(g)) * SIGMOID_FLUSH_BOUND, 0.0)
    du = np.where(flush, dh * np.abs(g) * SIGMOID_FLUSH_BOUND, 0.0)
    return np.concatenate([dg, du], axis=1)


def assert_swiglu_close(got: np.ndarray, ref: np.ndarray, slack: np.ndarray, what: str = ""):
    """got (kernel) and ref (the oracle's fp64 definition), bf16 bits: within one bf16 step,
    or within the sigmoid-flush bound `slack` (fp64, same shape)."""
    near = bf16_ulp_distance(got, ref) <= 1
    flushed = np.abs(bf16_to_f64(got) - bf16_to_f64(ref)) <= slack
    ok = near | flushed
    assert ok.all(), (what, first_diff(np.where(ok, 0, got), np.where(ok, 0, ref)))
