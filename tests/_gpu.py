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
