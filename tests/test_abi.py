"""The C ABI library builds, loads and exports every symbol include/mxq.h
declares (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from moe_expert_grouped_group_gb300.build import build
    from moe_expert_grouped_group_gb300.mxq import load

    return load(build())


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mxq.h")).read()
    return sorted(set(re.findall(r"MXQ_API\s+[\w\s\*]+?\b(mxq_\w+)\s*\(", text)))


def test_header_declares_the_hot_path():
    syms = declared_symbols()
    for s in ("mxq_group_quantize", "mxq_requant_colwise", "mxq_grouped_dbias", "mxq_grouped_gemm_fprop",
              "mxq_grouped_gemm_dgrad", "mxq_grouped_gemm_wgrad", "mxq_swiglu_fwd", "mxq_swiglu_bwd"):
        assert s in syms


def test_every_declared_symbol_is_exported(L):
    from moe_expert_grouped_group_gb300.mxq import SYMBOLS

    syms = declared_symbols()
    assert syms == sorted(SYMBOLS)
    for s in syms:
        assert hasattr(L, s), s
        assert ctypes.cast(getattr(L, s), ctypes.c_void_p).value


def test_host_only_helpers(L, orc):
    assert L.mxq_version() == 100
    for M, K in ((512, 512), (16384, 2048), (384, 1152), (200, 96)):
        r, c = orc.compact_shape(M, K, False)
        assert L.mxq_scale_bytes(M, K, 0) == r * c
        r, c = orc.compact_shape(M, K, True)
        assert L.mxq_scale_bytes(M, K, 1) == r * c
    assert L.mxq_workspace_bytes(1, 1024, 0, 512, 4, 0) == 8 * 512 * 4
    assert L.mxq_workspace_bytes(3, 1024, 640, 0, 4, 0) == 8 * 640 * 4
    assert L.mxq_workspace_bytes(4, 1024, 640, 512, 4, 0) == 0
    assert L.mxq_error_string(-3).decode().startswith("m_splits must be device memory")
    assert L.mxq_last_cuda_error() == 0


def test_no_cpu_fallback_in_the_product_path():
    """The package never imports the oracle or runs compute on the host."""
    pkg = os.path.join(ROOT, "moe_expert_grouped_group_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            src = open(os.path.join(pkg, name)).read()
            assert "oracle" not in src, name
            assert "numpy" not in src, name


def test_compute_entry_points_refuse_without_a_gb300(L):
    """On a host without a GB300 every compute entry point of the hot path returns MXQ_ERR_ARCH, with
    well-formed arguments, before any pointer is used: nothing runs on the host in its place. The
    addresses below are never dereferenced."""
    import torch

    if torch.cuda.is_available() and torch.cuda.get_device_capability(0) == (10, 3):
        pytest.skip("a GB300 is present: the GPU tests cover these calls")
    P, WS = 1 << 20, 1 << 30                     # a 16-byte-aligned address; a workspace size large enough
    M = N = K = 256
    E = 2
    ROW, COL, SWZ, ARCH = 1, 2, 4, -4
    calls = {
        "mxq_group_quantize": (P, M, K, E, P, ROW | COL | SWZ, P, P, P, P, None, None, P, P, WS, None),
        "mxq_requant_colwise": (P, P, M, K, E, P, COL | SWZ, P, P, P, None, None, None, P, P, WS, None),
        "mxq_grouped_dbias": (P, M, N, E, P, P, P, P, WS, None),
        "mxq_grouped_gemm_fprop": (P, P, P, P, None, M, N, K, E, P, P, P, P, WS, None),
        "mxq_grouped_gemm_dgrad": (P, P, P, P, M, N, K, E, P, P, P, P, WS, None),
        "mxq_grouped_gemm_wgrad": (P, P, P, P, M, N, K, E, P, 0, P, P, P, WS, None),
        "mxq_swiglu_fwd": (P, M, K, P, None),
    }
    for name, args in calls.items():
        assert getattr(L, name)(*args) == ARCH, name
