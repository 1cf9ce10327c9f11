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
