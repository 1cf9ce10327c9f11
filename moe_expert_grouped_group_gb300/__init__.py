"""GB300-native MXFP8 grouped quantization and grouped GEMM for MoE expert layers.

The compute path is the CUDA library ``libmxq.so`` (C ABI: ``include/mxq.h``),
built in-tree for sm_103a by :func:`moe_expert_grouped_group_gb300.build.build`.
:mod:`moe_expert_grouped_group_gb300.mxq` is its thin PyTorch binding.
"""
from . import mxq  # noqa: F401
from .mxq import (  # noqa: F401
    MXQError,
    group_quantize,
    group_quantize_scaled_bias,
    grouped_dbias,
    grouped_gemm_dgrad,
    grouped_gemm_dgrad_swiglu,
    grouped_gemm_fprop,
    grouped_gemm_fprop_swiglu,
    grouped_gemm_wgrad,
    new_status,
    probe_mma_stream,
    requant_colwise,
    requant_colwise_scaled_bias,
    scale_bytes,
    selftest_wait_timeout,
    status_read,
    swiglu_bwd,
    swiglu_bwd_quantize,
    swiglu_fwd,
    swiglu_quantize,
    workspace_bytes,
)

__version__ = "0.1.0"
