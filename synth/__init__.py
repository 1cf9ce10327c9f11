"""Seeded synthetic inputs for the MoE expert-layer hot path.

This module is shared by the CUDA path's tests/benchmarks and by the CPU
oracle's tests. It holds none of the method's arithmetic: it only draws
random bf16 tensors and per-expert token counts (``m_splits``) with the
shapes and distributions of the five MoE workloads below.

Every draw uses numpy's PCG64 generator seeded by a tuple
``(seed, workload id, tensor id, chunk)``; large tensors are filled chunk by
chunk on a thread pool, so the result is identical for any thread count.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_from_f32,
    f32_from_bf16_bits,
    bf16_normal,
    round_counts_to_128,
    make_m_splits,
    make_inputs,
)
