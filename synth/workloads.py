"""Workload definitions and seeded generators (see package docstring).

The five workloads mirror the MoE expert-layer shapes the method targets:
routed-token counts per expert that are multiples of 128 (the expert-parallel
dispatch guarantees this alignment), bf16 activations ~N(0,1), weights
~N(0,0.02), and for the largest one amax stress (rare x1000 outliers) plus
all-zero 32x32 tiles.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 23  # elements per independently seeded chunk


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int
    E: int
    K: int          # hidden (reduction width of the first GEMM's input)
    N: int          # out_features of the (first) grouped linear
    M: int          # total routed rows = sum(m_splits)
    F: int = 0      # SwiGLU inner width (0: a single grouped linear)
    prequant_x: bool = False     # X arrives rowwise-quantized (EP dispatch)
    prequant_dy: bool = False    # FC2 dY arrives rowwise-quantized
    bias: bool = False
    description: str = ""


WORKLOADS = {
    "e4_h512_n1024_t512": Workload(
        "e4_h512_n1024_t512", 1, E=4, K=512, N=1024, M=512,
        description="4 experts, hidden 512, out 1024, m_splits [128,256,0,128]"),
    "e8_h2048_n4096_t16k_prequant": Workload(
        "e8_h2048_n4096_t16k_prequant", 2, E=8, K=2048, N=4096, M=16384,
        prequant_x=True,
        description="8 experts, hidden 2048, out 4096, 16384 tokens, uniform "
                    "multinomial routing, X rowwise-prequantized"),
    "e32_h4096_f1536_t64k_swiglu": Workload(
        "e32_h4096_f1536_t64k_swiglu", 3, E=32, K=4096, N=2 * 1536, M=65536,
        F=1536,
        description="32 experts, hidden 4096, FC1 2x1536 -> SwiGLU -> FC2 "
                    "1536->4096, 65536 tokens, Zipf(1.2) routing"),
    "e64_h3072_f1024_t84k_prequant": Workload(
        "e64_h3072_f1024_t84k_prequant", 4, E=64, K=3072, N=2 * 1024,
        M=83968, F=1024, prequant_x=True, prequant_dy=True, bias=True,
        description="64 experts, hidden 3072, FC1 2x1024 -> SwiGLU -> FC2 "
                    "1024->3072, 83968 routed rows, top-8 Dirichlet(0.3)"),
    "e128_h7168_n2048_t128k_skew": Workload(
        "e128_h7168_n2048_t128k_skew", 5, E=128, K=7168, N=2048, M=131072,
        description="128 experts (32 empty), hidden 7168, out 2048, 131072 "
                    "tokens, Pareto(1.2) loads, x1000 outliers, zero tiles"),
}


# ---------------------------------------------------------------- bf16 bits
def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).copy()
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def bf16_normal(shape, std: float, key: tuple) -> np.ndarray:
    """bf16 bits of N(0, std^2) draws, generated in seeded chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c):
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        rng = np.random.default_rng([*key, c])
        a = rng.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        out[lo:hi] = bf16_bits_from_f32(a)

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


# ------------------------------------------------------------- m_splits
def round_counts_to_128(c, total: int) -> np.ndarray:
    """Round raw per-expert counts (summing to ``total``) to multiples of 128.

    Each expert first gets floor(c_e/128) units of 128; the remaining
    total/128 - sum units go to the largest fractional remainders, ties to
    the lower expert index. Experts with c_e == 0 stay 0.
    """
    c = np.asarray(c, dtype=np.float64)
    assert total % 128 == 0
    units = c / 128.0
    base = np.floor(units).astype(np.int64)
    rem = units - base
    left = total // 128 - int(base.sum())
    assert left >= 0
    order = sorted(range(len(c)), key=lambda e: (-rem[e], e))
    for e in order[:left]:
        assert c[e] > 0
        base[e] += 1
    out = base * 128
    assert int(out.sum()) == total
    return out.astype(np.int64)


def make_m_splits(w: Workload, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng([seed, w.wid, 0xA11])
    if w.wid == 1:
        return np.array([128, 256, 0, 128], dtype=np.int64)
    if w.wid == 2:
        c = rng.multinomial(w.M, np.full(w.E, 1.0 / w.E))
        return round_counts_to_128(c, w.M)
    if w.wid == 3:
        ranks = rng.permutation(np.arange(1, w.E + 1))
        p = ranks.astype(np.float64) ** -1.2
        p /= p.sum()
        c = rng.multinomial(w.M, p)
        return round_counts_to_128(c, w.M)
    if w.wid == 4:
        topk = 8
        src = w.M // topk
        p = rng.dirichlet(np.full(w.E, 0.3))
        c = np.zeros(w.E, dtype=np.int64)
        for _ in range(src):
            c[rng.choice(w.E, size=topk, replace=False, p=p)] += 1
        return round_counts_to_128(c, w.M)
    if w.wid == 5:
        zero = rng.choice(w.E, size=32, replace=False)
        wt = rng.pareto(1.2, size=w.E) + 1.0
        wt[zero] = 0.0
        c = w.M * wt / wt.sum()
        return round_counts_to_128(c, w.M)
    raise ValueError(w.name)


# -------------------------------------------------------------- tensors
def _stress(x_bits: np.ndarray, key: tuple) -> np.ndarray:
    """x1000 outliers on 0.1% of elements, then 0.5% of aligned 32x32 tiles zeroed."""
    M, K = x_bits.shape
    rng = np.random.default_rng([*key, 0x5EED])
    tiles = rng.random((M // 32, K // 32)) < 0.005
    rows = max(32, (_CHUNK // K) // 32 * 32)
    out = np.empty_like(x_bits)

    def fill(c):
        lo = c * rows
        hi = min(M, lo + rows)
        crng = np.random.default_rng([*key, 0x5EED, c])
        x = f32_from_bf16_bits(x_bits[lo:hi]).reshape(hi - lo, K)
        hit = crng.random((hi - lo, K), dtype=np.float32) < np.float32(0.001)
        x[hit] *= np.float32(1000.0)
        ti, tj = np.nonzero(tiles[lo // 32:hi // 32])
        for i, j in zip(ti, tj):
            x[32 * i:32 * i + 32, 32 * j:32 * j + 32] = 0.0
        out[lo:hi] = bf16_bits_from_f32(x)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range((M + rows - 1) // rows)))
    return out


def make_inputs(w: Workload, seed: int = 0, which=("x", "w", "dy")) -> dict:
    """Seeded bf16 inputs (uint16 bit arrays) for one workload.

    Keys: ``m_splits`` always; ``x`` (M,K), ``w`` (E,N,K), ``dy`` (M,N) for
    the first grouped linear; for SwiGLU workloads also ``w2`` (E,K,F) and
    ``dy2`` (M,K) of the second linear; ``b1``/``b2`` biases when the
    workload has them.
    """
    out = {"m_splits": make_m_splits(w, seed)}
    k = (seed, w.wid)
    if "x" in which:
        out["x"] = bf16_normal((w.M, w.K), 1.0, (*k, 1))
        if w.wid == 5:
            out["x"] = _stress(out["x"], (*k, 1))
    if "w" in which:
        out["w"] = bf16_normal((w.E, w.N, w.K), 0.02, (*k, 2))
    if "dy" in which:
        out["dy"] = bf16_normal((w.M, w.N), 1.0, (*k, 3))
    if w.F:
        if "w2" in which:
            out["w2"] = bf16_normal((w.E, w.K, w.F), 0.02, (*k, 4))
        if "dy2" in which:
            out["dy2"] = bf16_normal((w.M, w.K), 1.0, (*k, 5))
    if w.bias:
        if "b1" in which:
            out["b1"] = bf16_normal((w.E, w.N), 0.02, (*k, 6))
        if "b2" in which:
            out["b2"] = bf16_normal((w.E, w.K), 0.02, (*k, 7))
    return out
