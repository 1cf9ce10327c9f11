"""Test-side builders of MXFP8 operands that do not come from quantizing a
bf16 tensor: random valid E4M3 codes and E8M0 scales, and the swizzled scale
layouts the GEMMs consume, assembled from the compact layout with the
oracle's swizzle (the scale-atom rule of the tcgen05 block-scaled MMA; the
colwise scales of each member as a logical (cols, rows/32) matrix at byte
cols * offset / 32). `tests/test_layouts.py` pins these builders against the
oracle's own swizzled quantizer output."""
import numpy as np

import oracle as orc


def random_codes(rng, n: int, chunk: int = 1 << 28) -> np.ndarray:
    """n uniformly random E4M3 codes with the two NaN codes (0x7F, 0xFF)
    replaced by the largest finite magnitude of the same sign."""
    lo7 = np.uint64(0x7F7F7F7F7F7F7F7F)
    ones = np.uint64(0x0101010101010101)
    top = np.uint64(0x8080808080808080)
    out = np.empty(n, np.uint8)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        w = rng.bit_generator.random_raw((m + 7) // 8).astype(np.uint64, copy=False)
        # per byte: (b & 0x7F) + 1 carries into bit 7 exactly when b & 0x7F == 0x7F
        nan = ((w & lo7) + ones) & top
        w ^= nan >> np.uint64(7)  # S.1111.111 -> S.1111.110 (+-448)
        out[i:i + m] = w.view(np.uint8)[:m]
    return out


def random_scales(rng, shape, lo: int = 118, hi: int = 136) -> np.ndarray:
    """E8M0 codes uniform in [lo, hi] (2^(lo-127) .. 2^(hi-127))."""
    return rng.integers(lo, hi + 1, size=shape, dtype=np.uint8)


def swizzle_rowwise(S_compact: np.ndarray) -> np.ndarray:
    """Rowwise compact scales (R, C), R % 128 == 0, C % 4 == 0 -> swizzled bytes."""
    return orc.swizzle(S_compact)


def swizzle_colwise_grouped(S_compact: np.ndarray, m_splits, cols: int) -> np.ndarray:
    """Colwise compact scales (rows/32, cols) of a grouped tensor -> the
    per-member swizzled layout: member e's scales as the logical
    (cols, m_e/32) matrix, swizzled, at byte cols * off_e / 32."""
    S = np.ascontiguousarray(S_compact, np.uint8)
    out = np.zeros(S.size, np.uint8)
    off = 0
    for me in (int(v) for v in m_splits):
        if me:
            blk = S[off // 32:(off + me) // 32, :cols].T
            base = cols * off // 32
            out[base:base + blk.size] = orc.swizzle(blk)
        off += me
    return out
