"""CPU oracle for the MXFP8 grouped quantization + grouped GEMM hot path.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke
check and the benchmark's CPU-baseline leg, never by the product path. It
shares no code with the CUDA library; its arithmetic lives in the plain C
file ``mxq_oracle.c`` (fp64, one definition per function, each citing the
TransformerEngine pull-request page it follows). This module only marshals
numpy arrays into it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exhaustive codec enumeration, closed forms, invariants, brute force on tiny
inputs). There is no worked numeric example on the pages, so no end-to-end
golden tensor exists; see the pins for what fixes each part.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, library_path

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = library_path()
        src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "mxq_oracle.c")
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(src):
            build_oracle()
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int


def _declare(L):
    L.orc_bf16_value.argtypes = [ctypes.c_uint16]
    L.orc_bf16_value.restype = ctypes.c_double
    L.orc_bf16_round.argtypes = [ctypes.c_double]
    L.orc_bf16_round.restype = ctypes.c_uint16
    L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_value.restype = ctypes.c_double
    L.orc_e4m3_encode.argtypes = [ctypes.c_double]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_e8m0_exponent.argtypes = [ctypes.c_double]
    L.orc_e8m0_exponent.restype = _INT
    L.orc_quantize_block.argtypes = [_P, _INT, _P, _P]
    L.orc_e4m3_encode_n.argtypes = [_P, _I64, _P]
    L.orc_e8m0_exponent_n.argtypes = [_P, _I64, _P]
    L.orc_bf16_round_n.argtypes = [_P, _I64, _P]
    L.orc_swizzle_offset.argtypes = [_I64, _I64, _I64]
    L.orc_swizzle_offset.restype = _I64
    L.orc_swizzle.argtypes = [_P, _I64, _I64, _I64, _I64, _P]
    L.orc_compact_shape.argtypes = [_I64, _I64, _INT, _P, _P]
    L.orc_check_splits.argtypes = [_P, _INT, _I64]
    L.orc_check_splits.restype = _INT
    L.orc_group_quantize.argtypes = [_P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P]
    L.orc_group_quantize.restype = _INT
    L.orc_dequant_rowwise.argtypes = [_P, _P, _I64, _I64, _P]
    L.orc_dequant_colwise.argtypes = [_P, _P, _I64, _I64, _P]
    L.orc_requant_colwise.argtypes = [_P, _P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P]
    L.orc_requant_colwise.restype = _INT
    L.orc_grouped_dbias.argtypes = [_P, _I64, _I64, _INT, _P, _P]
    L.orc_grouped_dbias.restype = _INT
    L.orc_fprop_entries.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _I64, _P, _P, _P, _P]
    L.orc_dgrad_entries.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _I64, _P, _P, _P, _P]
    L.orc_wgrad_entries.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _I64, _P, _P, _P, _P, _P]
    L.orc_swiglu_fwd.argtypes = [_P, _I64, _I64, _P]
    L.orc_swiglu_bwd.argtypes = [_P, _P, _I64, _I64, _P]
    L.orc_scaled_bias_grads.argtypes = [_P, _I64, _I64, _INT, _P, _P, _P, _P, _P]
    L.orc_scaled_bias_grads.restype = _INT
    L.orc_num_threads.restype = _INT


def _p(a):
    return None if a is None else a.ctypes.data_as(_P)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ codecs
def bf16_value(b: int) -> float:
    return lib().orc_bf16_value(int(b))


def bf16_round(v: float) -> int:
    return lib().orc_bf16_round(float(v))


def e4m3_value(c: int) -> float:
    return lib().orc_e4m3_value(int(c))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def e8m0_exponent(amax: float) -> int:
    return lib().orc_e8m0_exponent(float(amax))


def e4m3_encode_array(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_n(_p(v), v.size, _p(out))
    return out


def e8m0_exponent_array(a) -> np.ndarray:
    a = _c(a, np.float64)
    out = np.empty(a.shape, np.int32)
    lib().orc_e8m0_exponent_n(_p(a), a.size, _p(out))
    return out


def bf16_round_array(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_round_n(_p(v), v.size, _p(out))
    return out


def quantize_block(v) -> tuple[np.ndarray, int]:
    v = _c(v, np.float64)
    codes = np.zeros(v.size, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().orc_quantize_block(_p(v), v.size, _p(codes), _p(sc))
    return codes, int(sc[0])


# ----------------------------------------------------------------- layouts
def compact_shape(M: int, K: int, colwise: bool) -> tuple[int, int]:
    r = np.zeros(1, np.int64)
    c = np.zeros(1, np.int64)
    lib().orc_compact_shape(M, K, int(colwise), _p(r), _p(c))
    return int(r[0]), int(c[0])


def swizzle_offset(r: int, c: int, C: int) -> int:
    return lib().orc_swizzle_offset(r, c, C)


def swizzle(S: np.ndarray) -> np.ndarray:
    """Swizzle a logical (R, C) uint8 scale matrix (R%128 == 0, C%4 == 0)."""
    S = _c(S, np.uint8)
    R, C = S.shape
    out = np.zeros(R * C, np.uint8)
    lib().orc_swizzle(_p(S), R, C, C, 1, _p(out))
    return out


# ---------------------------------------------------------------- quantize
def group_quantize(x_bits, m_splits, rowwise=True, colwise=True, swizzled=False):
    """Returns dict with row_q, row_s, col_q, col_s (None when not asked)."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    ms = _c(m_splits, np.int64)
    rr, rc = compact_shape(M, K, False)
    cr, cc = compact_shape(M, K, True)
    row_q = np.zeros((M, K), np.uint8) if rowwise else None
    col_q = np.zeros((M, K), np.uint8) if colwise else None
    row_s = np.zeros(rr * rc, np.uint8) if rowwise else None
    col_s = np.zeros(cr * cc, np.uint8) if colwise else None
    if not swizzled:
        if rowwise:
            row_s = row_s.reshape(rr, rc)
        if colwise:
            col_s = col_s.reshape(cr, cc)
    rc_ = lib().orc_group_quantize(_p(x), M, K, len(ms), _p(ms), int(swizzled),
                                   _p(row_q), _p(row_s), _p(col_q), _p(col_s))
    if rc_ != 0:
        raise ValueError(f"orc_group_quantize rejected the input ({rc_})")
    return {"row_q": row_q, "row_s": row_s, "col_q": col_q, "col_s": col_s}


def quantize_weights(w_bits, rowwise=True, colwise=True, swizzled=False):
    """Weights (E, N, K): E uniform members of N rows (the uniform-group mode)."""
    w = _c(w_bits, np.uint16)
    E, N, K = w.shape
    return group_quantize(w.reshape(E * N, K), np.full(E, N, np.int64), rowwise, colwise, swizzled)


def dequant_rowwise(q, S_compact):
    q = _c(q, np.uint8)
    M, K = q.shape
    out = np.empty((M, K), np.float64)
    lib().orc_dequant_rowwise(_p(q), _p(_c(S_compact, np.uint8)), M, K, _p(out))
    return out


def dequant_colwise(q, S_compact):
    q = _c(q, np.uint8)
    M, K = q.shape
    out = np.empty((M, K), np.float64)
    lib().orc_dequant_colwise(_p(q), _p(_c(S_compact, np.uint8)), M, K, _p(out))
    return out


def requant_colwise(row_q, row_s_compact, m_splits, swizzled=True, dbias=False, dequant=False):
    q = _c(row_q, np.uint8)
    M, K = q.shape
    ms = _c(m_splits, np.int64)
    cr, cc = compact_shape(M, K, True)
    col_q = np.zeros((M, K), np.uint8)
    col_s = np.zeros(cr * cc, np.uint8)
    if not swizzled:
        col_s = col_s.reshape(cr, cc)
    rr, rc = compact_shape(M, K, False)
    row_sw = np.zeros(rr * rc, np.uint8)
    db = np.zeros((len(ms), K), np.float64) if dbias else None
    deq = np.zeros((M, K), np.uint16) if dequant else None
    r = lib().orc_requant_colwise(_p(q), _p(_c(row_s_compact, np.uint8)), M, K, len(ms), _p(ms),
                                  int(swizzled), _p(col_q), _p(col_s), _p(row_sw), _p(db), _p(deq))
    if r != 0:
        raise ValueError(f"orc_requant_colwise rejected the input ({r})")
    return {"col_q": col_q, "col_s": col_s, "row_s_swizzled": row_sw, "dbias": db, "deq": deq}


# ------------------------------------------- experts not aligned to 128 rows
# TransformerEngine PR #3244's review notes that swizzling a grouped
# activation as one dense tensor is valid only when every expert's token count
# is padded to a multiple of 128, and that a grouped swizzle handles variable
# per-expert dims. Reading: each expert is padded with zero rows up to a
# multiple of 128 and quantized by the aligned rules. Zero rows never raise a block's
# amax, so a partial 32-row colwise block is scaled by its real rows only.
# The E4M3 codes keep the dense (M, K) layout and the compact rowwise scales
# stay dense (rowwise blocks do not depend on the grouping); swizzled scales
# and colwise compact scales live in the padded row space of
# R = sum_e round_up(m_e, 128) rows, expert e's rows starting at
# P_e = sum_{e' < e} round_up(m_e', 128); pad bytes are 0.

def padded_offsets(m_splits):
    """(P, mp): padded row offsets P[0..E] and padded counts round_up(m_e, 128)."""
    ms = np.asarray(m_splits, np.int64)
    mp = (ms + 127) // 128 * 128
    return np.concatenate([[0], np.cumsum(mp)]).astype(np.int64), mp


def pad_rows(a, m_splits):
    """Rows of a (M, ...) placed at their padded positions; pad rows are zero."""
    ms = np.asarray(m_splits, np.int64)
    P, _ = padded_offsets(ms)
    off = np.concatenate([[0], np.cumsum(ms)])
    out = np.zeros((int(P[-1]),) + a.shape[1:], a.dtype)
    for e in range(len(ms)):
        out[P[e]:P[e] + ms[e]] = a[off[e]:off[e + 1]]
    return out


def unpad_rows(a, m_splits):
    """Inverse of pad_rows: the real rows of a padded (R, ...) array, dense."""
    ms = np.asarray(m_splits, np.int64)
    P, _ = padded_offsets(ms)
    return np.concatenate([a[P[e]:P[e] + ms[e]] for e in range(len(ms))], axis=0)


def group_quantize_padded(x_bits, m_splits, rowwise=True, colwise=True, swizzled=False):
    """Grouped quantization with any expert counts (see above). Returns row_q, col_q (M, K);
    row_s: compact (round_up(M,128), K/32 padded to 4) dense, or swizzled over R rows;
    col_s: compact (R/32, K) or swizzled per expert at byte K*P_e/32."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    ms = _c(m_splits, np.int64)
    _, mp = padded_offsets(ms)
    o = group_quantize(pad_rows(x, ms), mp, rowwise, colwise, swizzled)
    out = {"row_q": None, "row_s": o["row_s"], "col_q": None, "col_s": o["col_s"]}
    if rowwise:
        out["row_q"] = unpad_rows(o["row_q"], ms)
        if not swizzled:
            rr, rc = compact_shape(M, K, False)
            dense = np.zeros((rr, rc), np.uint8)
            dense[:M] = unpad_rows(o["row_s"], ms)
            out["row_s"] = dense
    if colwise:
        out["col_q"] = unpad_rows(o["col_q"], ms)
    return out


def requant_colwise_padded(row_q, row_s_compact, m_splits, swizzled=True, dbias=False, dequant=False):
    """Requant with any expert counts: the dense wire format (codes + dense compact rowwise
    scales) is padded with zero rows (code 0 scales), requantized by the aligned rules, and the
    codes and dequantized rows are taken back to the dense layout; col_s and row_s_swizzled
    stay in the padded row space."""
    q = _c(row_q, np.uint8)
    M, K = q.shape
    ms = _c(m_splits, np.int64)
    P, mp = padded_offsets(ms)
    R = int(P[-1])
    rr, rc = compact_shape(R, K, False)
    s_p = np.zeros((rr, rc), np.uint8)
    s_p[:R] = pad_rows(np.asarray(row_s_compact).reshape(-1, rc)[:M], ms)
    o = requant_colwise(pad_rows(q, ms), s_p, mp, swizzled=swizzled, dbias=dbias, dequant=dequant)
    o["col_q"] = unpad_rows(o["col_q"], ms)
    if dequant:
        o["deq"] = unpad_rows(o["deq"], ms)
    return o


def grouped_dbias_padded(dy_bits, m_splits):
    """Per-expert column sums for any expert counts (pad rows are zero)."""
    ms = _c(m_splits, np.int64)
    _, mp = padded_offsets(ms)
    return grouped_dbias(pad_rows(_c(dy_bits, np.uint16), ms), mp)


def grouped_dbias(dy_bits, m_splits):
    dy = _c(dy_bits, np.uint16)
    M, N = dy.shape
    ms = _c(m_splits, np.int64)
    out = np.zeros((len(ms), N), np.float64)
    if lib().orc_grouped_dbias(_p(dy), M, N, len(ms), _p(ms), _p(out)) != 0:
        raise ValueError("orc_grouped_dbias rejected the input")
    return out


def scaled_bias_grads(dy_values, m_splits, probs, bias_bits, dbias=True, dprobs=True):
    """Scaled-bias and routing-scale gradients (see mxq_oracle.c): dy_values
    (M, N) exact values in float64, probs (M,) float32, bias_bits (E, N) bf16
    bits. Returns (db (E, N), ds (M,)) in float64 (None where not asked)."""
    dy = _c(dy_values, np.float64)
    M, N = dy.shape
    ms = _c(m_splits, np.int64)
    db = np.zeros((len(ms), N), np.float64) if dbias else None
    ds = np.zeros(M, np.float64) if dprobs else None
    rc = lib().orc_scaled_bias_grads(_p(dy), M, N, len(ms), _p(ms), _p(_c(probs, np.float32)),
                                     _p(_c(bias_bits, np.uint16)), _p(db), _p(ds))
    if rc != 0:
        raise ValueError("orc_scaled_bias_grads rejected the input")
    return db, ds


# ------------------------------------------------------------------- GEMMs
def fprop_entries(xq, xs, wq, ws, m_splits, rows, cols, bias=None):
    """xq (M,K) rowwise, xs compact; wq (E,N,K) rowwise, ws compact of (E*N,K)."""
    xq = _c(xq, np.uint8)
    M, K = xq.shape
    E, N, _ = wq.shape
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    val = np.empty(rows.size, np.float64)
    mag = np.empty(rows.size, np.float64)
    lib().orc_fprop_entries(_p(xq), _p(_c(xs, np.uint8)), _p(_c(wq, np.uint8)), _p(_c(ws, np.uint8)),
                            _p(None if bias is None else _c(bias, np.uint16)), M, N, K, E,
                            _p(_c(m_splits, np.int64)), rows.size, _p(rows), _p(cols), _p(val), _p(mag))
    return val, mag


def dgrad_entries(dyq, dys, wq_col, ws_col, m_splits, rows, cols):
    """dyq (M,N) rowwise; wq_col (E,N,K) colwise codes, ws_col compact colwise of (E*N,K)."""
    dyq = _c(dyq, np.uint8)
    M, N = dyq.shape
    E, _, K = wq_col.shape
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    val = np.empty(rows.size, np.float64)
    mag = np.empty(rows.size, np.float64)
    lib().orc_dgrad_entries(_p(dyq), _p(_c(dys, np.uint8)), _p(_c(wq_col, np.uint8)), _p(_c(ws_col, np.uint8)),
                            M, N, K, E, _p(_c(m_splits, np.int64)), rows.size, _p(rows), _p(cols),
                            _p(val), _p(mag))
    return val, mag


def wgrad_entries(dyq_col, dys_col, xq_col, xs_col, m_splits, experts, rows, cols):
    dyq_col = _c(dyq_col, np.uint8)
    M, N = dyq_col.shape
    K = xq_col.shape[1]
    E = len(m_splits)
    experts = _c(experts, np.int64)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    val = np.empty(rows.size, np.float64)
    mag = np.empty(rows.size, np.float64)
    lib().orc_wgrad_entries(_p(dyq_col), _p(_c(dys_col, np.uint8)), _p(_c(xq_col, np.uint8)),
                            _p(_c(xs_col, np.uint8)), M, N, K, E, _p(_c(m_splits, np.int64)), rows.size,
                            _p(experts), _p(rows), _p(cols), _p(val), _p(mag))
    return val, mag


def _all_entries(R, C):
    r, c = np.meshgrid(np.arange(R, dtype=np.int64), np.arange(C, dtype=np.int64), indexing="ij")
    return r.ravel(), c.ravel()


def fprop(xq, xs, wq, ws, m_splits, bias=None):
    M = xq.shape[0]
    N = wq.shape[1]
    r, c = _all_entries(M, N)
    v, a = fprop_entries(xq, xs, wq, ws, m_splits, r, c, bias)
    return v.reshape(M, N), a.reshape(M, N)


def dgrad(dyq, dys, wq_col, ws_col, m_splits):
    M = dyq.shape[0]
    K = wq_col.shape[2]
    r, c = _all_entries(M, K)
    v, a = dgrad_entries(dyq, dys, wq_col, ws_col, m_splits, r, c)
    return v.reshape(M, K), a.reshape(M, K)


def wgrad(dyq_col, dys_col, xq_col, xs_col, m_splits):
    N = dyq_col.shape[1]
    K = xq_col.shape[1]
    E = len(m_splits)
    e, n, k = np.meshgrid(np.arange(E), np.arange(N), np.arange(K), indexing="ij")
    v, a = wgrad_entries(dyq_col, dys_col, xq_col, xs_col, m_splits, e.ravel(), n.ravel(), k.ravel())
    return v.reshape(E, N, K), a.reshape(E, N, K)


# ------------------------------------------------------------------ SwiGLU
def swiglu_fwd(y_bits):
    y = _c(y_bits, np.uint16)
    M, F2 = y.shape
    h = np.zeros((M, F2 // 2), np.uint16)
    lib().orc_swiglu_fwd(_p(y), M, F2 // 2, _p(h))
    return h


def swiglu_bwd(dh_bits, y_bits):
    y = _c(y_bits, np.uint16)
    M, F2 = y.shape
    dy = np.zeros((M, F2), np.uint16)
    lib().orc_swiglu_bwd(_p(_c(dh_bits, np.uint16)), _p(y), M, F2 // 2, _p(dy))
    return dy


def num_threads() -> int:
    return lib().orc_num_threads()
