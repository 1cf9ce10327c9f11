"""Thin Python binding of libmxq.so (the C ABI in include/mxq.h).

Argument marshalling only: PyTorch supplies device memory and the current
CUDA stream; every step of the path runs in the library's CUDA kernels.
There is no fallback: if the library is missing or the device is not a
GB300 (sm_103), calls raise.

Tensors: activations/weights bf16; E4M3 data and E8M0 scales are uint8;
m_splits is a CUDA int64 tensor (host m_splits are rejected by the library).
"""
from __future__ import annotations

import ctypes
import functools
import os

import torch

from .build import LIB

ROWWISE, COLWISE, SWIZZLE, DEQUANT_OUT, ACCUMULATE, OUT_BF16, PAD_EXPERTS = 1, 2, 4, 8, 16, 32, 64
OP_GROUP_QUANTIZE, OP_REQUANT_COLWISE, OP_GROUPED_DBIAS = 1, 2, 3
OP_GEMM_FPROP, OP_GEMM_DGRAD, OP_GEMM_WGRAD, OP_SWIGLU_BWD_QUANTIZE, OP_SCALED_BIAS = 4, 5, 6, 7, 8
OP_GEMM_DGRAD_SWIGLU = 9
PROBE_ZEROS, PROBE_RANDOM = 0, 1
STATUS_SPLIT_UNALIGNED, STATUS_SPLIT_NEGATIVE, STATUS_SPLIT_SUM, STATUS_WAIT_TIMEOUT = 1, 2, 4, 8

SYMBOLS = [
    "mxq_version", "mxq_scale_bytes", "mxq_workspace_bytes", "mxq_group_quantize", "mxq_requant_colwise",
    "mxq_grouped_dbias", "mxq_grouped_gemm_fprop", "mxq_grouped_gemm_dgrad", "mxq_grouped_gemm_wgrad",
    "mxq_swiglu_fwd", "mxq_swiglu_bwd", "mxq_status_read", "mxq_error_string", "mxq_last_cuda_error",
    "mxq_grouped_dbias_noalloc", "mxq_swiglu_quantize", "mxq_swiglu_bwd_quantize", "mxq_group_quantize_scaled_bias",
    "mxq_requant_colwise_scaled_bias", "mxq_grouped_gemm_fprop_swiglu", "mxq_grouped_gemm_dgrad_swiglu",
    "mxq_scale_bytes_grouped", "mxq_grouped_gemm_fprop_ex", "mxq_grouped_gemm_dgrad_ex", "mxq_probe_mma_stream",
    "mxq_probe_mma_stream_ex", "mxq_selftest_wait_timeout",
]


class MXQError(RuntimeError):
    pass


_lib = None
_P, _I64, _INT, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t


def load(path: str = LIB) -> ctypes.CDLL:
    """Load libmxq.so and declare every exported symbol (no GPU needed)."""
    if not os.path.exists(path):
        raise MXQError(f"{path} is missing: build it with moe_expert_grouped_group_gb300.build.build()")
    L = ctypes.CDLL(path)
    L.mxq_version.restype = _INT
    L.mxq_scale_bytes.argtypes = [_I64, _I64, _INT]
    L.mxq_scale_bytes.restype = _SZ
    L.mxq_scale_bytes_grouped.argtypes = [_I64, _I64, _INT, _INT]
    L.mxq_scale_bytes_grouped.restype = _SZ
    L.mxq_workspace_bytes.argtypes = [_INT, _I64, _I64, _I64, _INT, _INT]
    L.mxq_workspace_bytes.restype = _SZ
    L.mxq_group_quantize.argtypes = [_P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.mxq_requant_colwise.argtypes = [_P, _P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_dbias.argtypes = [_P, _I64, _I64, _INT, _P, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_fprop.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_fprop_swiglu.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P,
                                                _P, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_dgrad_swiglu.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P,
                                                _P, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_fprop_ex.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_dgrad_ex.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_dgrad.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_gemm_wgrad.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _SZ, _P]
    L.mxq_grouped_dbias_noalloc.argtypes = [_P, _I64, _I64, _INT, _P, _P, _P, _P]
    L.mxq_grouped_dbias_noalloc.restype = _INT
    L.mxq_swiglu_fwd.argtypes = [_P, _I64, _I64, _P, _P]
    L.mxq_swiglu_quantize.argtypes = [_P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P, _P, _P, _P]
    L.mxq_swiglu_bwd_quantize.argtypes = [_P, _P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _SZ, _P]
    L.mxq_swiglu_bwd.argtypes = [_P, _P, _I64, _I64, _P, _P]
    L.mxq_group_quantize_scaled_bias.argtypes = [_P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P, _P, _P, _P,
                                                 _P, _P, _P, _SZ, _P]
    L.mxq_requant_colwise_scaled_bias.argtypes = [_P, _P, _I64, _I64, _INT, _P, _INT, _P, _P, _P, _P, _P, _P, _P,
                                                  _P, _P, _P, _P, _SZ, _P]
    L.mxq_status_read.argtypes = [_P, _P, _P]
    L.mxq_probe_mma_stream.argtypes = [_I64, _P, _P]
    L.mxq_probe_mma_stream.restype = _INT
    L.mxq_probe_mma_stream_ex.argtypes = [_I64, _INT, _P, _P]
    L.mxq_probe_mma_stream_ex.restype = _INT
    L.mxq_selftest_wait_timeout.argtypes = [_I64, _P, _P]
    L.mxq_selftest_wait_timeout.restype = _INT
    L.mxq_error_string.argtypes = [_INT]
    L.mxq_error_string.restype = ctypes.c_char_p
    L.mxq_last_cuda_error.restype = _INT
    for a in ("mxq_group_quantize", "mxq_requant_colwise", "mxq_grouped_dbias", "mxq_grouped_gemm_fprop",
              "mxq_grouped_gemm_dgrad", "mxq_grouped_gemm_wgrad", "mxq_swiglu_fwd", "mxq_swiglu_bwd",
              "mxq_status_read"):
        getattr(L, a).restype = _INT
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise MXQError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise MXQError("tensor arguments must be contiguous")
    return t.data_ptr()


# The current stream's raw handle without building a torch Stream object (about 3 us a call
# otherwise, as much as a small kernel); torch's public call where the fast one is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream():
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


_BF16 = (torch.bfloat16,)
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_BYTE = tuple(d for d in (torch.uint8, torch.int8, getattr(torch, "float8_e4m3fn", None),
                          getattr(torch, "float8_e8m0fnu", None)) if d is not None)


def _need(t, name, nbytes, dtypes):
    """The library takes raw pointers: check that a tensor the kernel reads or writes has the
    element type it expects and at least the bytes it touches (an undersized output would be
    written past its end). Outputs in the padded layouts are checked against the allocation bound
    (scale_bytes_grouped); padded inputs against the dense size, a lower bound of their exact size,
    which follows the device-resident expert counts."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype not in dtypes:
        raise MXQError(f"{name}: dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise MXQError(f"{name}: {have} bytes, the call touches {int(nbytes)}")


def _need_flags(noop, status):
    _need(noop, "noop", 4, _I32)
    _need(status, "status", 4, _I32)


def _check(rc: int, what: str):
    if rc != 0:
        L = lib()
        msg = L.mxq_error_string(rc).decode()
        cuda = L.mxq_last_cuda_error()
        raise MXQError(f"{what}: {msg} (code {rc}{', cuda error %d' % cuda if rc == -6 else ''})")


def _splits(m_splits):
    if m_splits is None:
        return None
    if not isinstance(m_splits, torch.Tensor) or not m_splits.is_cuda or m_splits.dtype != torch.int64:
        raise MXQError("m_splits must be a CUDA int64 tensor (host m_splits are rejected)")
    return m_splits


@functools.lru_cache(maxsize=4096)
def scale_bytes(rows: int, cols: int, colwise: bool) -> int:
    return int(lib().mxq_scale_bytes(rows, cols, int(colwise)))


@functools.lru_cache(maxsize=4096)
def scale_bytes_grouped(rows: int, cols: int, E: int, colwise: bool) -> int:
    """A scale-buffer size that holds the per-expert padded layout for any split of `rows`."""
    return int(lib().mxq_scale_bytes_grouped(rows, cols, E, int(colwise)))


@functools.lru_cache(maxsize=4096)
def workspace_bytes(op: int, M: int, N: int, K: int, E: int, flags: int = 0) -> int:
    return int(lib().mxq_workspace_bytes(op, M, N, K, E, flags))


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def status_read(status: torch.Tensor) -> int:
    out = ctypes.c_int32(0)
    _check(lib().mxq_status_read(_ptr(status), ctypes.byref(out), _stream()), "mxq_status_read")
    return int(out.value)


def _u8(n, dev):
    return torch.empty(n, dtype=torch.uint8, device=dev)


def _fill(o, key, make):
    """o[key] = make() unless the caller supplied it (setdefault with the default built only when needed:
    an eager default would allocate every output buffer on every call)."""
    if key not in o:
        o[key] = make()


def group_quantize(x, m_splits=None, E=None, rowwise=True, colwise=True, swizzle=True, dbias=False,
                   noop=None, status=None, out=None, workspace=None, pad_experts=False):
    """bf16 x (M, K) -> dict(row_data, row_scale, col_data, col_scale, dbias).
    pad_experts: expert counts need not be multiples of 128 (per-expert padded scale layouts)."""
    M, K = x.shape
    m_splits = _splits(m_splits)
    if E is None:
        if m_splits is None:
            raise MXQError("E is required for uniform members")
        E = m_splits.numel()
    dev = x.device
    flags = ((ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLE if swizzle else 0)
             | (PAD_EXPERTS if pad_experts else 0))
    o = dict(out or {})
    if rowwise:
        _fill(o, "row_data", lambda: _u8((M, K), dev))
        rs = scale_bytes_grouped(M, K, E, False) if (pad_experts and swizzle) else scale_bytes(M, K, False)
        _fill(o, "row_scale", lambda: _u8(rs, dev))
    if colwise:
        _fill(o, "col_data", lambda: _u8((M, K), dev))
        cs = scale_bytes_grouped(M, K, E, True) if pad_experts else scale_bytes(M, K, True)
        _fill(o, "col_scale", lambda: _u8(cs, dev))
    ws = None
    if dbias:
        _fill(o, "dbias", lambda: torch.empty((E, K), dtype=torch.float32, device=dev))
        ws = workspace if workspace is not None else _u8(
            max(16, workspace_bytes(OP_GROUP_QUANTIZE, M, 0, K, E, flags)), dev)
    _need(x, "x", M * K * 2, _BF16)
    _need(o.get("row_data"), "row_data", M * K, _BYTE)
    _need(o.get("row_scale"), "row_scale", rs if rowwise else 0, _BYTE)
    _need(o.get("col_data"), "col_data", M * K, _BYTE)
    _need(o.get("col_scale"), "col_scale",
          (scale_bytes_grouped(M, K, E, True) if pad_experts else scale_bytes(M, K, True)) if colwise else 0, _BYTE)
    _need(o.get("dbias"), "dbias", E * K * 4, _F32)
    _need_flags(noop, status)
    rc = lib().mxq_group_quantize(
        _ptr(x), M, K, E, _ptr(m_splits), flags, _ptr(o.get("row_data")), _ptr(o.get("row_scale")),
        _ptr(o.get("col_data")), _ptr(o.get("col_scale")), _ptr(o.get("dbias")), _ptr(noop), _ptr(status),
        _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream())
    _check(rc, "mxq_group_quantize")
    return o


def requant_colwise(row_data, row_scale_compact, m_splits, colwise=True, swizzle=True, row_scale_swizzled=True,
                    dbias=False, dequant=False, noop=None, status=None, out=None, workspace=None, pad_experts=False):
    """Rowwise E4M3 (M, K) + compact scales -> dict(col_data, col_scale, row_scale_swizzled, dbias, dequant).
    pad_experts: expert counts need not be multiples of 128 (per-expert padded scale layouts)."""
    M, K = row_data.shape
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    dev = row_data.device
    flags = ((COLWISE if colwise else 0) | (SWIZZLE if swizzle else 0) | (ROWWISE if row_scale_swizzled else 0)
             | (DEQUANT_OUT if dequant else 0) | (PAD_EXPERTS if pad_experts else 0))
    sb = (lambda r, c, cw: scale_bytes_grouped(r, c, E, cw)) if pad_experts else scale_bytes
    o = dict(out or {})
    if colwise:
        _fill(o, "col_data", lambda: _u8((M, K), dev))
        _fill(o, "col_scale", lambda: _u8(sb(M, K, True), dev))
    if row_scale_swizzled:
        _fill(o, "row_scale_swizzled", lambda: _u8(sb(M, K, False), dev))
    if dequant:
        _fill(o, "dequant", lambda: torch.empty((M, K), dtype=torch.bfloat16, device=dev))
    ws = None
    if dbias:
        _fill(o, "dbias", lambda: torch.empty((E, K), dtype=torch.float32, device=dev))
        ws = workspace if workspace is not None else _u8(
            max(16, workspace_bytes(OP_REQUANT_COLWISE, M, 0, K, E, flags)), dev)
    _need(row_data, "row_data", M * K, _BYTE)
    _need(row_scale_compact, "row_scale_compact", M * (K // 32), _BYTE)
    _need(o.get("col_data"), "col_data", M * K, _BYTE)
    _need(o.get("col_scale"), "col_scale", sb(M, K, True) if colwise else 0, _BYTE)
    _need(o.get("row_scale_swizzled"), "row_scale_swizzled", sb(M, K, False) if row_scale_swizzled else 0, _BYTE)
    _need(o.get("dequant"), "dequant", M * K * 2, _BF16)
    _need(o.get("dbias"), "dbias", E * K * 4, _F32)
    _need_flags(noop, status)
    rc = lib().mxq_requant_colwise(
        _ptr(row_data), _ptr(row_scale_compact), M, K, E, _ptr(m_splits), flags, _ptr(o.get("col_data")),
        _ptr(o.get("col_scale")), _ptr(o.get("row_scale_swizzled")), _ptr(o.get("dbias")), _ptr(o.get("dequant")),
        _ptr(noop), _ptr(status), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream())
    _check(rc, "mxq_requant_colwise")
    return o


def group_quantize_scaled_bias(x, m_splits, probs, bias, rowwise=True, colwise=True, swizzle=True, dbias=True,
                               dprobs=True, noop=None, status=None, out=None, workspace=None):
    """bf16 gradient x (M, K), routing scales probs (M,) fp32, expert biases bias (E, K) bf16 ->
    dict(row_data, row_scale, col_data, col_scale, dbias = sum s_m x_m per expert, dprobs = x_m . b_e)."""
    M, K = x.shape
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    dev = x.device
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLE if swizzle else 0)
    o = dict(out or {})
    if rowwise:
        _fill(o, "row_data", lambda: _u8((M, K), dev))
        _fill(o, "row_scale", lambda: _u8(scale_bytes(M, K, False), dev))
    if colwise:
        _fill(o, "col_data", lambda: _u8((M, K), dev))
        _fill(o, "col_scale", lambda: _u8(scale_bytes(M, K, True), dev))
    if dbias:
        _fill(o, "dbias", lambda: torch.empty((E, K), dtype=torch.float32, device=dev))
    if dprobs:
        _fill(o, "dprobs", lambda: torch.empty((M,), dtype=torch.float32, device=dev))
    ws = workspace if workspace is not None else _u8(max(16, workspace_bytes(OP_SCALED_BIAS, M, 0, K, E)), dev)
    _need(x, "x", M * K * 2, _BF16)
    _need(probs, "probs", M * 4, _F32)
    _need(bias, "bias", E * K * 2, _BF16)
    for k, n in (("row_data", M * K), ("row_scale", scale_bytes(M, K, False)), ("col_data", M * K),
                 ("col_scale", scale_bytes(M, K, True))):
        _need(o.get(k), k, n, _BYTE)
    _need(o.get("dbias"), "dbias", E * K * 4, _F32)
    _need(o.get("dprobs"), "dprobs", M * 4, _F32)
    _need_flags(noop, status)
    rc = lib().mxq_group_quantize_scaled_bias(
        _ptr(x), M, K, E, _ptr(m_splits), flags, _ptr(o.get("row_data")), _ptr(o.get("row_scale")),
        _ptr(o.get("col_data")), _ptr(o.get("col_scale")), _ptr(probs), _ptr(bias), _ptr(o.get("dbias")),
        _ptr(o.get("dprobs")), _ptr(noop), _ptr(status), _ptr(ws), ws.numel() * ws.element_size(), _stream())
    _check(rc, "mxq_group_quantize_scaled_bias")
    return o


def requant_colwise_scaled_bias(row_data, row_scale_compact, m_splits, probs, bias, colwise=True, swizzle=True,
                                row_scale_swizzled=True, dequant=False, dbias=True, dprobs=True, noop=None,
                                status=None, out=None, workspace=None):
    """Rowwise E4M3 gradient (M, K) + compact scales -> requant outputs as requant_colwise, plus the
    scaled-bias reductions of the dequantized values (dbias, dprobs) as group_quantize_scaled_bias."""
    M, K = row_data.shape
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    dev = row_data.device
    flags = ((COLWISE if colwise else 0) | (SWIZZLE if swizzle else 0) | (ROWWISE if row_scale_swizzled else 0)
             | (DEQUANT_OUT if dequant else 0))
    o = dict(out or {})
    if colwise:
        _fill(o, "col_data", lambda: _u8((M, K), dev))
        _fill(o, "col_scale", lambda: _u8(scale_bytes(M, K, True), dev))
    if row_scale_swizzled:
        _fill(o, "row_scale_swizzled", lambda: _u8(scale_bytes(M, K, False), dev))
    if dequant:
        _fill(o, "dequant", lambda: torch.empty((M, K), dtype=torch.bfloat16, device=dev))
    if dbias:
        _fill(o, "dbias", lambda: torch.empty((E, K), dtype=torch.float32, device=dev))
    if dprobs:
        _fill(o, "dprobs", lambda: torch.empty((M,), dtype=torch.float32, device=dev))
    ws = workspace if workspace is not None else _u8(max(16, workspace_bytes(OP_SCALED_BIAS, M, 0, K, E)), dev)
    _need(row_data, "row_data", M * K, _BYTE)
    _need(row_scale_compact, "row_scale_compact", M * (K // 32), _BYTE)
    _need(probs, "probs", M * 4, _F32)
    _need(bias, "bias", E * K * 2, _BF16)
    for k, n in (("col_data", M * K), ("col_scale", scale_bytes(M, K, True)),
                 ("row_scale_swizzled", scale_bytes(M, K, False))):
        _need(o.get(k), k, n, _BYTE)
    _need(o.get("dequant"), "dequant", M * K * 2, _BF16)
    _need(o.get("dbias"), "dbias", E * K * 4, _F32)
    _need(o.get("dprobs"), "dprobs", M * 4, _F32)
    _need_flags(noop, status)
    rc = lib().mxq_requant_colwise_scaled_bias(
        _ptr(row_data), _ptr(row_scale_compact), M, K, E, _ptr(m_splits), flags, _ptr(o.get("col_data")),
        _ptr(o.get("col_scale")), _ptr(o.get("row_scale_swizzled")), _ptr(probs), _ptr(bias), _ptr(o.get("dbias")),
        _ptr(o.get("dprobs")), _ptr(o.get("dequant")), _ptr(noop), _ptr(status), _ptr(ws),
        ws.numel() * ws.element_size(), _stream())
    _check(rc, "mxq_requant_colwise_scaled_bias")
    return o


def grouped_dbias(dy, m_splits, status=None, out=None, workspace=None):
    M, N = dy.shape
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    out = out if out is not None else torch.empty((E, N), dtype=torch.float32, device=dy.device)
    ws = workspace if workspace is not None else _u8(max(16, workspace_bytes(OP_GROUPED_DBIAS, M, N, 0, E)), dy.device)
    _need(dy, "dy", M * N * 2, _BF16)
    _need(out, "out", E * N * 4, _F32)
    _need_flags(None, status)
    rc = lib().mxq_grouped_dbias(_ptr(dy), M, N, E, _ptr(m_splits), _ptr(out), _ptr(status), _ptr(ws),
                                 ws.numel(), _stream())
    _check(rc, "mxq_grouped_dbias")
    return out


def grouped_gemm_fprop(x_data, x_scale, w_data, w_scale, m_splits, bias=None, status=None, out=None,
                       pad_experts=False):
    """Y = X W_e^T (+ b_e). x_data (M,K) u8, w_data (E,N,K) u8, swizzled scales.
    pad_experts: expert counts need not be multiples of 128 (x_scale in the padded layout)."""
    M, K = x_data.shape
    E, N, _ = w_data.shape
    m_splits = _splits(m_splits)
    out = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x_data.device)
    _need(x_data, "x_data", M * K, _BYTE)
    # padded inputs: the exact size follows the device-resident counts; the dense size is a lower bound
    _need(x_scale, "x_scale", scale_bytes(M, K, False), _BYTE)
    _need(w_data, "w_data", E * N * K, _BYTE)
    _need(w_scale, "w_scale", scale_bytes(E * N, K, False), _BYTE)
    _need(bias, "bias", E * N * 2, _BF16)
    _need(out, "out", M * N * 2, _BF16)
    _need_flags(None, status)
    rc = lib().mxq_grouped_gemm_fprop_ex(_ptr(x_data), _ptr(x_scale), _ptr(w_data), _ptr(w_scale), _ptr(bias), M, N,
                                         K, E, _ptr(m_splits), PAD_EXPERTS if pad_experts else 0, _ptr(out),
                                         _ptr(status), None, 0, _stream())
    _check(rc, "mxq_grouped_gemm_fprop_ex")
    return out


def grouped_gemm_fprop_swiglu(x_data, x_scale, w1_data, w1_scale, m_splits, bias=None, swizzle=True, status=None,
                              out=None, h_out=False):
    """FC1 of a SwiGLU MLP with the activation and its quantization in the GEMM epilogue.
    x_data (M, K) u8, w1_data (E, 2F, K) u8 ([gate | up] rows), swizzled scales ->
    dict(y1 (M, 2F) bf16, row_data, row_scale, col_data, col_scale of h (M, F)
    [, h (M, F) bf16: the values that were quantized, with h_out])."""
    M, K = x_data.shape
    E, N2, _ = w1_data.shape
    F = N2 // 2
    m_splits = _splits(m_splits)
    dev = x_data.device
    o = dict(out or {})
    _fill(o, "y1", lambda: torch.empty((M, 2 * F), dtype=torch.bfloat16, device=dev))
    _fill(o, "row_data", lambda: _u8((M, F), dev))
    _fill(o, "row_scale", lambda: _u8(scale_bytes(M, F, False), dev))
    _fill(o, "col_data", lambda: _u8((M, F), dev))
    _fill(o, "col_scale", lambda: _u8(scale_bytes(M, F, True), dev))
    if h_out:
        _fill(o, "h", lambda: torch.empty((M, F), dtype=torch.bfloat16, device=dev))
    _need(o.get("h"), "h", M * F * 2, _BF16)
    _need(x_data, "x_data", M * K, _BYTE)
    _need(x_scale, "x_scale", scale_bytes(M, K, False), _BYTE)
    _need(w1_data, "w1_data", E * 2 * F * K, _BYTE)
    _need(w1_scale, "w1_scale", scale_bytes(E * 2 * F, K, False), _BYTE)
    _need(bias, "bias", E * 2 * F * 2, _BF16)
    _need(o["y1"], "y1", M * 2 * F * 2, _BF16)
    for k, n in (("row_data", M * F), ("row_scale", scale_bytes(M, F, False)), ("col_data", M * F),
                 ("col_scale", scale_bytes(M, F, True))):
        _need(o[k], k, n, _BYTE)
    _need_flags(None, status)
    rc = lib().mxq_grouped_gemm_fprop_swiglu(
        _ptr(x_data), _ptr(x_scale), _ptr(w1_data), _ptr(w1_scale), _ptr(bias), M, K, F, E, _ptr(m_splits),
        (SWIZZLE if swizzle else 0) | (DEQUANT_OUT if "h" in o else 0), _ptr(o["y1"]), _ptr(o["row_data"]),
        _ptr(o["row_scale"]), _ptr(o["col_data"]), _ptr(o["col_scale"]), _ptr(o.get("h")), _ptr(status), None, 0,
        _stream())
    _check(rc, "mxq_grouped_gemm_fprop_swiglu")
    return o


def grouped_gemm_dgrad(dy_data, dy_scale, w_col_data, w_col_scale, m_splits, status=None, out=None,
                       pad_experts=False):
    """dX = dY W_e. dy_data (M,N) rowwise, w_col_data (E,N,K) colwise.
    pad_experts: expert counts need not be multiples of 128 (dy_scale in the padded layout)."""
    M, N = dy_data.shape
    E, _, K = w_col_data.shape
    m_splits = _splits(m_splits)
    out = out if out is not None else torch.empty((M, K), dtype=torch.bfloat16, device=dy_data.device)
    _need(dy_data, "dy_data", M * N, _BYTE)
    _need(dy_scale, "dy_scale", scale_bytes(M, N, False), _BYTE)  # padded: a lower bound, as in fprop
    _need(w_col_data, "w_col_data", E * N * K, _BYTE)
    _need(w_col_scale, "w_col_scale", scale_bytes(E * N, K, True), _BYTE)
    _need(out, "out", M * K * 2, _BF16)
    _need_flags(None, status)
    rc = lib().mxq_grouped_gemm_dgrad_ex(_ptr(dy_data), _ptr(dy_scale), _ptr(w_col_data), _ptr(w_col_scale), M, N,
                                         K, E, _ptr(m_splits), PAD_EXPERTS if pad_experts else 0, _ptr(out),
                                         _ptr(status), None, 0, _stream())
    _check(rc, "mxq_grouped_gemm_dgrad_ex")
    return out


def grouped_gemm_dgrad_swiglu(dy_data, dy_scale, w_col_data, w_col_scale, y1, m_splits, swizzle=True, dbias=True,
                              status=None, out=None, workspace=None, dy_out=False):
    """FC2 dgrad with the SwiGLU backward and the quantization of dY1 in the GEMM epilogue.
    dy_data (M, N) rowwise, w_col_data (E, N, F) colwise, y1 (M, 2F) bf16 saved FC1 output ->
    dict(row_data, row_scale, col_data, col_scale of dY1 (M, 2F), dbias (E, 2F)
    [, dy (M, 2F) bf16: the values that were quantized, with dy_out])."""
    M, N = dy_data.shape
    E, _, F = w_col_data.shape
    m_splits = _splits(m_splits)
    dev = dy_data.device
    o = dict(out or {})
    _fill(o, "row_data", lambda: _u8((M, 2 * F), dev))
    _fill(o, "row_scale", lambda: _u8(scale_bytes(M, 2 * F, False), dev))
    _fill(o, "col_data", lambda: _u8((M, 2 * F), dev))
    _fill(o, "col_scale", lambda: _u8(scale_bytes(M, 2 * F, True), dev))
    if dy_out:
        _fill(o, "dy", lambda: torch.empty((M, 2 * F), dtype=torch.bfloat16, device=dev))
    _need(o.get("dy"), "dy", M * 2 * F * 2, _BF16)
    ws = None
    if dbias:
        _fill(o, "dbias", lambda: torch.empty((E, 2 * F), dtype=torch.float32, device=dev))
        ws = workspace if workspace is not None else _u8(max(16, workspace_bytes(OP_GEMM_DGRAD_SWIGLU, M, N, F, E)),
                                                         dev)
    _need(dy_data, "dy_data", M * N, _BYTE)
    _need(dy_scale, "dy_scale", scale_bytes(M, N, False), _BYTE)
    _need(w_col_data, "w_col_data", E * N * F, _BYTE)
    _need(w_col_scale, "w_col_scale", scale_bytes(E * N, F, True), _BYTE)
    _need(y1, "y1", M * 2 * F * 2, _BF16)
    for k, n in (("row_data", M * 2 * F), ("row_scale", scale_bytes(M, 2 * F, False)), ("col_data", M * 2 * F),
                 ("col_scale", scale_bytes(M, 2 * F, True))):
        _need(o[k], k, n, _BYTE)
    _need(o.get("dbias"), "dbias", E * 2 * F * 4, _F32)
    _need_flags(None, status)
    rc = lib().mxq_grouped_gemm_dgrad_swiglu(
        _ptr(dy_data), _ptr(dy_scale), _ptr(w_col_data), _ptr(w_col_scale), _ptr(y1), M, N, F, E, _ptr(m_splits),
        (SWIZZLE if swizzle else 0) | (DEQUANT_OUT if "dy" in o else 0), _ptr(o["row_data"]), _ptr(o["row_scale"]),
        _ptr(o["col_data"]), _ptr(o["col_scale"]), _ptr(o.get("dbias")), _ptr(o.get("dy")), _ptr(status), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream())
    _check(rc, "mxq_grouped_gemm_dgrad_swiglu")
    return o


def grouped_gemm_wgrad(dy_col_data, dy_col_scale, x_col_data, x_col_scale, m_splits, accumulate=False,
                       out_bf16=False, status=None, out=None, pad_experts=False):
    """dW_e = dY_e^T X_e from the colwise copies; out (E, N, K) fp32 (or bf16).
    pad_experts: expert counts need not be multiples of 128 (colwise scales in the padded layout)."""
    M, N = dy_col_data.shape
    K = x_col_data.shape[1]
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    if out is None:
        out = torch.empty((E, N, K), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dy_col_data.device)
    flags = (ACCUMULATE if accumulate else 0) | (OUT_BF16 if out_bf16 else 0) | (PAD_EXPERTS if pad_experts else 0)
    _need(dy_col_data, "dy_col_data", M * N, _BYTE)
    _need(dy_col_scale, "dy_col_scale", scale_bytes(M, N, True), _BYTE)  # padded: a lower bound, as in fprop
    _need(x_col_data, "x_col_data", M * K, _BYTE)
    _need(x_col_scale, "x_col_scale", scale_bytes(M, K, True), _BYTE)
    _need(out, "out", E * N * K * (2 if out_bf16 else 4), _BF16 if out_bf16 else _F32)
    _need_flags(None, status)
    rc = lib().mxq_grouped_gemm_wgrad(_ptr(dy_col_data), _ptr(dy_col_scale), _ptr(x_col_data), _ptr(x_col_scale), M,
                                      N, K, E, _ptr(m_splits), flags, _ptr(out), _ptr(status), None, 0, _stream())
    _check(rc, "mxq_grouped_gemm_wgrad")
    return out


def probe_mma_stream(mmas_per_sm=8192, status=None, random=False):
    """Launch the tensor-pipe ceiling probe (not part of the MXFP8 path): one CTA per SM issues
    mmas_per_sm block-scaled 128x256x32 MMAs from resident shared memory, zero operands or (random)
    pseudo-random E4M3 ones. Returns its FLOPs (2*128*256*32*mmas_per_sm*SMs); time it with CUDA
    events on the current stream."""
    _need_flags(None, status)
    rc = lib().mxq_probe_mma_stream_ex(int(mmas_per_sm), PROBE_RANDOM if random else PROBE_ZEROS, _ptr(status),
                                       _stream())
    _check(rc, "mxq_probe_mma_stream_ex")
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 2.0 * 128 * 256 * 32 * mmas_per_sm * sms


def selftest_wait_timeout(status, limit_ns=20_000_000):
    """Make one bounded on-chip wait expire on purpose (an mbarrier nothing arrives on): sets
    STATUS_WAIT_TIMEOUT in `status` and returns, leaving the context usable."""
    _need_flags(None, status)
    _check(lib().mxq_selftest_wait_timeout(int(limit_ns), _ptr(status), _stream()), "mxq_selftest_wait_timeout")


def swiglu_fwd(y, out=None):
    M, F2 = y.shape
    out = out if out is not None else torch.empty((M, F2 // 2), dtype=torch.bfloat16, device=y.device)
    _need(y, "y", M * F2 * 2, _BF16)
    _need(out, "out", M * (F2 // 2) * 2, _BF16)
    _check(lib().mxq_swiglu_fwd(_ptr(y), M, F2 // 2, _ptr(out), _stream()), "mxq_swiglu_fwd")
    return out


def swiglu_bwd(dh, y, out=None):
    M, F2 = y.shape
    out = out if out is not None else torch.empty((M, F2), dtype=torch.bfloat16, device=y.device)
    _need(dh, "dh", M * (F2 // 2) * 2, _BF16)
    _need(y, "y", M * F2 * 2, _BF16)
    _need(out, "out", M * F2 * 2, _BF16)
    _check(lib().mxq_swiglu_bwd(_ptr(dh), _ptr(y), M, F2 // 2, _ptr(out), _stream()), "mxq_swiglu_bwd")
    return out


def _quant_outputs(o, M, K, rowwise, colwise, dev):
    if rowwise:
        _fill(o, "row_data", lambda: _u8((M, K), dev))
        _fill(o, "row_scale", lambda: _u8(scale_bytes(M, K, False), dev))
    if colwise:
        _fill(o, "col_data", lambda: _u8((M, K), dev))
        _fill(o, "col_scale", lambda: _u8(scale_bytes(M, K, True), dev))
    return o


def swiglu_quantize(y, m_splits, rowwise=True, colwise=True, swizzle=True, h_out=False, noop=None, status=None,
                    out=None):
    """SwiGLU forward fused with group_quantize: y (M, 2F) bf16 -> quantized h (M, F)
    (dict row_data/row_scale/col_data/col_scale, plus "h" in bf16 if h_out)."""
    M, F2 = y.shape
    F = F2 // 2
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    dev = y.device
    o = _quant_outputs(dict(out or {}), M, F, rowwise, colwise, dev)
    if h_out:
        _fill(o, "h", lambda: torch.empty((M, F), dtype=torch.bfloat16, device=dev))
    flags = ((ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLE if swizzle else 0)
             | (DEQUANT_OUT if h_out else 0))
    _need(y, "y", M * F2 * 2, _BF16)
    for k, n in (("row_data", M * F), ("row_scale", scale_bytes(M, F, False)), ("col_data", M * F),
                 ("col_scale", scale_bytes(M, F, True))):
        _need(o.get(k), k, n, _BYTE)
    _need(o.get("h"), "h", M * F * 2, _BF16)
    _need_flags(noop, status)
    rc = lib().mxq_swiglu_quantize(_ptr(y), M, F, E, _ptr(m_splits), flags, _ptr(o.get("row_data")),
                                   _ptr(o.get("row_scale")), _ptr(o.get("col_data")), _ptr(o.get("col_scale")),
                                   _ptr(o.get("h")), _ptr(noop), _ptr(status), _stream())
    _check(rc, "mxq_swiglu_quantize")
    return o


def swiglu_bwd_quantize(dh, y, m_splits, rowwise=True, colwise=True, swizzle=True, dbias=False, dy_out=False,
                        noop=None, status=None, out=None, workspace=None):
    """SwiGLU backward fused with group_quantize (+dbias): dh (M, F), y (M, 2F) ->
    quantized dY1 (M, 2F), optional "dbias" (E, 2F) fp32 and "dy" in bf16."""
    M, F2 = y.shape
    F = F2 // 2
    m_splits = _splits(m_splits)
    E = m_splits.numel()
    dev = y.device
    o = _quant_outputs(dict(out or {}), M, F2, rowwise, colwise, dev)
    if dy_out:
        _fill(o, "dy", lambda: torch.empty((M, F2), dtype=torch.bfloat16, device=dev))
    ws = None
    if dbias:
        _fill(o, "dbias", lambda: torch.empty((E, F2), dtype=torch.float32, device=dev))
        ws = workspace if workspace is not None else _u8(max(16, workspace_bytes(OP_SWIGLU_BWD_QUANTIZE, M, 0, F, E)),
                                                         dev)
    flags = ((ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLE if swizzle else 0)
             | (DEQUANT_OUT if dy_out else 0))
    _need(dh, "dh", M * F * 2, _BF16)
    _need(y, "y", M * F2 * 2, _BF16)
    for k, n in (("row_data", M * F2), ("row_scale", scale_bytes(M, F2, False)), ("col_data", M * F2),
                 ("col_scale", scale_bytes(M, F2, True))):
        _need(o.get(k), k, n, _BYTE)
    _need(o.get("dbias"), "dbias", E * F2 * 4, _F32)
    _need(o.get("dy"), "dy", M * F2 * 2, _BF16)
    _need_flags(noop, status)
    rc = lib().mxq_swiglu_bwd_quantize(_ptr(dh), _ptr(y), M, F, E, _ptr(m_splits), flags, _ptr(o.get("row_data")),
                                       _ptr(o.get("row_scale")), _ptr(o.get("col_data")), _ptr(o.get("col_scale")),
                                       _ptr(o.get("dbias")), _ptr(o.get("dy")), _ptr(noop), _ptr(status), _ptr(ws),
                                       0 if ws is None else ws.numel() * ws.element_size(), _stream())
    _check(rc, "mxq_swiglu_bwd_quantize")
    return o
