"""Python binding of libmxq (MX block-scaled quantization and MXFP8 GEMMs for GB300).

Argument marshalling only: every function named ``mxq_*`` here has the name,
arguments and meaning of the C entry point declared in ``include/mxq.h`` and
forwards to it through ctypes.  Tensor arguments are torch CUDA tensors (or raw
device addresses as ints); ``stream`` defaults to torch's current stream.  A
non-OK status raises :class:`MXQError` with the library's reason.

The compute path is the CUDA library only: if ``libmxq.so`` cannot be built or
loaded, every call raises -- there is no fallback.  With the environment
variable ``MXQ_LIBRARY=debug`` the debug build ``libmxq_debug.so`` (bounds
checks on every computed global access) is loaded instead.

The ``alloc_*`` / ``quantize_*`` helpers at the bottom only size and allocate
output tensors with the library's own size queries, then call the entry points.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "MXQError", "load", "BF16", "F32", "E4M3", "E2M1", "SAVE_QUANT", "RECOMPUTE", "GG_FWD", "GG_DX", "GG_DW",
    "mxq_scale_bytes", "mxq_grouped_padded_rows", "mxq_quantize", "mxq_quantize_grouped_col",
    "mxq_quantize_grouped_dual", "mxq_quantize_grouped_dual_padded", "mxq_qdq_mxfp4",
    "mxq_gemm", "mxq_grouped_gemm", "mxq_linear_ctx_bytes", "mxq_linear_saved_bytes",
    "mxq_linear_workspace_bytes", "mxq_linear_fwd", "mxq_linear_bwd_dx", "mxq_linear_bwd_dw",
    "mxq_last_error_string", "mxq_poll_device_error", "mxq_linear_fwd_noalloc", "NOALLOC_SCRATCH_BYTES",
    "mxq_mxfp4_ste_forward", "mxq_mxfp4_ste_backward", "mxfp4_ste_forward", "mxfp4_ste_backward",
    "mxq_qat_linear_workspace_bytes", "mxq_qat_linear_fwd", "qat_linear_fwd",
    "mxq_qat_grouped_fwd_workspace_bytes", "mxq_qat_grouped_fwd", "qat_grouped_fwd",
    "mxq_grouped_linear_ctx_bytes", "mxq_grouped_linear_saved_bytes", "mxq_grouped_linear_workspace_bytes",
    "mxq_grouped_linear_fwd", "mxq_grouped_linear_bwd_dx", "mxq_grouped_linear_bwd_dw", "mxq_qdq_mxfp4_bf16",
    "mxq_linear_weight_cache_bytes", "mxq_linear_wq_ctx_bytes", "mxq_linear_quantize_weight", "mxq_linear_fwd_wq",
    "mxq_linear_bwd_dx_wq", "mxq_selftest_wait_timeout", "mxq_validate_group_offsets", "mxq_check_group_offsets",
]

BF16, F32 = 0, 1
E4M3, E2M1 = 0, 1
SAVE_QUANT, RECOMPUTE = 0, 1
GG_FWD, GG_DX, GG_DW = 0, 1, 2
NOALLOC_SCRATCH_BYTES = 64 << 20  # MXQ_NOALLOC_SCRATCH_BYTES in include/mxq.h
_STATUS = {0: "MXQ_OK", 1: "MXQ_ERR_INVALID_ARG", 2: "MXQ_ERR_UNSUPPORTED", 3: "MXQ_ERR_ARCH",
           4: "MXQ_ERR_CUDA", 5: "MXQ_ERR_TIMEOUT"}


class MXQError(RuntimeError):
    def __init__(self, msg: str, status: int):
        super().__init__(msg)
        self.status = status


_lib = None

_I64, _I32, _P, _SZ, _F32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
_SIGNATURES = {
    "mxq_scale_bytes": (_SZ, [_I64, _I64]),
    "mxq_grouped_padded_rows": (_I64, [_I64, _I32]),
    "mxq_quantize": (_I32, [_P, _I32, _I64, _I64, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "mxq_quantize_grouped_col": (_I32, [_P, _I64, _I64, _P, _I32, _I64, _P, _P, _P]),
    "mxq_quantize_grouped_dual": (_I32, [_P, _I64, _I64, _P, _I32, _I64, _P, _P, _P, _P, _P]),
    "mxq_quantize_grouped_dual_padded": (_I32, [_P, _I64, _I64, _P, _I32, _I64, _P, _P, _P, _P, _P]),
    "mxq_qdq_mxfp4": (_I32, [_P, _P, _I64, _I64, _I32, _F32, _P]),
    "mxq_qdq_mxfp4_bf16": (_I32, [_P, _P, _I64, _I64, _I32, _F32, _P]),
    "mxq_mxfp4_ste_forward": (_I32, [_P, _P, _P, _I64, _I64, _I32, _F32, _P]),
    "mxq_mxfp4_ste_backward": (_I32, [_P, _P, _I64, _I64, _P, _P]),
    "mxq_qat_linear_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "mxq_qat_linear_fwd": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I32, _F32, _P, _P, _SZ, _P]),
    "mxq_qat_grouped_fwd_workspace_bytes": (_SZ, [_I64, _I32, _I64, _I64, _I32]),
    "mxq_grouped_linear_ctx_bytes": (_SZ, [_I64, _I32, _I64, _I64, _I32]),
    "mxq_grouped_linear_saved_bytes": (_SZ, [_I64, _I32, _I64, _I64, _I32]),
    "mxq_grouped_linear_workspace_bytes": (_SZ, [_I64, _I32, _I64, _I64, _I32]),
    "mxq_grouped_linear_fwd": (_I32, [_P, _P, _P, _I32, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_grouped_linear_bwd_dx": (_I32, [_P, _P, _P, _I32, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_grouped_linear_bwd_dw": (_I32, [_P, _P, _P, _I32, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_qat_grouped_fwd": (_I32, [_P, _P, _P, _I32, _I64, _I64, _I64, _I32, _F32, _P, _P, _SZ, _P]),
    "mxq_gemm": (_I32, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P]),
    "mxq_grouped_gemm": (_I32, [_I32, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _I64, _P, _P]),
    "mxq_linear_ctx_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "mxq_linear_saved_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "mxq_linear_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "mxq_linear_fwd": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_linear_bwd_dx": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_linear_bwd_dw": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_linear_fwd_noalloc": (_I32, [_P, _P, _I64, _I64, _I64, _P, _P]),
    "mxq_linear_weight_cache_bytes": (_SZ, [_I64, _I64]),
    "mxq_linear_wq_ctx_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "mxq_linear_quantize_weight": (_I32, [_P, _I64, _I64, _P, _SZ, _P]),
    "mxq_linear_fwd_wq": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_linear_bwd_dx_wq": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "mxq_last_error_string": (ctypes.c_char_p, []),
    "mxq_poll_device_error": (_I32, [ctypes.POINTER(ctypes.c_uint32)]),
    "mxq_selftest_wait_timeout": (_I32, [ctypes.c_uint32, _P, _P]),
    "mxq_validate_group_offsets": (_I32, [_P, _I32, _I64]),
    "mxq_check_group_offsets": (_I32, [_P, _I32, _I64, _P]),
}


def _debug_requested() -> bool:
    import os
    return os.environ.get("MXQ_LIBRARY", "") == "debug"


def library_path() -> str:
    return _build.DEBUG_LIB if _debug_requested() else _build.LIB


def load(build_if_needed: bool = True):
    """Load libmxq.so (compiling it in-tree first if it is missing or stale);
    libmxq_debug.so under MXQ_LIBRARY=debug."""
    global _lib
    if _lib is None:
        debug = _debug_requested()
        if not _build.up_to_date(debug):
            if not build_if_needed:
                raise MXQError(f"libmxq is not built at {library_path()}", -1)
            _build.build(debug=debug)
        lib = ctypes.CDLL(library_path())
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _s(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, name: str) -> None:
    if status != 0:
        reason = _lib.mxq_last_error_string().decode(errors="replace")
        raise MXQError(f"{name}: {_STATUS.get(status, status)}: {reason}", status)


# ---------------------------------------------------------------- entry points

def mxq_scale_bytes(rows: int, k_blocks: int) -> int:
    return int(load().mxq_scale_bytes(rows, k_blocks))


def mxq_grouped_padded_rows(T: int, E: int) -> int:
    return int(load().mxq_grouped_padded_rows(T, E))


def mxq_quantize(x, dtype, rows, cols, ldx, axis, fmt, dual_axis, q_row, s_row, q_colT, s_colT, stream=None):
    _check(load().mxq_quantize(_p(x), dtype, rows, cols, ldx, axis, fmt, int(dual_axis), _p(q_row), _p(s_row),
                               _p(q_colT), _p(s_colT), _s(stream)), "mxq_quantize")


def mxq_quantize_grouped_col(x, rows, cols, d_offsets, E, t_pad, q_colT, s_colT, stream=None):
    _check(load().mxq_quantize_grouped_col(_p(x), rows, cols, _p(d_offsets), E, t_pad, _p(q_colT), _p(s_colT),
                                           _s(stream)), "mxq_quantize_grouped_col")


def mxq_quantize_grouped_dual(x, rows, cols, d_offsets, E, t_pad, q_row, s_row, q_colT, s_colT, stream=None):
    _check(load().mxq_quantize_grouped_dual(_p(x), rows, cols, _p(d_offsets), E, t_pad, _p(q_row), _p(s_row),
                                            _p(q_colT), _p(s_colT), _s(stream)), "mxq_quantize_grouped_dual")


def mxq_quantize_grouped_dual_padded(x, rows, cols, d_offsets, E, t_pad, q_row, s_row, q_colT, s_colT,
                                     stream=None):
    _check(load().mxq_quantize_grouped_dual_padded(_p(x), rows, cols, _p(d_offsets), E, t_pad, _p(q_row),
                                                   _p(s_row), _p(q_colT), _p(s_colT), _s(stream)),
           "mxq_quantize_grouped_dual_padded")


def mxq_qdq_mxfp4(x, y, rows, cols, block_size=32, scale_factor=6.0, stream=None):
    _check(load().mxq_qdq_mxfp4(_p(x), _p(y), rows, cols, block_size, scale_factor, _s(stream)), "mxq_qdq_mxfp4")


def mxq_qdq_mxfp4_bf16(x, y, rows, cols, block_size=32, scale_factor=6.0, stream=None):
    _check(load().mxq_qdq_mxfp4_bf16(_p(x), _p(y), rows, cols, block_size, scale_factor, _s(stream)),
           "mxq_qdq_mxfp4_bf16")


def mxq_mxfp4_ste_forward(x, y, sat_mask, rows, cols, block_size=32, scale_factor=6.0, stream=None):
    _check(load().mxq_mxfp4_ste_forward(_p(x), _p(y), _p(sat_mask), rows, cols, block_size, scale_factor,
                                        _s(stream)), "mxq_mxfp4_ste_forward")


def mxq_mxfp4_ste_backward(grad_y, sat_mask, rows, cols, grad_x, stream=None):
    _check(load().mxq_mxfp4_ste_backward(_p(grad_y), _p(sat_mask), rows, cols, _p(grad_x), _s(stream)),
           "mxq_mxfp4_ste_backward")


def mxq_gemm(a, sa, b, sb, M, N, K, c, ldc, stream=None):
    _check(load().mxq_gemm(_p(a), _p(sa), _p(b), _p(sb), M, N, K, _p(c), ldc, _s(stream)), "mxq_gemm")


def mxq_grouped_gemm(kind, a, sa, b, sb, d_offsets, E, T, N, K, t_pad, out, stream=None):
    _check(load().mxq_grouped_gemm(kind, _p(a), _p(sa), _p(b), _p(sb), _p(d_offsets), E, T, N, K, t_pad, _p(out),
                                   _s(stream)), "mxq_grouped_gemm")


def mxq_linear_ctx_bytes(M, N, K, mode) -> int:
    return int(load().mxq_linear_ctx_bytes(M, N, K, mode))


def mxq_linear_saved_bytes(M, N, K, mode) -> int:
    return int(load().mxq_linear_saved_bytes(M, N, K, mode))


def mxq_linear_workspace_bytes(M, N, K, mode) -> int:
    return int(load().mxq_linear_workspace_bytes(M, N, K, mode))


def mxq_linear_fwd(x, w, M, N, K, mode, ctx, y, workspace, ws_bytes, stream=None):
    _check(load().mxq_linear_fwd(_p(x), _p(w), M, N, K, mode, _p(ctx), _p(y), _p(workspace), ws_bytes, _s(stream)),
           "mxq_linear_fwd")


def mxq_linear_bwd_dx(dy, w, M, N, K, mode, ctx, dx, workspace, ws_bytes, stream=None):
    _check(load().mxq_linear_bwd_dx(_p(dy), _p(w), M, N, K, mode, _p(ctx), _p(dx), _p(workspace), ws_bytes,
                                    _s(stream)), "mxq_linear_bwd_dx")


def mxq_linear_bwd_dw(dy, x, M, N, K, mode, ctx, dw, workspace, ws_bytes, stream=None):
    _check(load().mxq_linear_bwd_dw(_p(dy), _p(x), M, N, K, mode, _p(ctx), _p(dw), _p(workspace), ws_bytes,
                                    _s(stream)), "mxq_linear_bwd_dw")


def mxq_linear_weight_cache_bytes(N, K) -> int:
    return load().mxq_linear_weight_cache_bytes(N, K)


def mxq_linear_wq_ctx_bytes(M, N, K, mode) -> int:
    return load().mxq_linear_wq_ctx_bytes(M, N, K, mode)


def mxq_linear_quantize_weight(w, N, K, wcache, cache_bytes, stream=None):
    _check(load().mxq_linear_quantize_weight(_p(w), N, K, _p(wcache), cache_bytes, _s(stream)),
           "mxq_linear_quantize_weight")


def mxq_linear_fwd_wq(x, wcache, M, N, K, mode, ctx, y, workspace, ws_bytes, stream=None):
    _check(load().mxq_linear_fwd_wq(_p(x), _p(wcache), M, N, K, mode, _p(ctx), _p(y), _p(workspace), ws_bytes,
                                    _s(stream)), "mxq_linear_fwd_wq")


def mxq_linear_bwd_dx_wq(dy, wcache, M, N, K, mode, ctx, dx, workspace, ws_bytes, stream=None):
    _check(load().mxq_linear_bwd_dx_wq(_p(dy), _p(wcache), M, N, K, mode, _p(ctx), _p(dx), _p(workspace), ws_bytes,
                                       _s(stream)), "mxq_linear_bwd_dx_wq")


def mxq_linear_fwd_noalloc(x, w, M, N, K, y, stream=None):
    """Linear forward that allocates nothing: its scratch is a fixed array inside
    the library (for callers that may not allocate device memory)."""
    _check(load().mxq_linear_fwd_noalloc(_p(x), _p(w), M, N, K, _p(y), _s(stream)), "mxq_linear_fwd_noalloc")


def mxq_last_error_string() -> str:
    return load().mxq_last_error_string().decode(errors="replace")


def mxq_selftest_wait_timeout(timeout_ms, d_gave_up, stream=None):
    _check(load().mxq_selftest_wait_timeout(timeout_ms, _p(d_gave_up), _s(stream)), "mxq_selftest_wait_timeout")


def mxq_poll_device_error():
    """Returns the device error bits (0 = none; bit 2 = malformed group
    offsets; bit 3 = an access outside its buffer, found by the debug build);
    raises on a CUDA failure."""
    w = ctypes.c_uint32(0)
    st = load().mxq_poll_device_error(ctypes.byref(w))
    if w.value == 0 and st != 0:
        _check(st, "mxq_poll_device_error")
    return int(w.value)


def mxq_validate_group_offsets(offsets, E, T):
    """Host-side check of group offsets (a host int64 array of E+1 values);
    raises MXQError (MXQ_ERR_INVALID_ARG) with the first violation."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    if a.size < E + 1:
        raise ValueError("offsets holds fewer than E+1 values")
    _check(load().mxq_validate_group_offsets(a.ctypes.data, E, T), "mxq_validate_group_offsets")


def mxq_check_group_offsets(d_offsets, E, T, stream=None):
    _check(load().mxq_check_group_offsets(_p(d_offsets), E, T, _s(stream)), "mxq_check_group_offsets")


# ---------------------------------------------------------------- allocation helpers

def _u8(n: int, device) -> torch.Tensor:
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def quantize_mxfp8(x: torch.Tensor, axis: int = -1, dual: bool = False, stream=None):
    """MXFP8 quant of a 2-D bf16 CUDA tensor.  Returns (q_row, s_row, q_colT,
    s_colT) with None for the axis not requested; scales in swz layout."""
    R, C = x.shape
    q_row = s_row = qT = sT = None
    if dual or axis == -1:
        q_row = torch.empty((R, C), dtype=torch.uint8, device=x.device)
        s_row = _u8(mxq_scale_bytes(R, C // 32), x.device)
    if dual or axis == -2:
        qT = torch.empty((C, R), dtype=torch.uint8, device=x.device)
        sT = _u8(mxq_scale_bytes(C, (R + 31) // 32), x.device)
    mxq_quantize(x, BF16, R, C, x.stride(0), axis, E4M3, dual, q_row, s_row, qT, sT, stream)
    return q_row, s_row, qT, sT


def quantize_mxfp4(x: torch.Tensor, stream=None):
    """Packed MXFP4 quant (scale_factor 6) of a 2-D bf16/fp32 CUDA tensor:
    returns (nibbles [R x C/2], scales swz(R, C/32))."""
    R, C = x.shape
    q = torch.empty((R, C // 2), dtype=torch.uint8, device=x.device)
    s = _u8(mxq_scale_bytes(R, C // 32), x.device)
    mxq_quantize(x, F32 if x.dtype == torch.float32 else BF16, R, C, x.stride(0), -1, E2M1, 0, q, s, None, None,
                 stream)
    return q, s


def mxq_qat_linear_workspace_bytes(M, N, K, quantize_input=1):
    return load().mxq_qat_linear_workspace_bytes(M, N, K, quantize_input)


def mxq_qat_linear_fwd(x, w, bias, M, N, K, quantize_input, scale_factor, y, workspace, ws_bytes, stream=None):
    _check(load().mxq_qat_linear_fwd(_p(x), _p(w), _p(bias), M, N, K, quantize_input, scale_factor, _p(y),
                                     _p(workspace), ws_bytes, _s(stream)), "mxq_qat_linear_fwd")


def qat_linear_fwd(x: torch.Tensor, w: torch.Tensor, bias=None, quantize_input: bool = True,
                   scale_factor: float = 6.0, stream=None) -> torch.Tensor:
    """MXFP4 QAT linear forward of contiguous bf16 CUDA tensors x [M x K],
    w [N x K], bias [N] or None: returns bf16 [M x N]."""
    M, K = x.shape
    N = w.shape[0]
    ws_bytes = mxq_qat_linear_workspace_bytes(M, N, K, int(quantize_input))
    ws = _u8(ws_bytes, x.device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    mxq_qat_linear_fwd(x, w, bias, M, N, K, int(quantize_input), scale_factor, y, ws, ws_bytes, stream)
    return y


def mxq_grouped_linear_ctx_bytes(T, E, N, K, mode):
    return load().mxq_grouped_linear_ctx_bytes(T, E, N, K, mode)


def mxq_grouped_linear_saved_bytes(T, E, N, K, mode):
    return load().mxq_grouped_linear_saved_bytes(T, E, N, K, mode)


def mxq_grouped_linear_workspace_bytes(T, E, N, K, mode):
    return load().mxq_grouped_linear_workspace_bytes(T, E, N, K, mode)


def mxq_grouped_linear_fwd(x, w, d_offsets, E, T, N, K, mode, ctx, y, workspace, ws_bytes, stream=None):
    _check(load().mxq_grouped_linear_fwd(_p(x), _p(w), _p(d_offsets), E, T, N, K, mode, _p(ctx), _p(y),
                                         _p(workspace), ws_bytes, _s(stream)), "mxq_grouped_linear_fwd")


def mxq_grouped_linear_bwd_dx(dy, w, d_offsets, E, T, N, K, mode, ctx, dx, workspace, ws_bytes, stream=None):
    _check(load().mxq_grouped_linear_bwd_dx(_p(dy), _p(w), _p(d_offsets), E, T, N, K, mode, _p(ctx), _p(dx),
                                            _p(workspace), ws_bytes, _s(stream)), "mxq_grouped_linear_bwd_dx")


def mxq_grouped_linear_bwd_dw(dy, x, d_offsets, E, T, N, K, mode, ctx, dw, workspace, ws_bytes, stream=None):
    _check(load().mxq_grouped_linear_bwd_dw(_p(dy), _p(x), _p(d_offsets), E, T, N, K, mode, _p(ctx), _p(dw),
                                            _p(workspace), ws_bytes, _s(stream)), "mxq_grouped_linear_bwd_dw")


def mxq_qat_grouped_fwd_workspace_bytes(T, E, N, K, quantize_input=1):
    return load().mxq_qat_grouped_fwd_workspace_bytes(T, E, N, K, quantize_input)


def mxq_qat_grouped_fwd(x, w, d_offsets, E, T, N, K, quantize_input, scale_factor, y, workspace, ws_bytes,
                        stream=None):
    _check(load().mxq_qat_grouped_fwd(_p(x), _p(w), _p(d_offsets), E, T, N, K, quantize_input, scale_factor, _p(y),
                                      _p(workspace), ws_bytes, _s(stream)), "mxq_qat_grouped_fwd")


def qat_grouped_fwd(x: torch.Tensor, w: torch.Tensor, d_offsets: torch.Tensor, quantize_input: bool = True,
                    scale_factor: float = 6.0, stream=None) -> torch.Tensor:
    """MXFP4 QAT forward of an MoE expert layer: x bf16 [T x K] routed rows,
    w bf16 [E x N x K], d_offsets int64 [E+1] on the device: returns bf16
    [T x N]."""
    T, K = x.shape
    E, N = w.shape[0], w.shape[1]
    ws_bytes = mxq_qat_grouped_fwd_workspace_bytes(T, E, N, K, int(quantize_input))
    ws = _u8(max(ws_bytes, 1), x.device)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    mxq_qat_grouped_fwd(x, w, d_offsets, E, T, N, K, int(quantize_input), scale_factor, y, ws, ws_bytes, stream)
    return y


def mxfp4_ste_forward(x: torch.Tensor, scale_factor: float = 6.0, stream=None):
    """Clipped-STE forward of a contiguous fp32 CUDA tensor: returns (y, sat_mask)
    with sat_mask int32 [rows x ceil(cols/32)] holding the packed mask words."""
    assert x.dtype == torch.float32 and x.is_contiguous()
    y = torch.empty_like(x)
    cols = x.shape[-1] if x.dim() else 1
    rows = x.numel() // cols if cols else 0
    m = torch.empty((rows, (cols + 31) // 32), dtype=torch.int32, device=x.device)
    mxq_mxfp4_ste_forward(x, y, m, rows, cols, 32, scale_factor, stream)
    return y, m


def mxfp4_ste_backward(grad_y: torch.Tensor, sat_mask: torch.Tensor, stream=None) -> torch.Tensor:
    """Clipped-STE backward: grad_y with the saturated elements set to +0.0."""
    assert grad_y.dtype == torch.float32 and grad_y.is_contiguous() and sat_mask.is_contiguous()
    gx = torch.empty_like(grad_y)
    cols = grad_y.shape[-1] if grad_y.dim() else 1
    rows = grad_y.numel() // cols if cols else 0
    assert tuple(sat_mask.shape) == (rows, (cols + 31) // 32)
    mxq_mxfp4_ste_backward(grad_y, sat_mask, rows, cols, gx, stream)
    return gx


def qdq_mxfp4(x: torch.Tensor, scale_factor: float = 6.0, stream=None) -> torch.Tensor:
    """MXFP4 quant-dequant of a contiguous fp32 or bf16 CUDA tensor (blocks
    along the last dim); the result has x's dtype."""
    assert x.dtype in (torch.float32, torch.bfloat16) and x.is_contiguous()
    y = torch.empty_like(x)
    cols = x.shape[-1] if x.dim() else 1
    rows = x.numel() // cols if cols else 0
    if x.dtype == torch.bfloat16:
        mxq_qdq_mxfp4_bf16(x, y, rows, cols, 32, scale_factor, stream)
    else:
        mxq_qdq_mxfp4(x, y, rows, cols, 32, scale_factor, stream)
    return y
