"""CPU oracle for MX block-scaled quantization and block-scaled GEMMs.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``mx_block_scaled_mxq_gb300``) never imports it,
and the two share no code.

Element-wise quantization is plain C (``mxq_oracle.c``, compiled with gcc and
loaded with ctypes); the GEMM references are numpy binary64 products of the
exactly dequantized operands (``gemm.py``).  Inputs are numpy arrays; bf16
tensors are passed as their uint16 bit patterns.

Every function cites the passage it follows in its docstring; the readings
taken where the pages are silent are listed at the top of ``mxq_oracle.c``.
All functions here are pinned by ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_mxq.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into ``oracle/liboracle_mxq.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p, f64, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_float
        lib.oracle_e4m3_encode.argtypes = [f64]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = f64
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = f64
        lib.oracle_mxfp8_scale_exp.argtypes = [f64]
        lib.oracle_mxfp8_scale_exp.restype = ctypes.c_int
        lib.oracle_mxfp4_scale_exp.argtypes = [f64, f64]
        lib.oracle_mxfp4_scale_exp.restype = ctypes.c_int
        lib.oracle_mxfp8_quant_rows.argtypes = [p, i64, i64, i64, p, i64, p, i64]
        lib.oracle_mxfp8_quant_cols.argtypes = [p, i64, i64, i64, p, i64, p, i64]
        lib.oracle_mxfp8_quant_cols_grouped.argtypes = [p, i64, i64, p, ctypes.c_int, p, i64, p, i64]
        lib.oracle_swizzle_scales.argtypes = [p, i64, i64, i64, p]
        lib.oracle_mxfp4_qdq.argtypes = [p, p, i64, i64, f32]
        lib.oracle_mxfp4_quant.argtypes = [p, i64, i64, i64, f32, p, i64, p, i64]
        lib.oracle_mxfp4_saturation_mask.argtypes = [p, i64, i64, f32, p]
        lib.oracle_mxfp4_ste_backward.argtypes = [p, p, i64, i64, p]
        for name in ("oracle_mxfp8_quant_rows", "oracle_mxfp8_quant_cols",
                     "oracle_mxfp8_quant_cols_grouped", "oracle_swizzle_scales",
                     "oracle_mxfp4_qdq", "oracle_mxfp4_quant", "oracle_mxfp4_saturation_mask",
                     "oracle_mxfp4_ste_backward"):
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # local: torch is only used to reinterpret the bits
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ---------------------------------------------------------------------------
# scalar rules
# ---------------------------------------------------------------------------

def e4m3_encode(y: float) -> int:
    """E4M3 code of an exact value, round-to-nearest-even, saturating to +-448."""
    return int(_load().oracle_e4m3_encode(float(y)))


def e4m3_decode_table() -> np.ndarray:
    """binary64 value of each of the 256 E4M3 codes (NaN for 0x7F / 0xFF)."""
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e2m1_decode_table() -> np.ndarray:
    """binary64 value of each of the 16 E2M1 nibbles (codebook of the AMCT
    FakeQuant article, section 2)."""
    lib = _load()
    return np.array([lib.oracle_e2m1_decode(c) for c in range(16)], dtype=np.float64)


def mxfp8_scale_exp(amax: float) -> int:
    """OCP MX scale exponent floor(log2 amax) - 8, clamped to [-127, 127]."""
    return int(_load().oracle_mxfp8_scale_exp(float(amax)))


def mxfp4_scale_exp(amax: float, sf: float = 6.0) -> int:
    """round(log2(max(amax/sf, 2^-30))) exactly (AMCT FakeQuant article, section 2)."""
    return int(_load().oracle_mxfp4_scale_exp(float(amax), float(sf)))


# ---------------------------------------------------------------------------
# tensor quantizers (logical, row-major scale matrices)
# ---------------------------------------------------------------------------

def mxfp8_quant_rows(x):
    """Row MXFP8 quant of bf16 A[R x C] (blocks of 32 along C; torchtitan-npu
    feature guide, MXFP8 mode).  Returns (codes u8 [R x C], scales u8
    [R x ceil(C/32)])."""
    xb = _bf16_bits(x)
    R, C = xb.shape
    nb = (C + 31) // 32
    q = np.zeros((R, C), np.uint8)
    s = np.zeros((R, nb), np.uint8)
    if R and C:
        _load().oracle_mxfp8_quant_rows(_ptr(xb), R, C, C, _ptr(q), C, _ptr(s), nb)
    return q, s


def mxfp8_quant_cols(x):
    """Column MXFP8 quant of bf16 A[R x C] (blocks of 32 along R).  Returns
    (transposed codes u8 [C x R], scales u8 [C x ceil(R/32)])."""
    xb = _bf16_bits(x)
    R, C = xb.shape
    nb = (R + 31) // 32
    qT = np.zeros((C, R), np.uint8)
    s = np.zeros((C, nb), np.uint8)
    if R and C:
        _load().oracle_mxfp8_quant_cols(_ptr(xb), R, C, C, _ptr(qT), R, _ptr(s), nb)
    return qT, s


def padded_group_starts(offsets) -> np.ndarray:
    """P_e = sum_{j<e} ceil128(n_j): where group e starts in the padded
    token axis of the grouped column quant; last entry = total padded length."""
    off = np.asarray(offsets, dtype=np.int64)
    n = np.diff(off)
    return np.concatenate([[0], np.cumsum((n + 127) // 128 * 128)]).astype(np.int64)


def mxfp8_quant_cols_grouped(x, offsets, t_pad: int | None = None):
    """Per-group column MXFP8 quant (torchtitan-npu feature guide, MoE MXFP8
    mode: the weight-gradient operands are quantized per group, blocks of 32
    along tokens restarting at each group start).  Returns (codes u8
    [C x t_pad], scales u8 [C x t_pad/32]); padding is zero."""
    xb = _bf16_bits(x)
    T, C = xb.shape
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    E = len(off) - 1
    P = padded_group_starts(off)
    if t_pad is None:
        t_pad = int(P[-1])
    assert t_pad >= P[-1] and t_pad % 128 == 0
    qT = np.zeros((C, t_pad), np.uint8)
    s = np.zeros((C, t_pad // 32), np.uint8)
    if C and E:
        _load().oracle_mxfp8_quant_cols_grouped(_ptr(xb), C, C, _ptr(off), E,
                                                _ptr(qT), t_pad, _ptr(s), t_pad // 32)
    return qT, s


def swizzle_scales(L: np.ndarray) -> np.ndarray:
    """Logical scales [rows x kb] -> flat block-scaled operand layout (rows
    padded to 128, kb padded to 4, 512-byte tiles of 128x4)."""
    L = np.ascontiguousarray(L, dtype=np.uint8)
    rows, kb = L.shape
    rp, kp = (rows + 127) // 128 * 128, (kb + 3) // 4 * 4
    out = np.zeros(rp * kp, np.uint8)
    if rows and kb:
        _load().oracle_swizzle_scales(_ptr(L), rows, kb, kb, _ptr(out))
    return out


def mxfp4_qdq(x: np.ndarray, scale_factor: float = 6.0) -> np.ndarray:
    """MXFP4 quant-dequant of an fp32 array of any shape with blocks of 32
    along the last dim, zero-padded per row (AMCT FakeQuant article,
    sections 2 and 3.3)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    cols = x.shape[-1] if x.ndim else 1
    rows = x.size // cols if cols else 0
    y = np.empty_like(x)
    if x.size:
        _load().oracle_mxfp4_qdq(_ptr(x), _ptr(y), rows, cols, float(scale_factor))
    return y


def mxfp4_quant(x: np.ndarray, scale_factor: float = 6.0):
    """Packed MXFP4 quant of fp32 x[rows x cols] (cols even): returns
    (nibbles u8 [rows x cols/2], scales u8 [rows x ceil(cols/32)])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % 2 == 0
    nb = (cols + 31) // 32
    p = np.zeros((rows, cols // 2), np.uint8)
    s = np.zeros((rows, nb), np.uint8)
    if rows and cols:
        _load().oracle_mxfp4_quant(_ptr(x), rows, cols, cols, float(scale_factor),
                                   _ptr(p), cols // 2, _ptr(s), nb)
    return p, s


def mxfp4_saturation_mask(x: np.ndarray, scale_factor: float = 6.0) -> np.ndarray:
    """Packed saturation mask of MXFP4 quant-dequant (AMCT FakeQuant article,
    section 4.1, clipped STE): uint32 [rows x ceil(cols/32)], bit i of word
    (r, b) set when |x[r, 32b+i]| > 6 * (the block's scale)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    cols = x.shape[-1] if x.ndim else 1
    rows = x.size // cols if cols else 0
    m = np.zeros((rows, (cols + 31) // 32), np.uint32)
    if x.size:
        _load().oracle_mxfp4_saturation_mask(_ptr(x), rows, cols, float(scale_factor), _ptr(m))
    return m


def mxfp4_ste_backward(gy: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Clipped-STE gradient (AMCT FakeQuant article, section 4.1): gy with
    the saturated elements (mask bits, as from mxfp4_saturation_mask) set to
    +0.0."""
    gy = np.ascontiguousarray(gy, dtype=np.float32)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    cols = gy.shape[-1] if gy.ndim else 1
    rows = gy.size // cols if cols else 0
    assert mask.shape == (rows, (cols + 31) // 32)
    gx = np.empty_like(gy)
    if gy.size:
        _load().oracle_mxfp4_ste_backward(_ptr(gy), _ptr(mask), rows, cols, _ptr(gx))
    return gx


from .gemm import (dequant_mxfp8, dequant_mxfp4, gemm_ref, grouped_fwd_ref,  # noqa: E402
                   grouped_dw_ref, linear_ref, qat_linear_ref)

__all__ = [
    "build", "e4m3_encode", "e4m3_decode_table", "e2m1_decode_table", "mxfp8_scale_exp",
    "mxfp4_scale_exp", "mxfp8_quant_rows", "mxfp8_quant_cols", "mxfp8_quant_cols_grouped",
    "padded_group_starts", "swizzle_scales", "mxfp4_qdq", "mxfp4_quant", "mxfp4_saturation_mask",
    "mxfp4_ste_backward", "dequant_mxfp8",
    "dequant_mxfp4", "gemm_ref", "grouped_fwd_ref", "grouped_dw_ref", "linear_ref",
    "qat_linear_ref",
]
