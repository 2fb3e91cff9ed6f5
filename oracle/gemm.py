"""binary64 GEMM references over exactly dequantized MX operands.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Plain definition (torchtitan-npu feature guide, "线性层低精度" MXFP8 mode, and
"MoE 专家层低精度" MXFP8 mode): the layer's forward Y = X W^T, input gradient
dX = dY W and weight gradient dW = dY^T X are computed from MXFP8-quantized
operands; the result is the exact product of the dequantized operands, which
numpy's binary64 matmul reproduces to ~1e-16 relative -- far inside the bf16
tolerance the GPU result is checked against.  A library matmul is the only
step used beyond the definition.

Operand convention: every operand is "K-major": A[M x K] and B[N x K] with
the 32-element scale blocks running along K, and the product is
deq(A) @ deq(B)^T.
"""
from __future__ import annotations

import numpy as np


def _tables():
    from . import e2m1_decode_table, e4m3_decode_table
    return e4m3_decode_table(), e2m1_decode_table()


def _block_scales(s: np.ndarray, cols: int) -> np.ndarray:
    """E8M0 bytes [R x nb] -> binary64 multipliers [R x cols] (2^(byte-127);
    byte 0xFF is NaN)."""
    s = np.asarray(s, dtype=np.uint8)
    mult = np.ldexp(1.0, s.astype(np.int64) - 127)
    mult = np.where(s == 0xFF, np.nan, mult)
    return np.repeat(mult, 32, axis=1)[:, :cols]


def dequant_mxfp8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 codes q[R x C] under logical E8M0 scales
    s[R x ceil(C/32)]."""
    t8, _ = _tables()
    q = np.asarray(q, dtype=np.uint8)
    return t8[q] * _block_scales(s, q.shape[1])


def dequant_mxfp4(p: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Exact value of packed E2M1 nibbles p[R x C/2] (low nibble = even
    column) under logical E8M0 scales s[R x ceil(C/32)]."""
    _, t4 = _tables()
    p = np.asarray(p, dtype=np.uint8)
    nib = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    nib[:, 0::2] = p & 0xF
    nib[:, 1::2] = p >> 4
    return t4[nib] * _block_scales(s, nib.shape[1])


def gemm_ref(qa, sa, qb, sb) -> np.ndarray:
    """C = deq(A) @ deq(B)^T in binary64, A[M x K], B[N x K] K-major."""
    return dequant_mxfp8(qa, sa) @ dequant_mxfp8(qb, sb).T


def grouped_fwd_ref(qa, sa, qb, sb, offsets) -> np.ndarray:
    """Grouped product over row groups: for group e (rows [o_e, o_{e+1}) of
    A[T x K]) the rows of the result are deq(A_e) @ deq(B_e)^T with
    B_e = qb[e] (N x K).  Serves both the MoE forward (B = row-quantized W)
    and the MoE input gradient (A = dY, B = column-quantized W^T)."""
    off = np.asarray(offsets, dtype=np.int64)
    T = qa.shape[0]
    E, N = qb.shape[0], qb.shape[1]
    out = np.zeros((T, N), np.float64)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            out[r0:r1] = gemm_ref(qa[r0:r1], sa[r0:r1], qb[e], sb[e])
    return out


def grouped_dw_ref(qaT, saT, qbT, sbT, offsets) -> np.ndarray:
    """Grouped weight gradient: dW_e = deq(dY_e)^T deq(X_e), contracted over
    the rows of group e only.  Operands are the per-group column quants
    (codes [N x T_pad] / [K x T_pad], group e at padded offset P_e); a group
    with no rows gives an all-zero dW_e."""
    from . import padded_group_starts
    off = np.asarray(offsets, dtype=np.int64)
    P = padded_group_starts(off)
    E = len(off) - 1
    N, K = qaT.shape[0], qbT.shape[0]
    out = np.zeros((E, N, K), np.float64)
    for e in range(E):
        p0, p1 = int(P[e]), int(P[e + 1])
        if p1 > p0:
            out[e] = gemm_ref(qaT[:, p0:p1], saT[:, p0 // 32:p1 // 32],
                              qbT[:, p0:p1], sbT[:, p0 // 32:p1 // 32])
    return out


def linear_ref(x, w, dy):
    """MXFP8 linear layer, forward and both gradients (torchtitan-npu feature
    guide, MXFP8 mode; the MindSpeed fb-split PR for which axis each operand
    is quantized along):
      Y  = deq(row(X))  deq(row(W))^T          contraction over K
      dX = deq(row(dY)) deq(colT(W))^T         contraction over N
      dW = deq(colT(dY)) deq(colT(X))^T        contraction over M
    x: bf16 [M x K], w: bf16 [N x K], dy: bf16 [M x N].  Returns binary64
    (Y, dX, dW)."""
    from . import mxfp8_quant_cols, mxfp8_quant_rows
    qx, sx = mxfp8_quant_rows(x)
    qw, sw = mxfp8_quant_rows(w)
    qdy, sdy = mxfp8_quant_rows(dy)
    qwT, swT = mxfp8_quant_cols(w)
    qdyT, sdyT = mxfp8_quant_cols(dy)
    qxT, sxT = mxfp8_quant_cols(x)
    y = gemm_ref(qx, sx, qw, sw)
    dx = gemm_ref(qdy, sdy, qwT, swT)
    dw = gemm_ref(qdyT, sdyT, qxT, sxT)
    return y, dx, dw


def qat_linear_ref(x, w, bias=None, quantize_input: bool = True, scale_factor: float = 6.0):
    """Forward of the MXFP4 QAT linear layer ("AMCT FakeQuant" article,
    section 4.3): Y = F.linear(Q(x), Q(W), b) with Q the MXFP4 quant-dequant
    (blocks of 32 along the input-feature dim K) and the bias not quantized;
    quantize_input=False leaves x unquantized (W4A16).  x: bf16 [M x K],
    w: bf16 [N x K], bias: bf16 [N] or None.  bf16 values widen exactly to
    fp32 for the quant-dequant, whose outputs (codebook value x 2^e, e >= -30)
    are again exact; the product is binary64.  Returns binary64 [M x N]."""
    from . import _bf16_bits, mxfp4_qdq

    def widen(t):
        return (_bf16_bits(t).astype(np.uint32) << 16).view(np.float32)

    xf, wf = widen(x), widen(w)
    qx = mxfp4_qdq(xf, scale_factor) if quantize_input else xf
    qw = mxfp4_qdq(wf, scale_factor)
    y = qx.astype(np.float64) @ qw.astype(np.float64).T
    if bias is not None:
        y = y + widen(bias).astype(np.float64)[None, :]
    return y
