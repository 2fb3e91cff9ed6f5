"""Pins for the scale layout and the binary64 GEMM references.

The scale layout is the one the tcgen05 block-scaled MMA reads (public PTX ISA
/ cuBLAS block-scaling docs; the pages define none): it is checked against an
independent reshape/permute construction.  The GEMM references are checked
against exact rational brute force on tiny operands, a scaled-identity special
case, and the linear layer's algebra.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import mxq_inputs


@pytest.mark.parametrize("rows,kb", [(128, 4), (130, 5), (1, 1), (300, 129), (256, 128)])
def test_swizzle_vs_reshape_construction(rows, kb):
    rng = np.random.default_rng(rows * 1000 + kb)
    L = rng.integers(1, 255, size=(rows, kb), dtype=np.uint8)
    got = oracle.swizzle_scales(L)
    rp, kp = (rows + 127) // 128 * 128, (kb + 3) // 4 * 4
    padded = np.zeros((rp, kp), np.uint8)
    padded[:rows, :kb] = L
    # rows split as (tile, 4 x 32 sub-rows), columns as (tile, 4): 32 lines of
    # 16 bytes per tile, line i = sub-rows i, i+32, i+64, i+96
    ref = padded.reshape(rp // 128, 4, 32, kp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    assert np.array_equal(got, ref)


def _exact_gemm(qa, sa, qb, sb):
    t = oracle.e4m3_decode_table()
    M, K = qa.shape
    N = qb.shape[0]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = Fraction(t[qa[i, k]]) * Fraction(2) ** (int(sa[i, k // 32]) - 127)
                b = Fraction(t[qb[j, k]]) * Fraction(2) ** (int(sb[j, k // 32]) - 127)
                acc += a * b
            out[i, j] = float(acc)
    return out


def test_gemm_ref_vs_exact_rationals():
    x, w, _ = mxq_inputs.linear_inputs(5, 4, 96, seed=2)
    qa, sa = oracle.mxfp8_quant_rows(x)
    qb, sb = oracle.mxfp8_quant_rows(w)
    got = oracle.gemm_ref(qa, sa, qb, sb)
    ref = _exact_gemm(qa, sa, qb, sb)
    assert np.allclose(got, ref, rtol=1e-13, atol=0)


def test_gemm_ref_scaled_identity_is_dequant():
    x = mxq_inputs.normal_bf16((32, 64), 1.0, seed=9)
    qa, sa = oracle.mxfp8_quant_rows(x)
    qb = np.zeros((64, 64), np.uint8)
    np.fill_diagonal(qb, 0x38)                    # E4M3 1.0
    sb = np.full((64, 2), 127 + 3, np.uint8)      # 2^3
    got = oracle.gemm_ref(qa, sa, qb, sb)
    assert np.array_equal(got, 8.0 * oracle.dequant_mxfp8(qa, sa))


def test_linear_ref_tracks_unquantized_products():
    """A transposed or swapped operand would be off by O(1), not O(2^-4)."""
    x, w, dy = mxq_inputs.linear_inputs(64, 96, 128, seed=4)
    y, dx, dw = oracle.linear_ref(x, w, dy)
    X, W, DY = (t.to(torch.float64).numpy() for t in (x, w, dy))
    for got, ref in ((y, X @ W.T), (dx, DY @ W), (dw, DY.T @ X)):
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 0.05, rel


def test_grouped_refs_are_per_slice_and_zero_for_empty_groups():
    sizes = [3, 0, 40, 0, 21]
    off, x, w, dy = mxq_inputs.moe_inputs(5, 64, 64, 32, seed=6, sizes=sizes)
    qx, sx = oracle.mxfp8_quant_rows(x)
    qw = np.stack([oracle.mxfp8_quant_rows(w[e])[0] for e in range(5)])
    sw = np.stack([oracle.mxfp8_quant_rows(w[e])[1] for e in range(5)])
    y = oracle.grouped_fwd_ref(qx, sx, qw, sw, off)
    for e in range(5):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            assert np.array_equal(y[r0:r1], oracle.gemm_ref(qx[r0:r1], sx[r0:r1], qw[e], sw[e]))
    qdyT, sdyT = oracle.mxfp8_quant_cols_grouped(dy, off)
    qxT, sxT = oracle.mxfp8_quant_cols_grouped(x, off)
    dw = oracle.grouped_dw_ref(qdyT, sdyT, qxT, sxT, off)
    assert not np.any(dw[1]) and not np.any(dw[3])
    for e in (0, 2, 4):
        r0, r1 = off[e], off[e + 1]
        a, sa = oracle.mxfp8_quant_cols(dy[r0:r1])
        b, sb = oracle.mxfp8_quant_cols(x[r0:r1])
        assert np.array_equal(dw[e], oracle.gemm_ref(a, sa, b, sb))


# ---------------------------------------------------------------------------
# MXFP4 QAT linear forward (AMCT FakeQuant article, section 4.3)
# ---------------------------------------------------------------------------

def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _on_mxfp4_grid(R, K, seed):
    """bf16 [R x K] whose every 32-block along K holds +-6 * 2^e (so that the
    block's scale is exactly 2^e) and otherwise codebook values x 2^e, e
    varying per block: a fixed point of the MXFP4 quant-dequant along K only."""
    rng = np.random.default_rng(seed)
    book = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = rng.choice(book, size=(R, K)) * rng.choice([-1.0, 1.0], size=(R, K))
    v[:, ::32] = 6.0 * rng.choice([-1.0, 1.0], size=(R, K // 32))
    e = rng.integers(-8, 8, size=(R, K // 32))
    return v * np.repeat(np.exp2(e), 32, axis=1)


def test_qat_ref_is_exact_product_on_the_mxfp4_grid():
    """Inputs already on the MXFP4 grid along K are left unchanged by Q, so Y
    is their plain product; quantizing along any other axis would move them."""
    x, w = _on_mxfp4_grid(48, 128, 1), _on_mxfp4_grid(40, 128, 2)
    y = oracle.qat_linear_ref(_bf16(x), _bf16(w))
    assert np.array_equal(y, x @ w.T)
    assert not np.array_equal(oracle.mxfp4_qdq(x.T.astype(np.float32).copy()), x.T.astype(np.float32))


def test_qat_ref_w4a16_leaves_the_input_unquantized():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((32, 96)))
    w = _on_mxfp4_grid(24, 96, 4)
    xf = x.to(torch.float64).numpy()
    assert np.array_equal(oracle.qat_linear_ref(x, _bf16(w), quantize_input=False), xf @ w.T)
    assert not np.array_equal(oracle.qat_linear_ref(x, _bf16(w), quantize_input=True), xf @ w.T)


def test_qat_ref_bias_is_not_quantized():
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((8, 64)))
    b = _bf16(0.1 + 0.01 * rng.standard_normal(16))  # off the MXFP4 grid
    y = oracle.qat_linear_ref(x, _bf16(np.zeros((16, 64))), b)
    assert np.array_equal(y, np.broadcast_to(b.to(torch.float64).numpy(), (8, 16)))


def test_qat_ref_matches_packed_mxfp4_route():
    """Q via packed MXFP4 codes + scales, dequantized, gives the same product."""
    x = mxq_inputs.mxfp4_large(64, 256, seed=6)
    w = mxq_inputs.mxfp4_large(32, 256, seed=7)
    xb, wb = _bf16(x), _bf16(w)
    px, sx = oracle.mxfp4_quant(xb.to(torch.float32).numpy())
    pw, sw = oracle.mxfp4_quant(wb.to(torch.float32).numpy())
    ref = oracle.dequant_mxfp4(px, sx) @ oracle.dequant_mxfp4(pw, sw).T
    assert np.array_equal(oracle.qat_linear_ref(xb, wb), ref)
