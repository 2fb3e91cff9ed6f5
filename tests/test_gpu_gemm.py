"""GPU parity of the block-scaled MXFP8 GEMM against the binary64 oracle.

Tolerance (stated for the method): max |C - C_ref| / max |C_ref| <= 1e-2 and
||C - C_ref||_F / ||C_ref||_F <= 2e-3, C_ref = deq(A) deq(B)^T in binary64.
Where every partial sum is exact in fp32 the result must match bit for bit.
"""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAXREL, FROB = 1e-2, 2e-3


def _bf16_rne(ref: np.ndarray) -> np.ndarray:
    return torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy()


def check_close(got: torch.Tensor, ref: np.ndarray):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    maxrel = np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-300)
    frob = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300)
    assert maxrel <= MAXREL and frob <= FROB, (maxrel, frob)
    return maxrel, frob


def run_gemm(mxq, qa, sa, qb, sb, M, N, K):
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_gemm(torch.from_numpy(qa).to(DEV), torch.from_numpy(sa).to(DEV), torch.from_numpy(qb).to(DEV),
                 torch.from_numpy(sb).to(DEV), M, N, K, c, N)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    return c


def _exact_operands(R, K, rng):
    """Codes in {+-1, +-2} and scales in {2^-1, 2^0, 2^1}: every partial sum of
    a K <= 4096 contraction is an exact fp32 value (|sum| <= 2^18 in units of 2^-2)."""
    q = rng.choice(np.array([0x38, 0xB8, 0x40, 0xC0], np.uint8), size=(R, K))
    s = rng.integers(126, 129, size=(R, K // 32), dtype=np.uint8)
    return q, s


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (128, 256, 4096), (300, 384, 160), (1, 8, 32), (517, 1000, 96)])
def test_exact_sums_bit_exact(mxq, M, N, K):
    rng = np.random.default_rng(M * N + K)
    qa, la = _exact_operands(M, K, rng)
    qb, lb = _exact_operands(N, K, rng)
    c = run_gemm(mxq, qa, oracle.swizzle_scales(la), qb, oracle.swizzle_scales(lb), M, N, K)
    ref = oracle.gemm_ref(qa, la, qb, lb)
    assert np.array_equal(c.cpu().view(torch.int16).numpy(), _bf16_rne(ref))


def test_scaled_identity_is_dequant(mxq):
    x = mxq_inputs.normal_bf16((256, 256), 1.0, seed=1)
    qa, la = oracle.mxfp8_quant_rows(x)
    qb = np.zeros((256, 256), np.uint8)
    np.fill_diagonal(qb, 0x38)
    lb = np.full((256, 8), 127 + 5, np.uint8)
    c = run_gemm(mxq, qa, oracle.swizzle_scales(la), qb, oracle.swizzle_scales(lb), 256, 256, 256)
    ref = 32.0 * oracle.dequant_mxfp8(qa, la)
    assert np.array_equal(c.cpu().view(torch.int16).numpy(), _bf16_rne(ref))


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (1024, 768, 1024), (200, 136, 2080)])
def test_quantized_linear_forward_within_tolerance(mxq, M, N, K):
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=M)
    xq, xs, _, _ = mxq.quantize_mxfp8(x.to(DEV))
    wq, ws, _, _ = mxq.quantize_mxfp8(w.to(DEV))
    c = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_gemm(xq, xs, wq, ws, M, N, K, c, N)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    wq_o, ws_o = oracle.mxfp8_quant_rows(w)
    check_close(c, oracle.gemm_ref(oq, os_, wq_o, ws_o))


def test_full_size_gemm_sampled_rows(mxq):
    """Y = X W^T at M=8192, N=14336, K=4096 (the dense layer's forward), checked on
    96 sampled rows (every column) against the binary64 oracle."""
    M, N, K = 8192, 14336, 4096
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=0)
    xq, xs, _, _ = mxq.quantize_mxfp8(x.to(DEV))
    wq, ws, _, _ = mxq.quantize_mxfp8(w.to(DEV))
    c = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_gemm(xq, xs, wq, ws, M, N, K, c, N)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(0).choice(M, 96, replace=False))
    rows = np.unique(np.concatenate([rows, [0, 127, 128, M - 1]]))
    oq, os_ = oracle.mxfp8_quant_rows(x[torch.from_numpy(rows)])
    wq_o, ws_o = oracle.mxfp8_quant_rows(w)
    ref = oracle.gemm_ref(oq, os_, wq_o, ws_o)
    check_close(c[torch.from_numpy(rows).to(DEV)], ref)


@pytest.mark.parametrize("M,N,K,ldc", [(300, 384, 256, 448), (517, 1000, 96, 1008), (128, 256, 512, 4096),
                                       (1, 8, 32, 16)])
def test_strided_output(mxq, M, N, K, ldc):
    """C written with a row pitch ldc > N: the [M x N] block equals the
    exact product bit for bit, and the columns [N, ldc) keep their contents."""
    rng = np.random.default_rng(M + N + K + ldc)
    qa, la = _exact_operands(M, K, rng)
    qb, lb = _exact_operands(N, K, rng)
    big = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_gemm(torch.from_numpy(qa).to(DEV), torch.from_numpy(oracle.swizzle_scales(la)).to(DEV),
                 torch.from_numpy(qb).to(DEV), torch.from_numpy(oracle.swizzle_scales(lb)).to(DEV), M, N, K, big, ldc)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    ref = oracle.gemm_ref(qa, la, qb, lb)
    got = big.cpu().view(torch.int16).numpy()
    assert np.array_equal(got[:, :N], _bf16_rne(ref))
    assert torch.isnan(big[:, N:].float()).all()
