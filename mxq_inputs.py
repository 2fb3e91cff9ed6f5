"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds random-number recipes only -- none of the quantization or
GEMM arithmetic -- so that the oracle and the CUDA path can be fed the very
same bytes without sharing any of the method's code.

Recipe: numpy ``PCG64(SeedSequence(seed))`` spawns one child stream per tensor,
in the order X, W, dY, group sizes, outliers; values are drawn in fp32 and,
for bf16 tensors, rounded to bf16 (round-to-nearest-even) by torch's cast.
All tensors are returned on the CPU.
"""
from __future__ import annotations

import numpy as np
import torch


def _streams(seed: int, n: int = 5):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal_bf16(shape, std: float, seed: int = 0, stream: int = 0) -> torch.Tensor:
    rng = _streams(seed)[stream]
    return _bf16(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def linear_inputs(M: int, N: int, K: int, seed: int = 0):
    """Dense linear layer: X[M x K] ~ N(0,1), W[N x K] ~ N(0,0.02^2),
    dY[M x N] ~ N(0,(1e-3)^2), all bf16."""
    sx, sw, sdy, _, _ = _streams(seed)
    x = _bf16(sx.standard_normal((M, K), dtype=np.float32))
    w = _bf16(sw.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    dy = _bf16(sdy.standard_normal((M, N), dtype=np.float32) * np.float32(1e-3))
    return x, w, dy


def dirichlet_group_sizes(E: int, T: int, alpha: float = 0.5, seed: int = 0) -> np.ndarray:
    """Routed-token counts per expert: p ~ Dirichlet(alpha * 1_E),
    n_e = floor(p_e T), the remainder handed out largest-fraction-first
    (ties to the lower expert index).  Zero-size groups are allowed."""
    rng = _streams(seed)[3]
    p = rng.dirichlet(np.full(E, alpha))
    raw = p * T
    n = np.floor(raw).astype(np.int64)
    rem = int(T - n.sum())
    frac = raw - n
    order = sorted(range(E), key=lambda e: (-frac[e], e))
    for e in order[:rem]:
        n[e] += 1
    assert n.sum() == T
    return n


def offsets_from_sizes(n) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(n, dtype=np.int64))]).astype(np.int64)


def moe_inputs(E: int, T: int, K: int, N: int, seed: int = 0, alpha: float = 0.5,
               sizes=None, need_dy: bool = True):
    """MoE expert layer: group offsets from Dirichlet(alpha) sizes (or the
    given sizes), X[T x K] ~ N(0,1), W[E x N x K] ~ N(0,0.02^2),
    dY[T x N] ~ N(0,(1e-3)^2), all bf16."""
    sx, sw, sdy, _, _ = _streams(seed)
    n = dirichlet_group_sizes(E, T, alpha, seed) if sizes is None else np.asarray(sizes, np.int64)
    off = offsets_from_sizes(n)
    x = _bf16(sx.standard_normal((T, K), dtype=np.float32))
    w = _bf16(sw.standard_normal((E, N, K), dtype=np.float32) * np.float32(0.02))
    dy = _bf16(sdy.standard_normal((T, N), dtype=np.float32) * np.float32(1e-3)) if need_dy else None
    return off, x, w, dy


def heavy_tail(shape, outlier_mult: float, seed: int = 0, zero_block_frac: float = 0.0,
               outlier_rate: float = 0.01) -> np.ndarray:
    """fp32 values 0.1 * StudentT(nu=3); a Bernoulli(outlier_rate) mask
    multiplies entries by `outlier_mult`; `zero_block_frac` of the 32-element
    blocks along the last dim (chosen by the seed) are set to zero."""
    s = _streams(seed)
    a = (np.float32(0.1) * s[0].standard_t(3, size=shape)).astype(np.float32)
    mask = s[4].random(size=shape) < outlier_rate
    a = np.where(mask, a * np.float32(outlier_mult), a).astype(np.float32)
    if zero_block_frac > 0 and a.size:
        cols = a.shape[-1]
        nb = (cols + 31) // 32
        flat = a.reshape(-1, cols)
        blocks = s[3].random(size=(flat.shape[0], nb)) < zero_block_frac
        for r, b in zip(*np.nonzero(blocks)):
            flat[r, 32 * b:32 * b + 32] = 0
        a = flat.reshape(shape)
    return a


def mxfp4_small(shape, seed: int = 0) -> np.ndarray:
    """fp32 ~ N(0,1) for the ragged-shape MXFP4 cases."""
    return _streams(seed)[0].standard_normal(shape, dtype=np.float32)


def mxfp4_large(rows: int = 4096, cols: int = 4096, seed: int = 0) -> np.ndarray:
    """fp32 0.1*StudentT(3), 1% outliers x100, 1% of 32-blocks zeroed."""
    return heavy_tail((rows, cols), 100.0, seed, zero_block_frac=0.01)


def sweep_bf16(R: int, C: int, seed: int = 0) -> torch.Tensor:
    """bf16 0.1*StudentT(3) with 1% outliers x1000 (dual-quant bandwidth sweep)."""
    return _bf16(heavy_tail((R, C), 1000.0, seed))


def sweep_bf16_device(R: int, C: int, seed: int, device) -> torch.Tensor:
    """The sweep_bf16 distribution drawn on the device (seeded torch generator)
    for the sweep's largest sizes (up to 2^30 elements): 0.1 * Z / sqrt(V/3)
    with Z ~ N(0,1) and V a sum of 3 squared normals (StudentT(3)), entries
    multiplied by 1000 with probability 0.01, rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn((R, C), generator=g, device=device)
    v = torch.zeros((R, C), device=device)
    for _ in range(3):
        v.add_(torch.randn((R, C), generator=g, device=device).square_())
    t = z.mul_(0.1).div_(v.div_(3.0).sqrt_())
    del v
    out = torch.where(torch.rand((R, C), generator=g, device=device) < 0.01, t * 1000.0, t)
    return out.to(torch.bfloat16)
