"""Pins for the MXFP8 oracle.

The pages fix only the block (32 contiguous elements share one scale;
torchtitan-npu feature guide, "线性层低精度" MXFP8 mode).  The element/scale
rule is the OCP MX one: scale 2^X with X = floor(log2 amax) - 8 (clamped to
[-127, 127], X = -127 for an all-zero block), codes E4M3 of x * 2^-X rounded to
nearest-even and saturated to +-448.

Independent references used here: torch's float8_e4m3fn / float8_e8m0fnu casts
(library routines), a brute-force search for X, ml_dtypes, and invariants that
tie the row, column and grouped variants together.
"""
import numpy as np
import pytest
import torch

import oracle
import mxq_inputs


def _bf16_from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def _torch_e4m3_code(y: torch.Tensor) -> np.ndarray:
    """Library reference: clamp to +-448 then torch's RNE cast to E4M3."""
    c = y.to(torch.float32).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return c.view(torch.uint8).numpy()


def _brute_X(amax: float) -> int:
    """Largest X in [-127, 127] with 256 * 2^X <= amax (X = -127 for 0)."""
    best = -127
    for X in range(-127, 128):
        if 256.0 * 2.0 ** X <= amax:
            best = X
    return best


def test_e4m3_decode_matches_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_including_ties():
    vals = oracle.e4m3_decode_table()
    finite = np.sort(np.unique(np.abs(vals[~np.isnan(vals)])))
    mids = (finite[:-1] + finite[1:]) / 2            # every tie between neighbours
    rng = np.random.default_rng(0)
    rand = np.exp2(rng.uniform(-12, 9.5, 3000))
    ys = np.concatenate([finite, mids, rand, [448.0, 455.0, 464.0, 470.0, 1e4, 2.0 ** -10, 3 * 2.0 ** -11]])
    ys = np.concatenate([ys, -ys]).astype(np.float32)
    ref = _torch_e4m3_code(torch.from_numpy(ys))
    got = np.array([oracle.e4m3_encode(float(v)) for v in ys], np.uint8)
    assert np.array_equal(got, ref)
    # spot values: RNE 17 -> 16, 464 (tie) -> 448, 3*2^-11 -> 2^-9 (tie to even)
    assert oracle.e4m3_decode_table()[oracle.e4m3_encode(17.0)] == 16.0
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_decode_table()[oracle.e4m3_encode(3 * 2.0 ** -11)] == 2.0 ** -9


def test_exhaustive_single_element_blocks():
    """All 65,536 bf16 patterns as the only nonzero element of a block."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = _bf16_from_bits(bits).to(torch.float64).numpy()
    finite = np.isfinite(vals)
    blocks = np.zeros((65536, 32), np.uint16)
    blocks[:, 5] = bits
    q, s = oracle.mxfp8_quant_rows(blocks)
    # scale byte by brute-force search, once per distinct magnitude exponent
    for i in np.nonzero(finite)[0][::37]:
        assert s[i, 0] == _brute_X(abs(vals[i])) + 127, hex(bits[i])
    # scale byte vs torch's E8M0 cast of 2^X (all finite patterns)
    X = s[finite, 0].astype(np.int64) - 127
    e8 = torch.from_numpy(np.ldexp(1.0, X).astype(np.float32)).to(torch.float8_e8m0fnu).view(torch.uint8).numpy()
    assert np.array_equal(e8, s[finite, 0])
    # codes vs torch's cast of x * 2^-X (exact in fp32 here)
    y = torch.from_numpy(np.ldexp(vals[finite], -X))
    assert np.array_equal(q[finite, 5], _torch_e4m3_code(y))
    assert not np.any(q[finite, :5]) and not np.any(q[finite, 6:])
    # non-finite blocks: scale 0xFF (documented reading, unpinned)
    assert np.all(s[~finite, 0] == 0xFF)


def test_random_blocks_vs_torch_reference():
    x = mxq_inputs.sweep_bf16(96, 256, seed=7)           # heavy tail + 1000x outliers
    x[3, :32] = 0                                        # an all-zero block
    x[5, 32:64] = -0.0
    q, s = oracle.mxfp8_quant_rows(x)
    xf = x.to(torch.float64).view(96, 8, 32)
    amax = xf.abs().amax(-1)
    X = torch.where(amax > 0, torch.floor(torch.log2(amax)) - 8, torch.full_like(amax, -127)).clamp(-127, 127)
    assert np.array_equal(s.astype(np.int64) - 127, X.to(torch.int64).numpy())
    y = (xf * torch.exp2(-X)[..., None]).view(96, 256)
    assert np.array_equal(q, _torch_e4m3_code(y))
    assert s[3, 0] == 0 and not np.any(q[3, :32])
    assert np.all(q[5, 32:64] == 0x80)                   # -0.0 keeps its sign


def test_worked_examples():
    one = torch.zeros(1, 32, dtype=torch.bfloat16)
    one[0, 0] = 1.0
    q, s = oracle.mxfp8_quant_rows(one)
    assert s[0, 0] == 127 - 8 and q[0, 0] == 0x78        # 1.0 = 256 * 2^-8
    big = torch.tensor([[500.0] + [0.0] * 31], dtype=torch.bfloat16)
    q, s = oracle.mxfp8_quant_rows(big)
    assert s[0, 0] == 127 and q[0, 0] == 0x7E            # 500 saturates to 448
    q, s = oracle.mxfp8_quant_rows(torch.zeros(2, 64, dtype=torch.bfloat16))
    assert not np.any(s) and not np.any(q)


def test_dequant_error_and_range_invariants():
    x = mxq_inputs.normal_bf16((64, 512), 1.0, seed=3)
    q, s = oracle.mxfp8_quant_rows(x)
    deq = oracle.dequant_mxfp8(q, s)
    xv = x.to(torch.float64).numpy()
    X = s.astype(np.int64) - 127
    top = np.abs(deq).reshape(64, 16, 32).max(-1) / np.ldexp(1.0, X)
    assert np.all((top >= 256) & (top <= 448))
    # unsaturated normals: |x - deq| <= half an E4M3 ulp = 2^(floor(log2|x|) - 4)
    ok = (np.abs(xv) >= np.ldexp(1.0, np.repeat(X, 32, 1) - 6)) & (np.abs(xv) < 448 * np.ldexp(1.0, np.repeat(X, 32, 1)))
    ulp = np.ldexp(1.0, np.floor(np.log2(np.abs(np.where(ok, xv, 1.0)))).astype(int) - 4)
    assert np.all(np.abs(xv - deq)[ok] <= ulp[ok])


@pytest.mark.parametrize("R,C", [(64, 96), (100, 64), (37, 32), (1, 320)])
def test_col_quant_is_row_quant_of_transpose(R, C):
    x = mxq_inputs.normal_bf16((R, C), 1.0, seed=R * C)
    qT, sT = oracle.mxfp8_quant_cols(x)
    q2, s2 = oracle.mxfp8_quant_rows(x.t().contiguous())
    assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_grouped_cols_is_per_slice_concat():
    sizes = [0, 5, 128, 33, 0, 200, 1]
    off = mxq_inputs.offsets_from_sizes(sizes)
    x = mxq_inputs.normal_bf16((int(off[-1]), 64), 1.0, seed=11)
    qT, sT = oracle.mxfp8_quant_cols_grouped(x, off)
    P = oracle.padded_group_starts(off)
    assert P[-1] == 0 + 128 + 128 + 128 + 0 + 256 + 128
    for e in range(len(sizes)):
        r0, r1, p0 = off[e], off[e + 1], P[e]
        n = r1 - r0
        if n == 0:
            continue
        qe, se = oracle.mxfp8_quant_cols(x[r0:r1])
        assert np.array_equal(qT[:, p0:p0 + n], qe)
        assert np.array_equal(sT[:, p0 // 32:p0 // 32 + se.shape[1]], se)
        # the padded tail of the group is zero
        assert not np.any(qT[:, p0 + n:P[e + 1]])
        assert not np.any(sT[:, p0 // 32 + se.shape[1]:P[e + 1] // 32])
