"""Pins for the oracle's reading of blocks that hold an Inf or a NaN.

The pages say nothing about non-finite inputs.  What independent references
fix is pinned here:
  - the E8M0 scale byte of such a block is the library's E8M0 cast of its
    non-finite amax (torch float8_e8m0fnu: 0xFF, the format's NaN);
  - the MXFP8 code of a non-finite element is the library's E4M3 cast of
    that element (torch float8_e4m3fn: 0x7F with the element's sign);
  - every element of the block dequantizes to NaN (the E8M0 NaN scale, decoded
    by ml_dtypes), whatever code the finite elements carry;
  - in MXFP4 quant-dequant, evaluating the rule of the AMCT FakeQuant article
    (section 2) literally in IEEE binary32 -- scale 2^round(log2(max(amax/sf,
    2^-30))) overflows to +inf, so a finite element becomes 0 * inf -- gives
    NaN for every finite element of the block.
Left as readings, with nothing outside the oracle to fix them: the code bytes
of the FINITE elements of a non-finite MXFP8 block (0x7F with their sign), the
QDQ result of the non-finite element itself (NaN; the literal formula gives
NaN or +-inf there depending on how the codebook search orders NaN), and the
packed E2M1 nibble of a non-finite block (7 with the sign; E2M1 has no NaN)."""
import ml_dtypes
import numpy as np
import torch

import oracle

INF_NAN_BF16 = [0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81, 0xFFFF]   # +Inf, -Inf, NaNs of both signs


def _blocks(bad_bits):
    """One block of 32 bf16 per pattern: finite values of both signs, one of
    them replaced by the non-finite pattern."""
    rng = np.random.default_rng(7)
    fin = torch.from_numpy(rng.standard_normal((len(bad_bits), 32)).astype(np.float32)).to(torch.bfloat16)
    bits = fin.view(torch.int16).numpy().view(np.uint16).copy()
    for i, b in enumerate(bad_bits):
        bits[i, (5 * i) % 32] = b
    return bits


def test_mxfp8_scale_byte_is_the_e8m0_cast_of_the_amax():
    bits = _blocks(INF_NAN_BF16)
    _, s = oracle.mxfp8_quant_rows(bits)
    amax = np.abs(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy())
    amax = np.where(np.isnan(amax).any(axis=1), np.nan, amax.max(axis=1))
    lib = torch.from_numpy(amax.astype(np.float32)).to(torch.float8_e8m0fnu).view(torch.uint8).numpy()
    assert np.array_equal(s[:, 0], lib)
    assert (s[:, 0] == 0xFF).all()


def test_mxfp8_code_of_the_nonfinite_element_is_the_e4m3_cast():
    bits = _blocks(INF_NAN_BF16)
    q, _ = oracle.mxfp8_quant_rows(bits)
    for i, b in enumerate(INF_NAN_BF16):
        j = (5 * i) % 32
        v = torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float32)
        assert q[i, j] == v.to(torch.float8_e4m3fn).view(torch.uint8).item()


def test_mxfp8_nonfinite_block_dequantizes_to_nan():
    bits = _blocks(INF_NAN_BF16)
    q, s = oracle.mxfp8_quant_rows(bits)
    scale = np.array(s[:, 0].view(ml_dtypes.float8_e8m0fnu), dtype=np.float64)
    assert np.isnan(scale).all()
    assert np.isnan(oracle.dequant_mxfp8(q, s)).all()
    # the column direction gives the same block result
    qT, sT = oracle.mxfp8_quant_cols(np.ascontiguousarray(bits.T))
    assert (sT[:, 0] == 0xFF).all() and np.isnan(oracle.dequant_mxfp8(qT, sT)).all()


def _literal_qdq_finite(x: np.ndarray, sf: float = 6.0) -> np.ndarray:
    """The article's rule evaluated step by step in IEEE binary32 (numpy),
    for the FINITE elements of each 32-element row block."""
    x = x.astype(np.float32)
    with np.errstate(all="ignore"):
        amax = np.max(np.abs(x), axis=1, keepdims=True)               # propagates NaN / Inf
        r = np.maximum(amax / np.float32(sf), np.float32(2.0 ** -30))
        s = np.exp2(np.round(np.log2(r))).astype(np.float32)          # +inf for an Inf amax, NaN for a NaN one
        y = np.abs(x) / s
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
        vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
        q = vals[np.searchsorted(mids, np.nan_to_num(y, nan=0.0), side="right")]
        out = np.copysign(q * s, x)
    return np.where(np.isfinite(x), out, np.float32(0))


def test_mxfp4_finite_elements_of_a_nonfinite_block_are_nan():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 32)).astype(np.float32)
    x[0, 3], x[1, 30], x[2, 0], x[3, 17] = np.inf, -np.inf, np.nan, -np.nan
    got = oracle.mxfp4_qdq(x)
    lit = _literal_qdq_finite(x)
    fin = np.isfinite(x)
    assert np.isnan(lit[fin]).all()                  # the literal rule: 0 * inf or NaN arithmetic
    assert np.isnan(got[fin]).all()
    assert np.isnan(got).all()                       # the reading for the non-finite element itself


def test_mxfp4_packed_nonfinite_block_scale_byte():
    x = np.zeros((2, 32), np.float32)
    x[0, 1], x[1, 2] = np.inf, np.nan
    _, s = oracle.mxfp4_quant(x)
    lib = torch.tensor([np.inf, np.nan], dtype=torch.float32).to(torch.float8_e8m0fnu).view(torch.uint8).numpy()
    assert np.array_equal(s[:, 0], lib)
