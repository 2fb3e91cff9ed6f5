"""Pins of the oracle's MXFP4 saturation mask and clipped-STE backward
("AMCT FakeQuant" article, section 4.1 "STE 与 clipped STE": an element is
saturated when |x| > 6 * block scale; the clipped STE zeroes the gradient
there and passes it through elsewhere).

The pins do not re-run the oracle's formula: they use hand-derived worked
examples, the closed-form bounds on scale_factor under which nothing / every
block maximum saturates, the article's own statistical claim (a block maximum
is clipped about half the time), agreement with the separately pinned QDQ
oracle, and exact rational brute force on tiny blocks.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import mxq_inputs
import oracle


def _bits(mask: np.ndarray, cols: int) -> np.ndarray:
    """Unpack uint32 words [rows x nb] to bool [rows x cols]."""
    rows, nb = mask.shape
    b = (mask[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return b.reshape(rows, nb * 32)[:, :cols].astype(bool)


def _block(vals, cols=32):
    x = np.zeros((1, cols), np.float32)
    x[0, : len(vals)] = vals
    return x


# (scale_factor, block values, saturated positions).  Derivations, with
# r = amax / sf and e = round(log2 r) (rounds up iff r >= sqrt(2) * 2^floor):
WORKED = [
    # r = 1 exactly: e = 0, limit 6; 6 > 6 is false
    (6.0, [6.0], []),
    # r = 1.083: e = 0, limit 6; 6.5 saturates
    (6.0, [6.5], [0]),
    # r = 1.333 < 1.414: e = 0, limit 6; 8 saturates
    (6.0, [8.0], [0]),
    # r = 1.41333 < 1.41421: e = 0, limit 6; 8.48 saturates
    (6.0, [8.48], [0]),
    # r = 1.41667 > 1.41421: e = 1, limit 12; nothing saturates
    (6.0, [8.5], []),
    # r = 0.5: e = -1, limit 3; 3 > 3 is false
    (6.0, [3.0], []),
    # r = 0.667, log2 r = -0.585: e = -1, limit 3; 4 saturates
    (6.0, [4.0], [0]),
    # r = 0.7167 > 0.7071: e = 0, limit 6
    (6.0, [4.3], []),
    # amax = 0: scale clamped to 2^-30, nothing saturates
    (6.0, [0.0, -0.0], []),
    # r = 1.7e-11 < 2^-30: e = -30, limit 6 * 2^-30 = 5.6e-9 > 1e-10
    (6.0, [1e-10], []),
    # r = 1e-8/6 = 1.67e-9 (log2 = -29.16): e = -29, limit 1.1e-8 > 1e-8
    (6.0, [1e-8], []),
    # r = 3e-9/6 = 5e-10 < 2^-30 = 9.3e-10: e = -30, limit 5.59e-9 > 3e-9
    (6.0, [3e-9], []),
    # several elements: amax 8 -> e = 0, limit 6: 8, 7, -6.5 saturate; 6, 5, -6 do not
    (6.0, [8.0, 7.0, 6.0, 5.0, -6.5, -6.0, 0.25], [0, 1, 4]),
    # sf = 1: r = 1.3 -> e = 0, limit 6
    (1.0, [1.3, -1.0], []),
    # sf = 12 (inv_scale_factor_scale 0.5): r = 1/12, log2 r = -3.585 -> e = -4,
    # limit 6/16 = 0.375: 1 and -0.5 saturate, 0.375 does not
    (12.0, [1.0, -0.5, 0.375, 0.3], [0, 1]),
]


@pytest.mark.parametrize("sf,vals,sat", WORKED)
def test_worked_examples(sf, vals, sat):
    x = _block(vals)
    got = np.flatnonzero(_bits(oracle.mxfp4_saturation_mask(x, sf), 32)[0])
    assert got.tolist() == sat


def test_limit_is_the_top_codebook_value():
    """Saturated elements are exactly the ones QDQ maps to +-6 * scale while
    |x| lies above it (the codebook's top value, AMCT article section 2)."""
    x = mxq_inputs.mxfp4_large(256, 512, seed=3)
    for sf in (6.0, 7.0, 12.0, 5.0):
        m = _bits(oracle.mxfp4_saturation_mask(x, sf), x.shape[1])
        y = oracle.mxfp4_qdq(x, sf)
        xb = x.reshape(x.shape[0], -1, 32)
        amax = np.abs(xb).max(axis=2)
        scale = np.array([[2.0 ** oracle.mxfp4_scale_exp(float(a), sf) for a in row] for row in amax])
        top = np.repeat(6.0 * scale, 32, axis=1)
        qy = np.abs(y.astype(np.float64))
        ax = np.abs(x.astype(np.float64))
        assert np.array_equal(m, (qy == top) & (ax > top))
        assert m.any() or sf < 6.0 / math.sqrt(2)


@pytest.mark.parametrize("sf", [0.5, 1.0, 3.0, 4.2])
def test_no_saturation_below_6_over_sqrt2(sf):
    """e >= log2(amax/sf) - 1/2, so 6 * 2^e >= 6 amax / (sf sqrt 2) > amax
    whenever sf < 6/sqrt(2) = 4.243: nothing can saturate."""
    x = mxq_inputs.mxfp4_large(128, 1024, seed=11)
    assert not oracle.mxfp4_saturation_mask(x, sf).any()


@pytest.mark.parametrize("sf", [8.5, 10.0, 64.0])
def test_block_max_always_saturates_above_6_sqrt2(sf):
    """e <= log2(amax/sf) + 1/2, so 6 * 2^e <= 6 sqrt(2) amax / sf < amax
    whenever sf > 6 sqrt(2) = 8.485 (and amax/sf is above the 2^-30 clamp):
    every block's largest element saturates."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    m = _bits(oracle.mxfp4_saturation_mask(x, sf), 256).reshape(64, 8, 32)
    xb = np.abs(x).reshape(64, 8, 32)
    arg = xb.argmax(axis=2)
    assert np.take_along_axis(m, arg[:, :, None], axis=2).all()


def test_block_max_clipped_about_half_the_time():
    """The article (section 4.1) notes that because the scale exponent is
    rounded, a block's maximum exceeds 6 * scale with probability about 1/2.
    With sf = 6 and log2(amax) uniform, the block maximum saturates exactly
    when the fractional part of log2(amax/6) is in (0, 1/2): probability 1/2."""
    rng = np.random.default_rng(7)
    n = 200_000
    amax = np.exp2(rng.uniform(-10.0, 10.0, n)).astype(np.float32)
    x = np.zeros((n, 32), np.float32)
    x[:, 0] = amax
    x[:, 1:] = amax[:, None] * rng.uniform(-1.0, 1.0, (n, 31)).astype(np.float32)
    m = oracle.mxfp4_saturation_mask(x, 6.0)[:, 0]
    frac = ((m & 1) != 0).mean()
    assert abs(frac - 0.5) < 0.01, frac


def _exact_sat(vals, sf):
    """Brute force in rational arithmetic: e = nearest integer to log2(amax/sf)
    (clamped at -30), found by scanning k with 2^k <= r < 2^(k+1) and rounding
    up iff r^2 >= 2 * 4^k; then |x| > 6 * 2^e."""
    a = max(abs(Fraction(float(v))) for v in vals)
    r = a / Fraction(float(sf))
    if r < Fraction(1, 2 ** 30):
        e = -30
    else:
        k = -31
        while Fraction(2) ** (k + 1) <= r:
            k += 1
        e = k + 1 if r * r >= 2 * Fraction(4) ** k else k
    lim = 6 * Fraction(2) ** e
    return [i for i, v in enumerate(vals) if abs(Fraction(float(v))) > lim]


def test_brute_force_tiny_blocks():
    rng = np.random.default_rng(9)
    for t in range(300):
        n = int(rng.integers(1, 33))
        vals = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20))).astype(np.float32)
        sf = float(np.float32(rng.choice([6.0, 5.0, 7.5, 9.0, 4.5, 6.0 * 2 ** -0.5 + 0.01])))
        x = _block(vals, cols=n)
        got = np.flatnonzero(_bits(oracle.mxfp4_saturation_mask(x, sf), n)[0]).tolist()
        assert got == _exact_sat(vals.tolist(), sf), (t, sf, vals)


@pytest.mark.parametrize("shape", [(2, 33), (3, 17), (4, 48, 33), (5, 64)])
def test_ragged_rows_and_tail_bits(shape):
    """Blocks restart on every row (the QDQ's per-row padding, AMCT article
    section 3.3); bits past a ragged row's end are 0."""
    x = (np.random.default_rng(1).standard_normal(shape) * 4).astype(np.float32)
    cols = shape[-1]
    m = oracle.mxfp4_saturation_mask(x, 7.0)
    rows = x.size // cols
    assert m.shape == (rows, (cols + 31) // 32)
    tail = cols % 32
    if tail:
        assert not (m[:, -1] >> np.uint32(tail)).any()
    # each row on its own gives the same words
    flat = x.reshape(rows, cols)
    for r in range(rows):
        assert np.array_equal(oracle.mxfp4_saturation_mask(flat[r:r + 1], 7.0)[0], m[r])


def test_nonfinite_block_has_no_saturated_elements():
    x = _block([100.0, np.inf, 3.0])
    assert not oracle.mxfp4_saturation_mask(x, 6.0).any()
    x = _block([100.0, np.nan])
    assert not oracle.mxfp4_saturation_mask(x, 6.0).any()


def test_ste_backward_plain_and_clipped():
    """With sf < 6/sqrt(2) nothing saturates and the clipped STE is the plain
    STE (identity, bit for bit); otherwise saturated positions become +0.0 and
    every other gradient element is passed unchanged."""
    x = mxq_inputs.mxfp4_large(64, 96, seed=2)
    gy = np.random.default_rng(4).standard_normal(x.shape).astype(np.float32)
    gy[0, :4] = [-1.5, np.inf, -np.inf, -0.0]
    m0 = oracle.mxfp4_saturation_mask(x, 4.0)
    assert np.array_equal(oracle.mxfp4_ste_backward(gy, m0).view(np.uint32), gy.view(np.uint32))
    m = oracle.mxfp4_saturation_mask(x, 6.0)
    gx = oracle.mxfp4_ste_backward(gy, m)
    sat = _bits(m, x.shape[1])
    assert sat.any() and (~sat).any()
    assert np.all(gx.view(np.uint32)[sat] == 0)  # +0.0, not -0.0
    assert np.array_equal(gx.view(np.uint32)[~sat], gy.view(np.uint32)[~sat])
