"""Pins for the MXFP4 oracle against what the pages and the mathematics fix.

Rules (AMCT FakeQuant article, section 2): blocks of 32 along the last dim;
scale = 2^round(log2(max(amax/scale_factor, 2^-30))); elements snap to the
E2M1 codebook with midpoints compared by ">=" (ties away from zero); a ragged
last dim is zero-padded per row (section 3.3).

Each check below uses a method other than the oracle's own: a high-precision
log2 (mpmath), nearest-codebook brute force with exact rationals, ml_dtypes'
E2M1 cast away from midpoints, hand-derived examples, and shape semantics.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import mxq_inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _codebook():
    g = {r[0]: [float(v) for v in r[1:]] for r in _read_golden("mxfp4_codebook.txt")}
    return g["codebook"], g["midpoints"]


# ---------------------------------------------------------------------------
# independent brute-force reference (exact rationals + 60-digit log2)
# ---------------------------------------------------------------------------

def _brute_scale_exp(amax: float, sf: float) -> int:
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    r = max(mpmath.mpf(float(amax)) / mpmath.mpf(float(sf)), mpmath.mpf(2) ** -30)
    lg = mpmath.log(r, 2)
    return int(mpmath.nint(lg))  # no tie is possible for rational r


def _brute_snap(y: Fraction) -> Fraction:
    """Nearest codebook value to y >= 0; on a tie the larger magnitude."""
    book = [Fraction(v).limit_denominator(4) for v in _codebook()[0]]
    best = None
    for c in book:
        d = abs(y - c)
        if best is None or d < best[0] or (d == best[0] and c > best[1]):
            best = (d, c)
    return best[1]


def _brute_qdq_row(row: np.ndarray, sf: float) -> np.ndarray:
    out = np.empty_like(row)
    for b0 in range(0, len(row), 32):
        blk = row[b0:b0 + 32]
        amax = float(np.max(np.abs(blk))) if len(blk) else 0.0
        e = _brute_scale_exp(amax, sf)
        s = Fraction(2) ** e
        for i, v in enumerate(blk):
            q = _brute_snap(abs(Fraction(float(v))) / s) * s
            out[b0 + i] = np.copysign(np.float32(float(q)), v)
    return out


# ---------------------------------------------------------------------------
# pages' printed constants
# ---------------------------------------------------------------------------

def test_printed_constants():
    g = {r[0]: r[1] for r in _read_golden("mxfp4_constants.txt")}
    assert int(g["block_size"]) == 32
    assert float(g["scale_factor"]) == 6.0
    # the printed decimal is 2^-30 once rounded to fp32, as its comment says
    assert np.float32(float(g["min_scale_raw"])) == np.float32(2.0 ** -30)
    # below the clamp every block gets scale 2^-30 ...
    assert oracle.mxfp4_scale_exp(0.0, 6.0) == -30
    assert oracle.mxfp4_scale_exp(6.0 * 2.0 ** -40, 6.0) == -30
    # ... and exactly at it, too
    assert oracle.mxfp4_scale_exp(6.0 * 2.0 ** -30, 6.0) == -30


def test_codebook_closure_and_decode():
    book, mids = _codebook()
    t = oracle.e2m1_decode_table()
    assert list(t[:8]) == book
    assert list(-t[8:]) == book          # sign bit is bit 3
    assert mids == [(a + b) / 2 for a, b in zip(book[:-1], book[1:])]


def test_e2m1_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    ref = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(oracle.e2m1_decode_table(), ref)


# ---------------------------------------------------------------------------
# scale decision
# ---------------------------------------------------------------------------

def test_scale_exp_vs_high_precision_log2():
    rng = np.random.default_rng(1)
    cases = []
    # random magnitudes over the fp32 range
    for _ in range(400):
        cases.append((float(np.float32(np.exp2(rng.uniform(-60, 60)))), 6.0))
    # mantissas right at the sqrt(2) boundary, where a float log2 goes wrong
    for k in range(-40, 40, 3):
        for m in (0x3504F2, 0x3504F3, 0x3504F4, 0x3504F5):
            r = np.frombuffer(np.uint32((127 + k) << 23 | m).tobytes(), np.float32)[0]
            cases.append((float(np.float32(r * np.float32(6.0))), 6.0))
            cases.append((float(r), 1.0))
    # other scale factors (scale_factor = 6 / inv_scale_factor_scale)
    for sf in (1.0, 3.0, 4.5, 7.0, 0.75, 6.0 / 1.3):
        for _ in range(40):
            cases.append((float(np.float32(np.exp2(rng.uniform(-20, 20)))), float(np.float32(sf))))
    for amax, sf in cases:
        assert oracle.mxfp4_scale_exp(amax, sf) == _brute_scale_exp(amax, sf), (amax, sf)


# ---------------------------------------------------------------------------
# element rounding
# ---------------------------------------------------------------------------

def test_rounding_matches_e2m1_cast_away_from_midpoints():
    ml = pytest.importorskip("ml_dtypes")
    _, mids = _codebook()
    rng = np.random.default_rng(2)
    y = rng.uniform(0, 7.5, 4000).astype(np.float32)
    y = y[~np.isin(y, np.float32(mids))]
    # one block per value: amax = 6 pins the scale to 2^0, so QDQ(x) = snap(x)
    for v in y[:600]:
        x = np.array([[6.0, v]], np.float32)
        got = oracle.mxfp4_qdq(x)[0, 1]
        ref = np.float32(min(float(v), 6.0)).astype(ml.float4_e2m1fn).astype(np.float32)
        assert got == ref, (v, got, ref)


def test_midpoints_round_up_in_magnitude():
    book, mids = _codebook()
    for i, m in enumerate(mids):
        x = np.array([[6.0, m, -m]], np.float32)
        got = oracle.mxfp4_qdq(x)[0]
        assert got[1] == book[i + 1] and got[2] == -book[i + 1], (m, got)


def test_saturation_beyond_top_midpoint():
    # amax/6 = 1.25 -> log2 = 0.32 -> scale 1; 7.5 >= 5 snaps to 6
    got = oracle.mxfp4_qdq(np.array([[7.5, 5.0, 4.99]], np.float32))[0]
    assert list(got) == [6.0, 6.0, 4.0]


# ---------------------------------------------------------------------------
# worked examples, derived by hand from section 2's three rules
# ---------------------------------------------------------------------------
# {1.0, 0.3, -0.1}: amax/6 = 1/6, log2 = -2.585 -> -3, s = 1/8; y = 8, 2.4, 0.8
#   -> 6 (saturated), 2, 1 -> {0.75, 0.25, -0.125}
# {6, 5, -2.9}: log2(1) = 0, s = 1; 5 is a tie -> 6; 2.9 -> 3
# {0.5, 0.2, 0}: log2(1/12) = -3.585 -> -4, s = 1/16; y = 8, 3.2, 0 -> 6, 3, 0
# {1.0, 0.74, -0.75}: s = 1/8; y = 8, 5.92, 6 -> 6, 6, 6
# {3, 1}: log2(1/2) = -1, s = 1/2; y = 6, 2 -> 6, 2
# {0, -0}: amax 0 -> clamp 2^-30; outputs keep the sign of zero
WORKED = [
    ([1.0, 0.3, -0.1], -3, [0.75, 0.25, -0.125]),
    ([6.0, 5.0, -2.9], 0, [6.0, 6.0, -3.0]),
    ([0.5, 0.2, 0.0], -4, [0.375, 0.1875, 0.0]),
    ([1.0, 0.74, -0.75], -3, [0.75, 0.75, -0.75]),
    ([3.0, 1.0], -1, [3.0, 1.0]),
    ([0.0, -0.0], -30, [0.0, -0.0]),
]


@pytest.mark.parametrize("vals,e,out", WORKED)
def test_worked_examples(vals, e, out):
    x = np.array([vals], np.float32)
    amax = float(np.max(np.abs(x)))
    assert oracle.mxfp4_scale_exp(amax, 6.0) == e
    got = oracle.mxfp4_qdq(x)[0]
    assert np.array_equal(got, np.array(out, np.float32))
    assert np.array_equal(np.signbit(got), np.signbit(np.array(out, np.float32)))
    assert np.array_equal(got, _brute_qdq_row(x[0], 6.0))


# ---------------------------------------------------------------------------
# brute force on small random inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("sf", [6.0, 4.0, 6.0 / 1.25])
def test_qdq_vs_brute_force(sf):
    x = mxq_inputs.heavy_tail((3, 70), 100.0, seed=5, zero_block_frac=0.2)
    got = oracle.mxfp4_qdq(x, sf)
    ref = np.stack([_brute_qdq_row(r, np.float32(sf)) for r in x])
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------------------
# shape semantics: per-row blocks, not flatten-then-pad
# ---------------------------------------------------------------------------

def test_ragged_shapes_are_per_row():
    shapes = [tuple(int(v) for v in r) for r in _read_golden("mxfp4_ragged_shapes.txt")]
    assert shapes == [(2, 33), (3, 17), (4, 48, 33)]
    for i, shp in enumerate(shapes):
        x = mxq_inputs.mxfp4_small(shp, seed=10 + i)
        got = oracle.mxfp4_qdq(x)
        rows = x.reshape(-1, shp[-1])
        ref = np.stack([_brute_qdq_row(r, 6.0) for r in rows]).reshape(shp)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        # flattening first would let neighbouring rows share blocks: with rows of
        # very different magnitude the shared block's scale, hence the result, differs
        z = (rows * (100.0 ** (np.arange(rows.shape[0]) % 4))[:, None]).astype(np.float32).reshape(shp)
        per_row = oracle.mxfp4_qdq(z)
        flat = oracle.mxfp4_qdq(z.reshape(1, -1)).reshape(shp)
        assert not np.array_equal(flat, per_row)


def test_closure_and_zero_blocks():
    x = mxq_inputs.mxfp4_large(64, 256, seed=3)
    y = oracle.mxfp4_qdq(x)
    book = np.array(_codebook()[0])
    for r in range(x.shape[0]):
        for b in range(0, x.shape[1], 32):
            blk, out = x[r, b:b + 32], y[r, b:b + 32]
            e = oracle.mxfp4_scale_exp(float(np.max(np.abs(blk))))
            assert np.all(np.isin(np.abs(out.astype(np.float64)) / 2.0 ** e, book))
            if not np.any(blk):
                assert not np.any(out)


def test_packed_quant_dequantizes_to_qdq():
    x = mxq_inputs.mxfp4_large(48, 160, seed=4)
    p, s = oracle.mxfp4_quant(x)
    deq = oracle.dequant_mxfp4(p, s)
    qdq = oracle.mxfp4_qdq(x)
    assert np.array_equal(deq.astype(np.float32).view(np.uint32), qdq.view(np.uint32))
    # scale byte is the biased exponent
    for r in range(0, 48, 7):
        for b in range(5):
            amax = float(np.max(np.abs(x[r, 32 * b:32 * b + 32])))
            assert s[r, b] == oracle.mxfp4_scale_exp(amax) + 127
