/*
 * mxq_oracle.c -- plain, slow CPU oracle for MX block-scaled quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's shared object.  The product
 * library (libmxq) neither links nor calls it, and the two share no code,
 * header, table or helper.
 *
 * Every floating-point step is done in binary64 on exactly-representable
 * values, so each function below is the definition of the operation written
 * out, one element at a time, with no blocking, fusion or reordering.
 *
 * Sources of the rules (web pages, cited by title and section):
 *  - "低精度训练特性（MXFP8 / HiFloat8）" (torchtitan-npu feature guide),
 *    section "线性层低精度", MXFP8 mode: blocks of 32 contiguous elements share
 *    one scale.  The pages fix no MXFP8 element/scale rule; the OCP MX rule is
 *    taken: scale exponent X = floor(log2(amax)) - 8 clamped to [-127,127]
 *    (amax == 0 -> X = -127), elements E4M3 = x * 2^-X rounded to nearest-even
 *    and saturated to +-448.
 *  - "AMCT FakeQuant 模拟伪量化工具包" article, section 2 "MXFP4 数值模型":
 *    block of 32 along the last dim, scale = 2^round(log2(max_abs/scale_factor))
 *    with max_abs/scale_factor clamped below at 2^-30 (the MIN_SCALE_RAW
 *    constant of the tiling header quoted in section 2 (3)), element codebook
 *    {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}, midpoints
 *    (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0) compared with ">=" (ties go up in
 *    magnitude), and per-row zero padding of a ragged last dimension
 *    (section 3.3, padding convention).
 *
 * Readings taken where the pages are silent:
 *  - round(log2 r) is evaluated in exact real arithmetic.  r = amax/sf is
 *    rational and log2 r is a half-integer only for irrational r, so no tie can
 *    occur and the rounding direction of "round" never matters.
 *  - non-finite blocks: an MXFP8 block whose amax is Inf or NaN gets scale byte
 *    0xFF and every code 0x7F | sign; an MXFP4 block with a non-finite amax
 *    yields NaN for every element (QDQ) and scale byte 0xFF with nibble 0x7|sign
 *    (packed).  Partly pinned by library casts and IEEE arithmetic (the scale
 *    byte, the non-finite elements' E4M3 codes, NaN on dequantization, NaN for
 *    the finite elements' QDQ); parity unpinned for the finite elements' code
 *    bytes, the non-finite element's own QDQ result and the packed nibble.
 *  - negative inputs that round to zero keep their sign (E4M3 code 0x80, QDQ
 *    output -0.0, E2M1 nibble 0x8).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 / fp32 widening                                                 */
/* ------------------------------------------------------------------ */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* E4M3 (OCP FP8 "fn": bias 7, no infinities, S.1111.111 = NaN, max 448) */
/* ------------------------------------------------------------------ */

/* Round an exact binary64 value to E4M3, nearest-even, saturating to +-448. */
uint8_t oracle_e4m3_encode(double y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    if (isnan(y))
        return (uint8_t)(sign | 0x7F);
    /* Every value >= 448 saturates: [448, 464] rounds to 448 (464 is a tie
     * and 448's mantissa 110 is even), anything above would round to 480,
     * which E4M3 cannot hold. */
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < 0x1p-6) {
        /* subnormal range: value = m * 2^-9, m in [0, 8]; m == 8 is the
         * smallest normal 2^-6 whose encoding is 0x08, i.e. also "m". */
        double m = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int k;
    (void)frexp(a, &k);      /* a = f * 2^k, f in [0.5, 1) */
    int e = k - 1;           /* floor(log2 a), in [-6, 8] */
    double mant = ldexp(a, -e);             /* in [1, 2), exact */
    double m = nearbyint((mant - 1.0) * 8.0);
    if (m == 8.0) {
        e += 1;
        m = 0.0;
    }
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (int)m));
}

double oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* ------------------------------------------------------------------ */
/* MXFP8 block scale (OCP MX rule)                                      */
/* ------------------------------------------------------------------ */

/* Returns X, the unbiased exponent of the shared scale 2^X, for a block
 * whose largest magnitude is amax (finite, >= 0). */
int oracle_mxfp8_scale_exp(double amax)
{
    if (amax == 0.0)
        return -127;
    int k;
    (void)frexp(amax, &k);
    int X = (k - 1) - 8;     /* floor(log2 amax) - 8 */
    if (X < -127)
        X = -127;
    if (X > 127)
        X = 127;
    return X;
}

/* Quantize one block of n values (already widened to binary64) with stride
 * `qs` between output codes; returns the scale byte. */
static uint8_t mxfp8_block(const double *v, int n, uint8_t *q, int64_t qs)
{
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < n; i++) {
        if (!isfinite(v[i]))
            nonfinite = 1;
        else if (fabs(v[i]) > amax)
            amax = fabs(v[i]);
    }
    if (nonfinite) {
        for (int i = 0; i < n; i++)
            q[i * qs] = (uint8_t)((signbit(v[i]) ? 0x80 : 0) | 0x7F);
        return 0xFF;
    }
    int X = oracle_mxfp8_scale_exp(amax);
    for (int i = 0; i < n; i++)
        q[i * qs] = oracle_e4m3_encode(ldexp(v[i], -X));   /* x * 2^-X, exact */
    return (uint8_t)(X + 127);
}

/* Row quant of bf16 A[R x C] (leading dim ldx, elements): blocks of 32 along
 * C.  q[r*ldq + c] gets the code, s[r*lds + b] the scale byte of block b.
 * The last block of a row holds C - 32*b < 32 elements when C % 32 != 0. */
void oracle_mxfp8_quant_rows(const uint16_t *x, int64_t R, int64_t C, int64_t ldx,
                             uint8_t *q, int64_t ldq, uint8_t *s, int64_t lds)
{
    double v[32];
    int64_t nb = (C + 31) / 32;
    for (int64_t r = 0; r < R; r++) {
        for (int64_t b = 0; b < nb; b++) {
            int n = (int)((C - 32 * b) < 32 ? (C - 32 * b) : 32);
            for (int i = 0; i < n; i++)
                v[i] = bf16_bits_to_double(x[r * ldx + 32 * b + i]);
            s[r * lds + b] = mxfp8_block(v, n, q + r * ldq + 32 * b, 1);
        }
    }
}

/* Column quant of bf16 A[R x C]: blocks of 32 along R.  The codes are
 * written transposed, qT[c*ldq + r], and the scale of rows [32b, 32b+32) of
 * column c goes to s[c*lds + b]. */
void oracle_mxfp8_quant_cols(const uint16_t *x, int64_t R, int64_t C, int64_t ldx,
                             uint8_t *qT, int64_t ldq, uint8_t *s, int64_t lds)
{
    double v[32];
    int64_t nb = (R + 31) / 32;
    for (int64_t c = 0; c < C; c++) {
        for (int64_t b = 0; b < nb; b++) {
            int n = (int)((R - 32 * b) < 32 ? (R - 32 * b) : 32);
            for (int i = 0; i < n; i++)
                v[i] = bf16_bits_to_double(x[(32 * b + i) * ldx + c]);
            s[c * lds + b] = mxfp8_block(v, n, qT + c * ldq + 32 * b, 1);
        }
    }
}

/* Column quant whose blocks restart at every group start (the per-group MX
 * quant used for the grouped weight gradient).  Group e owns rows
 * [off[e], off[e+1]) of A and is written at column offset P_e of the
 * transposed output, P_e = sum_{j<e} ceil128(off[j+1]-off[j]).  Positions of
 * qT and s that no group covers are left as the caller set them. */
void oracle_mxfp8_quant_cols_grouped(const uint16_t *x, int64_t C, int64_t ldx,
                                     const int64_t *off, int E,
                                     uint8_t *qT, int64_t ldq, uint8_t *s, int64_t lds)
{
    double v[32];
    int64_t P = 0;
    for (int e = 0; e < E; e++) {
        int64_t r0 = off[e], n_e = off[e + 1] - off[e];
        int64_t nb = (n_e + 31) / 32;
        for (int64_t c = 0; c < C; c++) {
            for (int64_t b = 0; b < nb; b++) {
                int n = (int)((n_e - 32 * b) < 32 ? (n_e - 32 * b) : 32);
                for (int i = 0; i < n; i++)
                    v[i] = bf16_bits_to_double(x[(r0 + 32 * b + i) * ldx + c]);
                s[c * lds + P / 32 + b] = mxfp8_block(v, n, qT + c * ldq + P + 32 * b, 1);
            }
        }
        P += (n_e + 127) / 128 * 128;
    }
}

/* ------------------------------------------------------------------ */
/* Scale-factor layout used by the tcgen05 block-scaled MMA             */
/* ------------------------------------------------------------------ */

/* Scatter a logical scale matrix L[rows x kb] (leading dim ld) into the
 * block-scaled operand layout: rows padded to 128, scale columns padded to 4,
 * tiles of 128 rows x 4 columns stored as 512 contiguous bytes, tile (i, j)
 * at index i * (kb_pad/4) + j, and inside a tile element (r, c) at byte
 * 16*(r%32) + 4*(r/32) + c.  Padding bytes are 0. */
void oracle_swizzle_scales(const uint8_t *L, int64_t rows, int64_t kb, int64_t ld,
                           uint8_t *out)
{
    int64_t rows_pad = (rows + 127) / 128 * 128;
    int64_t kb_pad = (kb + 3) / 4 * 4;
    memset(out, 0, (size_t)(rows_pad * kb_pad));
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < kb; c++) {
            int64_t tile = (r / 128) * (kb_pad / 4) + c / 4;
            int64_t off = tile * 512 + 16 * (r % 32) + 4 * ((r % 128) / 32) + (c % 4);
            out[off] = L[r * ld + c];
        }
}

/* ------------------------------------------------------------------ */
/* MXFP4 (E2M1 elements, E8M0 power-of-two block scale)                */
/* ------------------------------------------------------------------ */

static const double kE2M1Mid[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
static const double kE2M1Val[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* e = round(log2(max(amax/sf, 2^-30))) in exact arithmetic. */
int oracle_mxfp4_scale_exp(double amax, double sf)
{
    if (!(amax > 0.0))
        return -30;                     /* amax/sf = 0 is clamped to 2^-30 */
    int ka, ks;
    double fa = frexp(amax, &ka), fs = frexp(sf, &ks);
    /* amax/sf = (fa/fs) * 2^(ka-ks) with fa/fs in (1/2, 2) */
    int e0 = (ka - ks) + (fa >= fs ? 0 : -1);   /* floor(log2(amax/sf)) */
    if (e0 < -30)
        return -30;                     /* amax/sf < 2^-30: clamp */
    /* log2(amax/sf) in [e0, e0+1); it rounds up iff amax/sf >= sqrt(2)*2^e0,
     * i.e. amax^2 >= 2 * sf^2 * 4^e0.  Both sides are exact in binary64
     * (24-bit significands squared, power-of-two scaling). */
    double lhs = amax * amax;
    double rhs = ldexp(sf * sf, 2 * e0 + 1);
    int e = (lhs >= rhs) ? e0 + 1 : e0;
    /* Reading: capped at 2^127, the largest power of two an E8M0 byte holds
     * (reached only when amax/sf > 2^126.5, i.e. scale_factor < ~2.8 with
     * amax near the fp32 maximum; the pages give no upper clamp). */
    return e > 127 ? 127 : e;
}

/* Index into the E2M1 codebook of |x| / 2^e: the number of midpoints <= y. */
static int e2m1_index(double ax, int e)
{
    double y = ldexp(ax, -e);           /* exact */
    int i = 0;
    while (i < 7 && y >= kE2M1Mid[i])
        i++;
    return i;
}

/* Quantize-dequantize fp32 x[rows x cols] (row-major, last dim = cols) to
 * MXFP4 with blocks of 32 restarting on every row. */
void oracle_mxfp4_qdq(const float *x, float *y, int64_t rows, int64_t cols, float sf)
{
    int64_t nb = (cols + 31) / 32;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            int64_t c0 = 32 * b, c1 = (c0 + 32 < cols) ? c0 + 32 : cols;
            double amax = 0.0;
            int nonfinite = 0;
            for (int64_t c = c0; c < c1; c++) {
                double v = x[r * cols + c];
                if (!isfinite(v))
                    nonfinite = 1;
                else if (fabs(v) > amax)
                    amax = fabs(v);
            }
            if (nonfinite) {
                for (int64_t c = c0; c < c1; c++)
                    y[r * cols + c] = NAN;
                continue;
            }
            int e = oracle_mxfp4_scale_exp(amax, (double)sf);
            for (int64_t c = c0; c < c1; c++) {
                double v = x[r * cols + c];
                double out = kE2M1Val[e2m1_index(fabs(v), e)] * ldexp(1.0, e);
                y[r * cols + c] = (float)copysign(out, v);
            }
        }
    }
}

/* Packed MXFP4 quant of fp32 x[rows x cols] (cols even): nibble of element
 * (r, c) goes to p[r*ldp + c/2], low nibble for even c; nibble = sign<<3 |
 * codebook index.  s[r*lds + b] = e + 127. */
void oracle_mxfp4_quant(const float *x, int64_t rows, int64_t cols, int64_t ldx, float sf,
                        uint8_t *p, int64_t ldp, uint8_t *s, int64_t lds)
{
    int64_t nb = (cols + 31) / 32;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            int64_t c0 = 32 * b, c1 = (c0 + 32 < cols) ? c0 + 32 : cols;
            double amax = 0.0;
            int nonfinite = 0;
            for (int64_t c = c0; c < c1; c++) {
                double v = x[r * ldx + c];
                if (!isfinite(v))
                    nonfinite = 1;
                else if (fabs(v) > amax)
                    amax = fabs(v);
            }
            int e = nonfinite ? 0 : oracle_mxfp4_scale_exp(amax, (double)sf);
            s[r * lds + b] = nonfinite ? 0xFF : (uint8_t)(e + 127);
            for (int64_t c = c0; c < c1; c++) {
                double v = x[r * ldx + c];
                int nib = (signbit(v) ? 8 : 0) | (nonfinite ? 7 : e2m1_index(fabs(v), e));
                uint8_t *dst = p + r * ldp + c / 2;
                if (c % 2 == 0)
                    *dst = (uint8_t)((*dst & 0xF0) | nib);
                else
                    *dst = (uint8_t)((*dst & 0x0F) | (nib << 4));
            }
        }
    }
}

/* Saturation mask of MXFP4 quant-dequant ("AMCT FakeQuant" article, section
 * 4.1 "STE 与 clipped STE"): element x of a block with scale 2^e is saturated
 * when |x| > 6 * 2^e, i.e. when the codebook's top value 6 had to clip it.
 * Packed as one 32-bit word per block: mask[r*nb + b] bit i is element
 * (r, 32b + i); bits past the end of a ragged row are 0.  Reading: a block
 * with a non-finite element has an Inf/NaN scale, so |x| > 6*scale is false
 * for all of its elements and its word is 0. */
void oracle_mxfp4_saturation_mask(const float *x, int64_t rows, int64_t cols, float sf, uint32_t *mask)
{
    int64_t nb = (cols + 31) / 32;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            int64_t c0 = 32 * b, c1 = (c0 + 32 < cols) ? c0 + 32 : cols;
            double amax = 0.0;
            int nonfinite = 0;
            for (int64_t c = c0; c < c1; c++) {
                double v = x[r * cols + c];
                if (!isfinite(v))
                    nonfinite = 1;
                else if (fabs(v) > amax)
                    amax = fabs(v);
            }
            uint32_t word = 0;
            if (!nonfinite) {
                double limit = 6.0 * ldexp(1.0, oracle_mxfp4_scale_exp(amax, (double)sf));
                for (int64_t c = c0; c < c1; c++)
                    if (fabs((double)x[r * cols + c]) > limit)
                        word |= 1u << (c - c0);
            }
            mask[r * nb + b] = word;
        }
    }
}

/* Clipped straight-through estimator, backward (same section): the gradient
 * passes through unchanged except at saturated elements, where it is set to
 * +0.0 (a masked fill with zero). */
void oracle_mxfp4_ste_backward(const float *gy, const uint32_t *mask, int64_t rows, int64_t cols, float *gx)
{
    int64_t nb = (cols + 31) / 32;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            int sat = (mask[r * nb + c / 32] >> (c % 32)) & 1u;
            gx[r * cols + c] = sat ? 0.0f : gy[r * cols + c];
        }
}

double oracle_e2m1_decode(uint8_t nib)
{
    double v = kE2M1Val[nib & 7];
    return (nib & 8) ? -v : v;
}
