// mxq_quant.cu -- single-pass MX quantization kernels (HBM-bound).
//
// MXFP8 ("低精度训练特性（MXFP8 / HiFloat8）", section "线性层低精度", MXFP8 mode:
// blocks of 32 elements share one scale) with the OCP MX rule: scale 2^X,
// X = floor(log2 amax) - 8 clamped to [-127, 127] (-127 for an all-zero
// block), codes E4M3(x * 2^-X) by cvt.rn.satfinite (nearest-even, saturating
// to +-448).  MXFP4 ("AMCT FakeQuant 模拟伪量化工具包", section 2): scale
// 2^round(log2(max(amax/sf, 2^-30))) decided exactly with integer arithmetic,
// elements snapped to the E2M1 codebook with midpoints rounding away from zero.
//
// Layout of the work: a CTA owns a 128 x 128 tile of the input, which makes
// exactly one 512-byte scale tile per output axis, so scales are staged in
// shared memory and written with coalesced 16-byte stores directly in the
// tcgen05 block-scale layout.  Data moves with 16-byte vector loads/stores;
// the column (transposed) output goes through a shared-memory copy of the tile
// read back as 32-bit column pairs (conflict-free).
#include <cuda_bf16.h>
#include <cstdint>
#include <mutex>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;

// 32 bytes in one load; p must be 32-byte aligned.
__device__ __forceinline__ void ldg_nc_v8(const void *p, uint4 &a, uint4 &b) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void stg_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// 32 bytes in one store (a whole L2 sector); p must be 32-byte aligned.
__device__ __forceinline__ void stg_v8(void *p, uint4 a, uint4 b) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w),
                 "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// Four fp32 values -> four E4M3 codes (a in the low byte); the two halves are
// packed by register pairing.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- MXFP8 scale
// X from the magnitude bits of a bf16 amax; 128 marks a non-finite block.
__device__ __forceinline__ int mx8_exp_from_bf16(uint32_t a) {
    if (a >= 0x7F80u) return 128;
    if (a == 0) return -127;
    const int E = static_cast<int>(a >> 7);
    const int fl = E ? E - 127 : -133 + (31 - __clz(static_cast<int>(a)));
    return max(fl - 8, -127);  // fl <= 127 so X <= 119
}
__device__ __forceinline__ uint8_t mx8_scale_byte(int X) { return X > 127 ? 0xFF : static_cast<uint8_t>(X + 127); }
// 2^-X as a bf16 bit pattern (normal for X in [-127, 119]).
__device__ __forceinline__ uint32_t pow2_neg_bf16(int X) { return static_cast<uint32_t>(127 - X) << 7; }
// Two bf16 products in one instruction.  x * 2^-X is exact in bf16 whenever
// it is at least 2^-126; smaller products round to E4M3 zero either way, so
// the codes equal those of the exact product.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// E4M3 codes of 8 bf16 (4 packed words, element 2k in the low half of word k).
__device__ __forceinline__ uint2 e4m3_codes8(const uint32_t (&w)[4], int X) {
    uint2 out;
    if (X > 127) {  // non-finite block: every code NaN, sign kept
        uint32_t b[8];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            b[2 * k] = 0x7Fu | ((w[k] >> 8) & 0x80u);
            b[2 * k + 1] = 0x7Fu | ((w[k] >> 24) & 0x80u);
        }
        out.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
        out.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
        return out;
    }
    const uint32_t inv2 = pow2_neg_bf16(X) * 0x00010001u;
    const uint32_t s0 = mul_bf16x2(w[0], inv2), s1 = mul_bf16x2(w[1], inv2);
    const uint32_t s2 = mul_bf16x2(w[2], inv2), s3 = mul_bf16x2(w[3], inv2);
    out.x = e4m3x4(bf16lo(s0), bf16hi(s0), bf16lo(s1), bf16hi(s1));
    out.y = e4m3x4(bf16lo(s2), bf16hi(s2), bf16lo(s3), bf16hi(s3));
    return out;
}

// Max over the 8 bf16 magnitudes of a 16-byte chunk (integer compare of |bits|).
__device__ __forceinline__ uint32_t amax8_bf16(const uint32_t (&w)[4]) {
    const uint32_t m = 0x7FFF7FFFu;
    const uint32_t t = __vmaxu2(__vmaxu2(w[0] & m, w[1] & m), __vmaxu2(w[2] & m, w[3] & m));
    return max(t & 0xFFFFu, t >> 16);
}

// ---------------------------------------------------------------- MXFP4 scale
// e = round(log2(max(amax/sf, 2^-30))) exactly, capped at 127; amax finite
// >= 0, sf finite > 0.
__device__ __forceinline__ int mx4_exp(float amax, float sf) {
    if (amax == 0.0f) return -30;
    const uint32_t ab = __float_as_uint(amax), sb = __float_as_uint(sf);
    int ea = static_cast<int>(ab >> 23), es = static_cast<int>(sb >> 23);
    uint32_t ma = ab & 0x7FFFFFu, ms = sb & 0x7FFFFFu;
    // value = M * 2^(e-150) with M in [2^23, 2^24)
    if (ea == 0) { const int sh = __clz(static_cast<int>(ma)) - 8; ma <<= sh; ea = 1 - sh; } else { ma |= 0x800000u; }
    if (es == 0) { const int sh = __clz(static_cast<int>(ms)) - 8; ms <<= sh; es = 1 - sh; } else { ms |= 0x800000u; }
    const int d = ma < ms ? 1 : 0;
    const int e0 = ea - es - d;                       // floor(log2(amax/sf))
    if (e0 < -30) return -30;                         // clamp at 2^-30
    // q = (ma/ms) * 2^d in [1, 2) is amax/sf / 2^e0: round up iff q^2 >= 2
    const unsigned long long lhs = (static_cast<unsigned long long>(ma) * ma) << (2 * d);
    const unsigned long long rhs = 2ull * ms * ms;
    const int e = lhs >= rhs ? e0 + 1 : e0;
    return min(e, 127);
}
// The MXFP4 element rule ("AMCT FakeQuant 模拟伪量化工具包", section 2) in the
// input's own scale.  With the block scale s = 2^e, an element's magnitude
// y = |x| / s is snapped to the codebook {0, .5, 1, 1.5, 2, 3, 4, 6}, a
// midpoint going up.  Above 1 the codebook is every value with one mantissa
// bit, so snapping there is rounding |x|'s mantissa to one bit, half away from
// zero: add half of bit 22 and clear the bits below it -- the exponent is
// untouched, so no division by s is needed -- then clamp at 6 s.  Below s the
// two midpoints 0.25 s and 0.75 s decide between 0, s/2 and s.  Everything is
// integer arithmetic on the fp32 bit patterns of non-negative values, whose
// order is the order of the values (an overflow to +inf included).
struct Mx4Blk {
    uint32_t s, half_s, t025, t075, six_s;  // fp32 bits of s, s/2, s/4, 3s/4, 6s (+inf when 6s overflows)
    int e;
};
__device__ __forceinline__ Mx4Blk mx4_block(int e) {  // e in [-30, 127]
    Mx4Blk B;
    B.e = e;
    B.s = static_cast<uint32_t>(e + 127) << 23;
    B.half_s = static_cast<uint32_t>(e + 126) << 23;
    B.t025 = static_cast<uint32_t>(e + 125) << 23;
    B.t075 = B.half_s | 0x400000u;
    B.six_s = e <= 125 ? (static_cast<uint32_t>(e + 129) << 23) | 0x400000u : 0x7F800000u;
    return B;
}
// |x| snapped to (codebook value) x s, as fp32 bits; ax = |x|'s bits, finite.
__device__ __forceinline__ uint32_t mx4_snap(uint32_t ax, const Mx4Blk &B) {
    const uint32_t r = min((ax + 0x200000u) & 0xFFC00000u, B.six_s);
    const uint32_t lo = ax >= B.t075 ? B.s : (ax >= B.t025 ? B.half_s : 0u);
    return ax >= B.s ? r : lo;
}
// Codebook index (0..7) of the snapped magnitude: above s, the rounded bits
// hold value 2^k (1 + m/2) x s, index 2 + 2 k + m.
__device__ __forceinline__ uint32_t mx4_index(uint32_t ax, const Mx4Blk &B) {
    const uint32_t r = min((ax + 0x200000u) & 0xFFC00000u, B.six_s);
    const uint32_t lo = ax >= B.t075 ? 2u : (ax >= B.t025 ? 1u : 0u);
    return ax >= B.s ? (r >> 22) - static_cast<uint32_t>(2 * B.e + 252) : lo;
}
// E4M3 code of the snapped magnitude's codebook value (0.5 -> 0x30, 1 -> 0x38,
// ..., 6 -> 0x4C): above s it is the rounded bits' exponent and top mantissa
// bit, rebased from the fp32 bias 127 + e to the E4M3 bias 7.
__device__ __forceinline__ uint32_t mx4_e4m3_code(uint32_t ax, const Mx4Blk &B) {
    const uint32_t r = min((ax + 0x200000u) & 0xFFC00000u, B.six_s);
    const uint32_t lo = ax >= B.t075 ? 0x38u : (ax >= B.t025 ? 0x30u : 0u);
    return ax >= B.s ? (r >> 20) - static_cast<uint32_t>(0x3C0 + 8 * B.e) : lo;
}
// The same rule through the hardware E2M1 conversion, which rounds to nearest
// with ties to the even code and saturates at +-6: it agrees with the rule
// everywhere but on the midpoints whose lower neighbour is the even code --
// y = 1/4 and y = 1.25 x 2^k (k = 0, 1, 2: 1.25, 2.5, 5) -- where the rule
// goes up.  Moving |x| one ulp up exactly there (x's bits + 1; the scaled
// value is then no longer a tie) makes the conversion go up too; elsewhere
// the ulp moves no value across a midpoint, since every midpoint is an fp32
// value of that exponent.  y = x 2^-e is exact (a power-of-two scaling; a
// result too small for a normal fp32 rounds to zero either way).
__device__ __forceinline__ float mx4_scaled(uint32_t xb, uint32_t t025, float inv_s) {
    const bool tie = (xb & 0x7FFFFFu) == 0x200000u || (xb & 0x7FFFFFFFu) == t025;
    return __uint_as_float(xb + (tie ? 1u : 0u)) * inv_s;
}
// For bf16 inputs no tie fix-up is needed: a bf16 value has 8 significant
// bits, so |x| * 2^-e * (1 + 2^-9) is exact in fp32 and lies strictly above y
// exactly when y is a midpoint, and it never reaches the next midpoint from a
// bf16 value below one (those are at least m * 2^-8 under the midpoint m, the
// nudge is at most m * 2^-9).  One multiply per element takes the place of
// mx4_untie2; the factor is exact too (a power of two times 1 + 2^-9).
constexpr float kBf16Nudge = 1.001953125f;  // 1 + 2^-9
// 2^-e for a block exponent e in [-30, 127] (2^-127 is a subnormal).
__device__ __forceinline__ float mx4_inv_scale(int e) {
    return __uint_as_float(e <= 126 ? static_cast<uint32_t>(127 - e) << 23 : 0x00400000u);
}
// E2M1 codes (sign | index) of two scaled values: lo in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u16.u8 %0, b;\n\t}" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// bf16 pair of the rule's values of two scaled values lo, hi (RNE E2M1
// conversion, tie-fixed inputs) times 2^e: lo in the low half (exact: a
// codebook value times a power of two).
__device__ __forceinline__ uint32_t e2m1_qdq_bf16x2(float lo, float hi, float s) {
    float f0, f1;
    asm("{\n\t.reg .b8 b;\n\t.reg .b32 h;\n\t.reg .f16 a0, a1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b, %3, %2;\n\t"
        "cvt.rn.f16x2.e2m1x2 h, b;\n\t"
        "mov.b32 {a0, a1}, h;\n\t"
        "cvt.f32.f16 %0, a0;\n\t"
        "cvt.f32.f16 %1, a1;\n\t}"
        : "=f"(f0), "=f"(f1) : "f"(lo), "f"(hi));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f1 * s), "f"(f0 * s));
    return r;
}
// ============================================================================
// Row quant: 128 x 128 tile per CTA, blocks along cols (cols % 32 == 0).
//   FMT 0: bf16 -> E4M3 codes [R x C] (MXFP8)
//   FMT 1: bf16/fp32 -> packed E2M1 nibbles [R x C/2] (MXFP4)
//   FMT 2: bf16 -> MXFP4 values written as E4M3 codes [R x C]: every E2M1
//          value is an E4M3 value, so with the same E8M0 scale the MXFP8
//          block-scaled MMA multiplies exactly the MXFP4 quant-dequant.
// MXFP4 formats take the scale factor sf (6 by default).
// Each thread owns 8 chunks of 8 elements; 4 lanes form one 32-block.
// ============================================================================
// E4M3 codes of the MXFP4 values of 8 bf16 (4 packed words, element 2k in the
// low half of word k) under block B: sign | the E4M3 code of the E2M1 value;
// the NaN code 0x7F | sign for a non-finite block.
__device__ __forceinline__ uint2 mx4_as_e4m3_codes8(const uint32_t (&w)[4], const Mx4Blk &B, bool nonfinite) {
    // the signs: bit 7 of byte k <- bit 15 of element k's bf16
    const uint32_t sg0 = __byte_perm(w[0], w[1], 0x7531) & 0x80808080u;
    const uint32_t sg1 = __byte_perm(w[2], w[3], 0x7531) & 0x80808080u;
    if (nonfinite) return make_uint2(0x7F7F7F7Fu | sg0, 0x7F7F7F7Fu | sg1);
    const float f = mx4_inv_scale(B.e) * kBf16Nudge;
    uint32_t nb[4];  // E2M1 indices (no sign) of elements 2k, 2k + 1 in the low byte
#pragma unroll
    for (int k = 0; k < 4; k++)
        nb[k] = cvt_e2m1x2(__uint_as_float((w[k] & 0x7FFFu) << 16) * f, __uint_as_float(w[k] & 0x7FFF0000u) * f);
    // E4M3 code of E2M1 index i (value 0, .5, 1, 1.5, 2, 3, 4, 6): byte i of
    // the 8-byte table {kLo, kHi}, picked by a byte permute whose selector
    // nibbles are the indices
    constexpr uint32_t kLo = 0x3C383000u, kHi = 0x4C484440u;
    const uint32_t c0 = __byte_perm(kLo, kHi, (nb[0] | (nb[1] << 8)) & 0x7777u);
    const uint32_t c1 = __byte_perm(kLo, kHi, (nb[2] | (nb[3] << 8)) & 0x7777u);
    return make_uint2(c0 | sg0, c1 | sg1);
}

template <typename InT, int FMT>
__global__ void __launch_bounds__(kThreads) k_quant_rows(const InT *__restrict__ x, int64_t R, int64_t C,
                                                         int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                         uint8_t *__restrict__ s, int64_t kb_tiles, float sf,
                                                         unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    // buffer extents in bytes (checked by debug builds)
    const uint64_t x_bytes = static_cast<uint64_t>((R - 1) * ldx + C) * sizeof(InT);
    const uint64_t q_bytes = static_cast<uint64_t>(R * ldq), s_bytes = static_cast<uint64_t>((R + 127) / 128 * kb_tiles * 512);
    (void)x_bytes; (void)q_bytes; (void)s_bytes; (void)err;
    __shared__ __align__(16) uint8_t satom[512];
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTile, c0 = static_cast<int64_t>(blockIdx.x) * kTile;
    // all of this thread's loads first (8 or 16 x 16 B in flight), then compute
    constexpr int kVec = sizeof(InT) == 4 ? 2 : 1;
    // fp32 rows: one 32-byte load per 8 elements where x is 32-byte aligned (ldx % 8 == 0)
    const bool al32 = kVec == 2 && (reinterpret_cast<uintptr_t>(x) & 31) == 0;
    uint4 v[8][kVec];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int id = tid + kThreads * i;
        const int64_t gr = r0 + (id >> 4), gc = c0 + (id & 15) * 8;
#pragma unroll
        for (int h = 0; h < kVec; h++) v[i][h] = make_uint4(0, 0, 0, 0);
        if (gr < R && gc < C && MXQ_IN_BOUNDS(x + gr * ldx + gc, 8 * sizeof(InT), x, x_bytes, err)) {
            const InT *src = x + gr * ldx + gc;
            if (kVec == 2 && al32) {
                ldg_nc_v8(src, v[i][0], v[i][kVec - 1]);
            } else {
#pragma unroll
                for (int h = 0; h < kVec; h++) v[i][h] = ldg_nc_v4(reinterpret_cast<const uint32_t *>(src) + 4 * h);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int id = tid + kThreads * i;
        const int row = id >> 4, ch = id & 15, col = ch * 8;
        const int64_t gr = r0 + row, gc = c0 + col;
        const bool valid = gr < R && gc < C;
        uint32_t w[8] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w, 0, 0, 0, 0};  // bf16: 4 words; fp32: 8
        if (kVec == 2) {
            w[4] = v[i][kVec - 1].x; w[5] = v[i][kVec - 1].y; w[6] = v[i][kVec - 1].z; w[7] = v[i][kVec - 1].w;
        }
        uint8_t sbyte;
        if (FMT == 0) {
            const uint32_t (&w4)[4] = *reinterpret_cast<const uint32_t(*)[4]>(w);
            uint32_t a = amax8_bf16(w4);
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const int X = mx8_exp_from_bf16(a);
            sbyte = mx8_scale_byte(X);
            if (valid && MXQ_IN_BOUNDS(q + gr * ldq + gc, 8, q, q_bytes, err)) {
                const uint2 codes = e4m3_codes8(w4, X);
                asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(q + gr * ldq + gc), "r"(codes.x), "r"(codes.y)
                             : "memory");
            }
        } else {
            float v[8];
            uint32_t a = 0;
            if (sizeof(InT) == 2) {
#pragma unroll
                for (int k = 0; k < 4; k++) { v[2 * k] = bf16lo(w[k]); v[2 * k + 1] = bf16hi(w[k]); }
            } else {
#pragma unroll
                for (int k = 0; k < 8; k++) v[k] = __uint_as_float(w[k]);
            }
#pragma unroll
            for (int k = 0; k < 8; k++) a = max(a, __float_as_uint(v[k]) & 0x7FFFFFFFu);
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const bool nonfinite = a >= 0x7F800000u;
            const int e = nonfinite ? 0 : mx4_exp(__uint_as_float(a), sf);
            sbyte = nonfinite ? 0xFF : static_cast<uint8_t>(e + 127);
            const Mx4Blk B = mx4_block(e);
            if (FMT == 1) {
                uint32_t packed = 0;
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t bits = __float_as_uint(v[k]);
                    const uint32_t idx = nonfinite ? 7u : mx4_index(bits & 0x7FFFFFFFu, B);
                    const uint32_t nib = ((bits >> 28) & 8u) | idx;
                    packed |= nib << (4 * k);
                }
                if (valid && MXQ_IN_BOUNDS(q + gr * ldq + gc / 2, 4, q, q_bytes, err)) {
                    asm volatile("st.global.u32 [%0], %1;" ::"l"(q + gr * ldq + gc / 2), "r"(packed) : "memory");
                }
            } else {
                // E4M3 byte: sign | code of the E2M1 value; a non-finite block
                // gets the NaN code 0x7F | sign under scale byte 0xFF
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t bits = __float_as_uint(v[k]);
                    const uint32_t mag = nonfinite ? 0x7Fu : mx4_e4m3_code(bits & 0x7FFFFFFFu, B);
                    const uint32_t code = ((bits >> 24) & 0x80u) | mag;
                    if (k < 4) lo |= code << (8 * k);
                    else hi |= code << (8 * (k - 4));
                }
                if (valid && MXQ_IN_BOUNDS(q + gr * ldq + gc, 8, q, q_bytes, err)) {
                    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(q + gr * ldq + gc), "r"(lo), "r"(hi)
                                 : "memory");
                }
            }
        }
        if (!valid) sbyte = 0;  // padding rows / blocks of the scale tile
        if ((lane & 3) == 0) satom[16 * (row & 31) + 4 * (row >> 5) + (ch >> 2)] = sbyte;
    }
    __syncthreads();
    if (tid < 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(satom + 16 * tid);
        uint8_t *dst = s + (static_cast<int64_t>(blockIdx.y) * kb_tiles + blockIdx.x) * 512 + 16 * tid;
        if (MXQ_IN_BOUNDS(dst, 16, s, s_bytes, err)) stg_v4(dst, v);
    }
}

// ============================================================================
// Column quant (optionally dual): 128 x 128 bf16 tile per CTA.
//   ROWS:    also emit the row quant (dual-axis, one read of x).
//   GROUPED: tile rows come from one group of a per-group column quant; the
//            padded tile index selects the group, blocks restart at the
//            group start and padding rows are zero.
// The column pass: thread (p, b) = (column pair 0..63, 32-row block 0..3)
// reads 32 words of the shared tile, one per row.
// ============================================================================
struct ColParams {
    const uint16_t *x;
    int64_t R, C, ldx;
    uint8_t *q_row;      // [R x C]               (ROWS)
    uint8_t *s_row;      // swz(R, C/32)           (ROWS)
    int64_t kb_row_tiles;
    uint8_t *qT;         // [C x ldqT]
    uint8_t *sT;         // swz(C, ldqT/32)
    int64_t ldqT;
    int64_t kb_col_tiles;
    const int64_t *offsets;  // GROUPED: E+1 device offsets
    int E;
    int row_pad;             // GROUPED with ROWS: row scales in the per-group padded layout swz(ldqT, C/32)
    float sf;                // MXFP4 scale factor (row pass in FMT 2)
    unsigned int *err;       // device error word (malformed offsets; debug-build bounds checks)
};

// Extents in bytes of the buffers of a column (dual, grouped) quant, checked
// by debug builds.
struct ColExtents {
    uint64_t x, q_row, s_row, qT, sT;
};
__device__ __forceinline__ ColExtents col_extents(const ColParams &P) {
    ColExtents e;
    e.x = P.R > 0 ? static_cast<uint64_t>((P.R - 1) * P.ldx + P.C) * 2 : 0;
    e.q_row = static_cast<uint64_t>(P.R * P.C);
    e.s_row = static_cast<uint64_t>(((P.row_pad ? P.ldqT : P.R) + 127) / 128 * P.kb_row_tiles * 512);
    e.qT = static_cast<uint64_t>(P.C * P.ldqT);
    e.sT = static_cast<uint64_t>((P.C + 127) / 128 * P.kb_col_tiles * 512);
    return e;
}

template <bool ROWS, bool GROUPED>
__global__ void __launch_bounds__(kThreads) k_quant_cols(ColParams P) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    __shared__ __align__(16) uint8_t tile[kTile * kTile * 2];
    __shared__ __align__(16) uint8_t srow_atom[512];
    __shared__ __align__(16) uint8_t scol_atom[512];
    __shared__ int64_t sh_src0;
    __shared__ int sh_nvalid;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t rt = blockIdx.y, ct = blockIdx.x;
    const int64_t c0 = ct * kTile;
    const ColExtents ext = col_extents(P);
    (void)ext;
    int64_t src0 = rt * kTile;  // first source row of the tile
    int nvalid;                 // rows of the tile that hold data
    if (GROUPED) {
        // malformed offsets: this CTA reads and writes nothing
        __shared__ int sh_bad;
        if (warp == 0) {
            const bool good = group_offsets_valid(P.offsets, P.E, P.R, lane);
            if (lane == 0) {
                sh_bad = good ? 0 : 1;
                if (!good) atomicOr(P.err, kErrBadOffsets);
            }
        }
        __syncthreads();
        if (sh_bad) return;
        if (tid == 0) sh_nvalid = 0;
        __syncwarp();
        if (warp == 0) {
            const int64_t t0 = rt * kTile;  // padded row of the tile
            int64_t run = 0;
            for (int base = 0; base < P.E; base += 32) {
                const int e = base + lane;
                int64_t n = 0;
                if (e < P.E) n = P.offsets[e + 1] - P.offsets[e];
                const int64_t padn = (n + 127) / 128 * 128;
                int64_t incl = padn;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const int64_t start = run + incl - padn;
                if (e < P.E && padn > 0 && t0 >= start && t0 < start + padn) {
                    sh_src0 = P.offsets[e] + (t0 - start);
                    const int64_t left = n - (t0 - start);
                    sh_nvalid = static_cast<int>(left < kTile ? left : kTile);
                }
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        __syncthreads();
        src0 = sh_src0;
        nvalid = sh_nvalid;
    } else {
        const int64_t left = P.R - src0;
        nvalid = static_cast<int>(left < kTile ? left : kTile);
    }

    // ---- load the tile (and the row quant) ----
    // all 8 of this thread's 16-byte loads first, then compute
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int id = tid + kThreads * i;
        const int row = id >> 4;
        const int64_t gc = c0 + (id & 15) * 8;
        v[i] = make_uint4(0, 0, 0, 0);
        if (row < nvalid && gc < P.C && MXQ_IN_BOUNDS(P.x + (src0 + row) * P.ldx + gc, 16, P.x, ext.x, P.err))
            v[i] = ldg_nc_v4(P.x + (src0 + row) * P.ldx + gc);
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int id = tid + kThreads * i;
        const int row = id >> 4, ch = id & 15, col = ch * 8;
        const int64_t gc = c0 + col;
        const bool valid = row < nvalid && gc < P.C;
        uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        if (ROWS) {
            uint32_t a = amax8_bf16(w);
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const int X = mx8_exp_from_bf16(a);
            if (valid && MXQ_IN_BOUNDS(P.q_row + (src0 + row) * P.C + gc, 8, P.q_row, ext.q_row, P.err)) {
                const uint2 codes = e4m3_codes8(w, X);
                asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(P.q_row + (src0 + row) * P.C + gc),
                             "r"(codes.x), "r"(codes.y)
                             : "memory");
            }
            if ((lane & 3) == 0) srow_atom[16 * (row & 31) + 4 * (row >> 5) + (ch >> 2)] = mx8_scale_byte(X);
        }
        *reinterpret_cast<uint4 *>(tile + row * (kTile * 2) + ch * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();

    // ---- column pass ----
    {
        const int p = tid & 63, b = tid >> 6;  // column pair, 32-row block
        uint32_t col[32];
#pragma unroll
        for (int i = 0; i < 32; i++) col[i] = *reinterpret_cast<const uint32_t *>(tile + (32 * b + i) * (kTile * 2) + 4 * p);
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 32; i++) m2 = __vmaxu2(m2, col[i] & 0x7FFF7FFFu);
        const int Xlo = mx8_exp_from_bf16(m2 & 0xFFFFu), Xhi = mx8_exp_from_bf16(m2 >> 16);
        const int cl = 2 * p, ch2 = 2 * p + 1;
        scol_atom[16 * (cl & 31) + 4 * (cl >> 5) + b] = mx8_scale_byte(Xlo);
        scol_atom[16 * (ch2 & 31) + 4 * (ch2 >> 5) + b] = mx8_scale_byte(Xhi);

        const int64_t gcol = c0 + cl;
        if (gcol < P.C) {
            uint32_t lo[8], hi[8];
            // column 2p's scale in the low half, column 2p + 1's in the high half
            const uint32_t inv2 = pow2_neg_bf16(Xlo > 127 ? 0 : Xlo) | (pow2_neg_bf16(Xhi > 127 ? 0 : Xhi) << 16);
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const uint32_t a0 = mul_bf16x2(col[4 * k], inv2), a1 = mul_bf16x2(col[4 * k + 1], inv2);
                const uint32_t a2 = mul_bf16x2(col[4 * k + 2], inv2), a3 = mul_bf16x2(col[4 * k + 3], inv2);
                lo[k] = e4m3x4(bf16lo(a0), bf16lo(a1), bf16lo(a2), bf16lo(a3));
                hi[k] = e4m3x4(bf16hi(a0), bf16hi(a1), bf16hi(a2), bf16hi(a3));
            }
            if (Xlo > 127 || Xhi > 127) {  // non-finite blocks: NaN codes with the sign kept
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    uint32_t sl = 0, sh = 0;
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        sl |= (0x7Fu | ((col[4 * k + j] >> 8) & 0x80u)) << (8 * j);
                        sh |= (0x7Fu | ((col[4 * k + j] >> 24) & 0x80u)) << (8 * j);
                    }
                    if (Xlo > 127) lo[k] = sl;
                    if (Xhi > 127) hi[k] = sh;
                }
            }
            const int64_t pos = rt * kTile + 32 * b;  // first output column (token) of the block
            uint8_t *dlo = P.qT + gcol * P.ldqT + pos;
            uint8_t *dhi = dlo + P.ldqT;
            const int64_t limit = GROUPED ? P.ldqT : P.R;  // grouped tiles write padding zeros too
            if (pos < limit && (!MXQ_IN_BOUNDS(dlo, limit - pos < 32 ? limit - pos : 32, P.qT, ext.qT, P.err) ||
                                !MXQ_IN_BOUNDS(dhi, limit - pos < 32 ? limit - pos : 32, P.qT, ext.qT, P.err))) {
            } else if (pos + 32 <= limit && (P.ldqT & 15) == 0) {
                stg_v4(dlo, make_uint4(lo[0], lo[1], lo[2], lo[3]));
                stg_v4(dlo + 16, make_uint4(lo[4], lo[5], lo[6], lo[7]));
                stg_v4(dhi, make_uint4(hi[0], hi[1], hi[2], hi[3]));
                stg_v4(dhi + 16, make_uint4(hi[4], hi[5], hi[6], hi[7]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    if (pos + j < limit) {
                        dlo[j] = static_cast<uint8_t>(lo[j >> 2] >> (8 * (j & 3)));
                        dhi[j] = static_cast<uint8_t>(hi[j >> 2] >> (8 * (j & 3)));
                    }
                }
            }
        }
    }
    __syncthreads();
    if (ROWS && tid < 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(srow_atom + 16 * tid);
        uint8_t *dst = P.s_row + (rt * P.kb_row_tiles + ct) * 512 + 16 * tid;
        if (MXQ_IN_BOUNDS(dst, 16, P.s_row, ext.s_row, P.err)) stg_v4(dst, v);
    } else if (tid >= 32 && tid < 64) {
        const int l = tid - 32;
        const uint4 v = *reinterpret_cast<const uint4 *>(scol_atom + 16 * l);
        uint8_t *dst = P.sT + (ct * P.kb_col_tiles + rt) * 512 + 16 * l;
        if (MXQ_IN_BOUNDS(dst, 16, P.sT, ext.sT, P.err)) stg_v4(dst, v);
    }
}

// Launch with programmatic stream serialization: the kernel begins with
// pdl_launch_dependents / pdl_wait (mxq_device.cuh), so the next launch in
// the stream overlaps this one's last CTAs and touches memory only after it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ============================================================================
// Persistent column quant (optionally dual / grouped) with TMA staging.
// Same output as k_quant_cols; each CTA walks tiles blockIdx.x, +gridDim.x, ...
// and keeps a ring of 128 x 128 bf16 tiles in shared memory (QuantRing): warp
// 0 keeps the cp.async.bulk.tensor loads of the next tiles in flight while the
// CTA works on the current one, so HBM reads overlap the quantization.  Grid =
// CTAs resident on all SMs.  Waits are bounded: a timeout sets the device
// error word and the CTA stops after its copies have landed.
// ============================================================================
constexpr uint32_t kTileBytes = kTile * kTile * 2;
// Tiles a CTA keeps in its ring (one being quantized, the rest loading) and
// the CTAs per SM that leaves room for.  The plain quant runs best with two
// slots at three CTAs per SM (dual quant of 131072 x 7168: 661 vs 673 us with
// three slots at two); the per-group quant, whose tiles start at arbitrary
// rows and end early at group boundaries, with three slots at two
// (grouped dual of 32768 x 7168: 174 vs 184 us).
template <bool GROUPED>
struct QuantRing {
    static constexpr int kSlots = GROUPED ? 3 : 2, kCtasPerSm = GROUPED ? 2 : 3;
};

// Groups whose offsets and padded starts a CTA keeps in shared memory.
constexpr int kQuantTableE = 256;

// The same from the CTA's shared tables: off[e] = group offsets, pre[e] =
// padded start P_e of group e (pre[E] = the padded total).
__device__ __forceinline__ void grouped_tile_source_tab(const int64_t *off, const int64_t *pre, int E, int64_t rt,
                                                        int64_t &src0, int &nvalid) {
    const int64_t t0 = rt * kTile;
    if (t0 >= pre[E]) {  // a padding tile past the last group: all zeros
        src0 = 0;
        nvalid = 0;
        return;
    }
    int lo = 0, hi = E;  // pre[lo] <= t0 < pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= t0) lo = mid; else hi = mid;
    }
    src0 = off[lo] + (t0 - pre[lo]);
    const int64_t left = off[lo + 1] - src0;
    nvalid = static_cast<int>(left < kTile ? left : kTile);
}

// First source row and the number of data rows of padded tile `rt` of a
// per-group column quant (warp-wide; lane 0's result is returned to all).
__device__ void grouped_tile_source(const ColParams &P, int64_t rt, int lane, int64_t &src0, int &nvalid) {
    const int64_t t0 = rt * kTile;
    int64_t run = 0, f_src0 = 0;
    int f_nvalid = 0;
    for (int base = 0; base < P.E; base += 32) {
        const int e = base + lane;
        int64_t n = 0;
        if (e < P.E) n = P.offsets[e + 1] - P.offsets[e];
        const int64_t padn = (n + 127) / 128 * 128;
        int64_t incl = padn;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const int64_t start = run + incl - padn;
        const bool mine = e < P.E && padn > 0 && t0 >= start && t0 < start + padn;
        const unsigned bal = __ballot_sync(0xffffffffu, mine);
        if (mine) {
            f_src0 = P.offsets[e] + (t0 - start);
            const int64_t left = n - (t0 - start);
            f_nvalid = static_cast<int>(left < kTile ? left : kTile);
        }
        if (bal) {
            const int src = __ffs(bal) - 1;
            src0 = __shfl_sync(0xffffffffu, f_src0, src);
            nvalid = __shfl_sync(0xffffffffu, f_nvalid, src);
            return;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    src0 = 0;
    nvalid = 0;  // a padding tile past the last group: all zeros
}

// COLS = false leaves out the column pass (a row quant alone); FMT selects the
// row pass's format: 0 MXFP8, 2 MXFP4 values as E4M3 codes (scale factor P.sf).
template <bool ROWS, bool GROUPED, bool COLS = true, int FMT = 0>
__global__ void __launch_bounds__(kThreads, QuantRing<GROUPED>::kCtasPerSm)
    k_quant_cols_tma(const __grid_constant__ CUtensorMap tmX, ColParams P, int64_t n_tiles, int64_t ct_tiles,
                     unsigned int *err) {
    constexpr int kRing = QuantRing<GROUPED>::kSlots;
    extern __shared__ __align__(128) uint8_t ring[];  // kRing x kTileBytes
    // scale tiles staged per tile, two deep: tile k + 1's passes fill one while
    // tile k's are still being stored from the other
    __shared__ __align__(16) uint8_t srow_atoms[2][512];
    __shared__ __align__(16) uint8_t scol_atoms[2][512];
    __shared__ __align__(8) uint64_t bars[kRing];
    __shared__ int64_t sh_src0[kRing];
    __shared__ int sh_nvalid[kRing];
    __shared__ int abort_flag;
    __shared__ int64_t g_tab[GROUPED ? 2 * (kQuantTableE + 1) : 1];  // group offsets, padded starts

    pdl_wait();  // no global access before the previous kernel in the stream has completed
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t ring_s = smem_u32(ring), bar0 = smem_u32(&bars[0]);
    const ColExtents ext = col_extents(P);
    (void)ext;
    volatile int *abort_v = &abort_flag;
    if (tid == 0) {
        abort_flag = 0;
        for (int j = 0; j < kRing; j++) mbar_init(bar0 + 8 * j, 1);
        fence_mbar_init();
    }
    const bool tables = GROUPED && P.E <= kQuantTableE;
    // 32-byte code stores where the output rows allow them (block starts are
    // multiples of 32 bytes from the row start)
    const bool row_v8 = ROWS && ((reinterpret_cast<uintptr_t>(P.q_row) | static_cast<uintptr_t>(P.C)) & 31) == 0;
    const bool col_v8 = ((reinterpret_cast<uintptr_t>(P.qT) | static_cast<uintptr_t>(P.ldqT)) & 31) == 0;
    int64_t *g_off = g_tab, *g_pre = g_tab + (kQuantTableE + 1);
    if (GROUPED && warp == 0) {
        // malformed offsets: no tile is decoded from them, no load or store is issued
        const bool good = group_offsets_valid(P.offsets, P.E, P.R, lane);
        if (lane == 0 && !good) {
            abort_flag = 1;
            atomicOr(err, kErrBadOffsets);
        }
    }
    if (tables && warp == 0) {
        // one scan of the offsets per CTA instead of one per tile
        int64_t run = 0;
        for (int base = 0; base <= P.E; base += 32) {
            const int e = base + lane;
            int64_t o0 = 0, padn = 0;
            if (e <= P.E) o0 = P.offsets[e];
            if (e < P.E) padn = (P.offsets[e + 1] - o0 + 127) / 128 * 128;
            int64_t incl = padn;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (e <= P.E) {
                g_off[e] = o0;
                g_pre[e] = run + incl - padn;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    if (GROUPED && abort_flag) return;  // (uniform: set before the barrier)

    // warp 0: resolve tile t into slot `buf` and start its load
    auto issue = [&](int64_t t, int buf) {
        const int64_t rt = t / ct_tiles, ct = t % ct_tiles;
        int64_t src0 = rt * kTile;
        int nvalid;
        if (GROUPED && tables) {
            grouped_tile_source_tab(g_off, g_pre, P.E, rt, src0, nvalid);
        } else if (GROUPED) {
            grouped_tile_source(P, rt, lane, src0, nvalid);
        } else {
            const int64_t left = P.R - src0;
            nvalid = static_cast<int>(left < kTile ? left : kTile);
        }
        if (lane == 0) {
            sh_src0[buf] = src0;
            sh_nvalid[buf] = nvalid;
            fence_proxy_async_smem();  // the slot's earlier generic reads come first
            mbar_arrive_expect_tx(bar0 + 8 * buf, kTileBytes);
            tma_load_2d(ring_s + buf * kTileBytes, &tmX, bar0 + 8 * buf, static_cast<int>(ct * kTile),
                        static_cast<int>(src0));
        }
    };

    if (ROWS && GROUPED && !P.row_pad && blockIdx.x == 0) {
        // row scales of the padding rows [R, ceil128(R)) of the last scale tile:
        // no tile owns them
        const int64_t npad = (P.R + 127) / 128 * 128 - P.R;
        for (int64_t i = tid; i < npad * P.kb_row_tiles; i += kThreads) {
            const int64_t r = P.R + i / P.kb_row_tiles, kt = i % P.kb_row_tiles;
            uint8_t *dst = P.s_row + ((r >> 7) * P.kb_row_tiles + kt) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3);
            if (MXQ_IN_BOUNDS(dst, 4, P.s_row, ext.s_row, err)) *reinterpret_cast<uint32_t *>(dst) = 0u;
        }
    }

    // One barrier per tile.  A thread may start tile k once its slot's mbarrier
    // completes (the arrive that armed it also publishes sh_src0/sh_nvalid);
    // after the barrier that ends tile k every thread is done with its slot,
    // and the load kRing tiles ahead goes there.
    int64_t t = blockIdx.x;
    if (warp == 0) {
        for (int j = 0; j < kRing; j++)
            if (t + j * static_cast<int64_t>(gridDim.x) < n_tiles) issue(t + j * static_cast<int64_t>(gridDim.x), j);
    }
    uint32_t k = 0;
    for (; t < n_tiles; t += gridDim.x, k++) {
        // the next launch may begin once every CTA has started its last tile
        // (triggering at the start let a run of small launches pile their
        // waiting CTAs onto the idle SMs, which measured slower)
        if (t + static_cast<int64_t>(gridDim.x) >= n_tiles) pdl_launch_dependents();
        const int buf = static_cast<int>(k % kRing);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * buf, (k / kRing) & 1, abort_v, err));
        uint8_t *srow_atom = srow_atoms[k & 1], *scol_atom = scol_atoms[k & 1];

        const uint8_t *tile = ring + buf * kTileBytes;
        const int64_t rt = t / ct_tiles, ct = t % ct_tiles;
        const int64_t c0 = ct * kTile;
        const int64_t src0 = sh_src0[buf];  // read before the barrier that frees the slot
        const int nvalid = sh_nvalid[buf];
        if (ok) {

            if (ROWS) {
                // ---- row pass: thread (row, blk) quantizes one 32-element block ----
                // Its four 16-byte chunks are read starting at chunk g, which
                // differs between the 8 threads of each quarter-warp that share
                // a bank window (blk & 1 x g covers 8 distinct 16-byte slots),
                // so the reads are conflict-free; the codes are put back in
                // column order before the two 16-byte stores.
                const int blk = tid & 3;
                const int g = (blk >> 1) + 2 * ((tid >> 2) & 1);
                const int64_t gc = c0 + 32 * blk;
#pragma unroll
                for (int it = 0; it < 2; it++) {
                    const int row = (tid >> 2) + 64 * it;
                    const uint8_t *src = tile + row * (kTile * 2) + 64 * blk;
                    uint32_t w[4][4];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(src + 16 * ((j + g) & 3));
                        w[j][0] = v.x; w[j][1] = v.y; w[j][2] = v.z; w[j][3] = v.w;
                    }
                    const uint32_t a = max(max(amax8_bf16(w[0]), amax8_bf16(w[1])), max(amax8_bf16(w[2]), amax8_bf16(w[3])));
                    int X = 0;            // FMT 0: MXFP8 scale exponent
                    Mx4Blk T{};           // FMT 2: MXFP4 block constants
                    bool nonfinite = false;
                    uint8_t sbyte;
                    if (FMT == 0) {
                        X = mx8_exp_from_bf16(a);
                        sbyte = mx8_scale_byte(X);
                    } else {
                        nonfinite = (a << 16) >= 0x7F800000u;
                        const int e = nonfinite ? 0 : mx4_exp(__uint_as_float(a << 16), P.sf);
                        sbyte = nonfinite ? 0xFF : static_cast<uint8_t>(e + 127);
                        T = mx4_block(e);
                    }
                    const bool valid = row < nvalid && gc < P.C;
                    if (valid) {
                        uint2 cd[4];
#pragma unroll
                        for (int j = 0; j < 4; j++) cd[j] = FMT == 0 ? e4m3_codes8(w[j], X) : mx4_as_e4m3_codes8(w[j], T, nonfinite);
                        // cd[j] holds chunk (j + g) & 3: rotate back by g (1, then 2)
                        if (g & 1) {
                            const uint2 t = cd[3];
                            cd[3] = cd[2]; cd[2] = cd[1]; cd[1] = cd[0]; cd[0] = t;
                        }
                        if (g & 2) {
                            uint2 t = cd[0]; cd[0] = cd[2]; cd[2] = t;
                            t = cd[1]; cd[1] = cd[3]; cd[3] = t;
                        }
                        uint8_t *dst = P.q_row + (src0 + row) * P.C + gc;
                        const uint4 lo4 = make_uint4(cd[0].x, cd[0].y, cd[1].x, cd[1].y);
                        const uint4 hi4 = make_uint4(cd[2].x, cd[2].y, cd[3].x, cd[3].y);
                        if (!MXQ_IN_BOUNDS(dst, 32, P.q_row, ext.q_row, err)) {
                        } else if (row_v8) {
                            stg_v8(dst, lo4, hi4);
                        } else {
                            stg_v4(dst, lo4);
                            stg_v4(dst + 16, hi4);
                        }
                    }
                    if (GROUPED && !P.row_pad)  // row-major staging: row r's four blocks form word r
                        srow_atom[4 * row + blk] = gc < P.C ? sbyte : 0;
                    else
                        srow_atom[16 * (row & 31) + 4 * (row >> 5) + blk] = valid ? sbyte : 0;
                }
            }

            // ---- column pass: thread (p, b) = (column pair, 32-row block) ----
            if constexpr (COLS) {
                const int p = tid & 63, b = tid >> 6;
                uint32_t col[32];
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const uint32_t wv = *reinterpret_cast<const uint32_t *>(tile + (32 * b + i) * (kTile * 2) + 4 * p);
                    col[i] = (!GROUPED || 32 * b + i < nvalid) ? wv : 0u;  // rows of the next group read as zero
                }
                uint32_t m2 = 0;
#pragma unroll
                for (int i = 0; i < 32; i++) m2 = __vmaxu2(m2, col[i] & 0x7FFF7FFFu);
                const int Xlo = mx8_exp_from_bf16(m2 & 0xFFFFu), Xhi = mx8_exp_from_bf16(m2 >> 16);
                const int cl = 2 * p, ch2 = 2 * p + 1;
                scol_atom[16 * (cl & 31) + 4 * (cl >> 5) + b] = mx8_scale_byte(Xlo);
                scol_atom[16 * (ch2 & 31) + 4 * (ch2 >> 5) + b] = mx8_scale_byte(Xhi);

                const int64_t gcol = c0 + cl;
                if (gcol < P.C) {
                    uint32_t lo[8], hi[8];
                    // column 2p's scale in the low half, column 2p + 1's in the high half
                    const uint32_t inv2 = pow2_neg_bf16(Xlo > 127 ? 0 : Xlo) | (pow2_neg_bf16(Xhi > 127 ? 0 : Xhi) << 16);
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        const uint32_t a0 = mul_bf16x2(col[4 * q], inv2), a1 = mul_bf16x2(col[4 * q + 1], inv2);
                        const uint32_t a2 = mul_bf16x2(col[4 * q + 2], inv2), a3 = mul_bf16x2(col[4 * q + 3], inv2);
                        lo[q] = e4m3x4(bf16lo(a0), bf16lo(a1), bf16lo(a2), bf16lo(a3));
                        hi[q] = e4m3x4(bf16hi(a0), bf16hi(a1), bf16hi(a2), bf16hi(a3));
                    }
                    if (Xlo > 127 || Xhi > 127) {  // non-finite blocks: NaN codes with the sign kept
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            uint32_t sl = 0, sh = 0;
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                sl |= (0x7Fu | ((col[4 * q + j] >> 8) & 0x80u)) << (8 * j);
                                sh |= (0x7Fu | ((col[4 * q + j] >> 24) & 0x80u)) << (8 * j);
                            }
                            if (Xlo > 127) lo[q] = sl;
                            if (Xhi > 127) hi[q] = sh;
                        }
                    }
                    const int64_t pos = rt * kTile + 32 * b;  // first output column (token) of the block
                    uint8_t *dlo = P.qT + gcol * P.ldqT + pos;
                    uint8_t *dhi = dlo + P.ldqT;
                    const int64_t limit = GROUPED ? P.ldqT : P.R;  // grouped tiles write padding zeros too
                    if (pos < limit && (!MXQ_IN_BOUNDS(dlo, limit - pos < 32 ? limit - pos : 32, P.qT, ext.qT, err) ||
                                        !MXQ_IN_BOUNDS(dhi, limit - pos < 32 ? limit - pos : 32, P.qT, ext.qT, err))) {
                    } else if (pos + 32 <= limit && col_v8) {
                        stg_v8(dlo, make_uint4(lo[0], lo[1], lo[2], lo[3]), make_uint4(lo[4], lo[5], lo[6], lo[7]));
                        stg_v8(dhi, make_uint4(hi[0], hi[1], hi[2], hi[3]), make_uint4(hi[4], hi[5], hi[6], hi[7]));
                    } else if (pos + 32 <= limit && (P.ldqT & 15) == 0) {
                        stg_v4(dlo, make_uint4(lo[0], lo[1], lo[2], lo[3]));
                        stg_v4(dlo + 16, make_uint4(lo[4], lo[5], lo[6], lo[7]));
                        stg_v4(dhi, make_uint4(hi[0], hi[1], hi[2], hi[3]));
                        stg_v4(dhi + 16, make_uint4(hi[4], hi[5], hi[6], hi[7]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++) {
                            if (pos + j < limit) {
                                dlo[j] = static_cast<uint8_t>(lo[j >> 2] >> (8 * (j & 3)));
                                dhi[j] = static_cast<uint8_t>(hi[j >> 2] >> (8 * (j & 3)));
                            }
                        }
                    }
                }
            }
        }
        if (!__syncthreads_and(ok)) break;
        {
            const int64_t tn = t + kRing * static_cast<int64_t>(gridDim.x);
            if (warp == 0 && tn < n_tiles) issue(tn, buf);
        }
        if (ROWS && GROUPED && !P.row_pad && tid >= kThreads - kTile && tid - (kThreads - kTile) < nvalid) {
            // A group's rows start anywhere inside a 128-row scale tile: each
            // row's word goes to its own place, and only this tile's rows.
            const int row = tid - (kThreads - kTile);
            const int64_t r = src0 + row;
            uint8_t *dst = P.s_row + ((r >> 7) * P.kb_row_tiles + ct) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3);
            if (MXQ_IN_BOUNDS(dst, 4, P.s_row, ext.s_row, err))
                *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(srow_atom + 4 * row);
        }
        if (ROWS && (!GROUPED || P.row_pad) && tid < 32) {
            // (per-group padded layout: padded tile rt is scale tile rt, its
            // padding rows zero)
            const uint4 v = *reinterpret_cast<const uint4 *>(srow_atom + 16 * tid);
            uint8_t *dst = P.s_row + (rt * P.kb_row_tiles + ct) * 512 + 16 * tid;
            if (MXQ_IN_BOUNDS(dst, 16, P.s_row, ext.s_row, err)) stg_v4(dst, v);
        } else if (COLS && tid >= 32 && tid < 64) {
            const int l = tid - 32;
            const uint4 v = *reinterpret_cast<const uint4 *>(scol_atom + 16 * l);
            uint8_t *dst = P.sT + (ct * P.kb_col_tiles + rt) * 512 + 16 * l;
            if (MXQ_IN_BOUNDS(dst, 16, P.sT, ext.sT, err)) stg_v4(dst, v);
        }
    }
    // stopped early: let the loads still in flight (this tile's and the
    // prefetched ones) land before shared memory goes away; bounded as well
    if (tid == 0 && t < n_tiles) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t j = 0; j < static_cast<uint32_t>(kRing); j++) {
            const uint32_t kk = k + j;
            if (t + j * static_cast<int64_t>(gridDim.x) >= n_tiles) break;
            while (!mbar_try_wait(bar0 + 8 * (kk % kRing), (kk / kRing) & 1)) {
                if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
            }
        }
    }
}

// ============================================================================
// MXFP4 quant-dequant, optionally with the saturation mask of the clipped
// straight-through estimator (|x| > 6 * block scale; one 32-bit word per
// block, bit i = element i of the block; 0 for a block with a non-finite
// element, whose scale is not finite).
//  Vector path (cols % 32 == 0, 16-byte aligned): a CTA takes a window of
//  kEwChunks x 256 chunks of 8 floats; thread t handles chunks t and t + 256
//  of it, both loaded before any arithmetic, and the 4 lanes holding one
//  32-element block exchange their maxima by shuffles.  General path: one
//  warp per block of 32 (ragged rows).
// Loops are warp-uniform so that every shuffle has all 32 lanes.
// ============================================================================
constexpr int kEwChunks = 2;  // 8-element chunks per thread in flight
constexpr int64_t kEwWindow = static_cast<int64_t>(kThreads) * kEwChunks;

template <bool MASK>
__global__ void __launch_bounds__(kThreads) k_qdq_mxfp4_vec(const float *__restrict__ x, float *y,
                                                            uint32_t *__restrict__ mask, int64_t nchunks, float sf,
                                                            unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t xy_bytes = static_cast<uint64_t>(nchunks) * 32, m_bytes = static_cast<uint64_t>(nchunks);  // extents
    (void)xy_bytes; (void)m_bytes; (void)err;
    // one 32-byte access per chunk where both tensors are 32-byte aligned
    const bool al32 = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 31) == 0;
    for (int64_t w0 = static_cast<int64_t>(blockIdx.x) * kEwWindow; w0 < nchunks;
         w0 += static_cast<int64_t>(gridDim.x) * kEwWindow) {
        uint4 in[kEwChunks][2];
#pragma unroll
        for (int u = 0; u < kEwChunks; u++) {
            const int64_t g = w0 + u * kThreads + threadIdx.x;
            in[u][0] = in[u][1] = make_uint4(0, 0, 0, 0);
            if (g < nchunks && MXQ_IN_BOUNDS(x + 8 * g, 32, x, xy_bytes, err)) {
                if (al32) {
                    ldg_nc_v8(x + 8 * g, in[u][0], in[u][1]);
                } else {
                    in[u][0] = ldg_nc_v4(x + 8 * g);
                    in[u][1] = ldg_nc_v4(x + 8 * g + 4);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kEwChunks; u++) {
            const int64_t g = w0 + u * kThreads + threadIdx.x;
            const uint32_t v[8] = {in[u][0].x, in[u][0].y, in[u][0].z, in[u][0].w,
                                   in[u][1].x, in[u][1].y, in[u][1].z, in[u][1].w};
            uint32_t a = 0;
#pragma unroll
            for (int k = 0; k < 8; k++) a = max(a, v[k] & 0x7FFFFFFFu);
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
            uint32_t o[8];
            uint32_t bits = 0;
            if (a >= 0x7F800000u) {
#pragma unroll
                for (int k = 0; k < 8; k++) o[k] = 0x7FC00000u;
            } else {
                const Mx4Blk B = mx4_block(mx4_exp(__uint_as_float(a), sf));
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t ax = v[k] & 0x7FFFFFFFu;
                    o[k] = mx4_snap(ax, B) | (v[k] & 0x80000000u);
                    if (MASK) bits |= (ax > B.six_s ? 1u : 0u) << k;
                }
            }
            if (MASK) {
                // the block's word from its 4 lanes, then lanes 0-7 write the
                // warp's 8 consecutive words
                const int64_t wb = w0 + u * kThreads + 32 * warp;  // the warp's first chunk
                uint32_t w = bits << (8 * (lane & 3));
                w |= __shfl_xor_sync(0xffffffffu, w, 1);
                w |= __shfl_xor_sync(0xffffffffu, w, 2);
                w = __shfl_sync(0xffffffffu, w, (4 * lane) & 31);
                if (lane < 8 && wb + 4 * lane < nchunks && MXQ_IN_BOUNDS(mask + wb / 4 + lane, 4, mask, m_bytes, err))
                    mask[wb / 4 + lane] = w;
            }
            if (g >= nchunks || !MXQ_IN_BOUNDS(y + 8 * g, 32, y, xy_bytes, err)) continue;
            const uint4 o0 = make_uint4(o[0], o[1], o[2], o[3]), o1 = make_uint4(o[4], o[5], o[6], o[7]);
            if (al32) {
                stg_v8(y + 8 * g, o0, o1);
            } else {
                stg_v4(y + 8 * g, o0);
                stg_v4(y + 8 * g + 4, o1);
            }
        }
    }
}

template <bool MASK>
__global__ void __launch_bounds__(kThreads) k_qdq_mxfp4_gen(const float *__restrict__ x, float *y,
                                                            uint32_t *__restrict__ mask, int64_t rows, int64_t cols,
                                                            float sf, unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    const uint64_t xy_bytes = static_cast<uint64_t>(rows * cols) * 4;  // extents (debug builds)
    (void)xy_bytes; (void)err;
    const int lane = threadIdx.x & 31;
    const int64_t nb = (cols + 31) / 32;
    const int64_t nblocks = rows * nb;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t wstride = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    for (int64_t k = warp0; k < nblocks; k += wstride) {
        const int64_t r = k / nb, b = k % nb;
        const int64_t c = 32 * b + lane;
        const bool valid = c < cols;
        const uint32_t v = valid && MXQ_IN_BOUNDS(x + r * cols + c, 4, x, xy_bytes, err) ? __float_as_uint(x[r * cols + c]) : 0u;
        const uint32_t ax = v & 0x7FFFFFFFu;
        uint32_t a = ax;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
        uint32_t out;
        bool sat = false;
        if (a >= 0x7F800000u) {
            out = 0x7FC00000u;
        } else {
            const Mx4Blk B = mx4_block(mx4_exp(__uint_as_float(a), sf));
            out = mx4_snap(ax, B) | (v & 0x80000000u);
            sat = valid && ax > B.six_s;
        }
        if (MASK) {
            const uint32_t w = __ballot_sync(0xffffffffu, sat);
            if (lane == 0 && MXQ_IN_BOUNDS(mask + k, 4, mask, static_cast<uint64_t>(nblocks) * 4, err)) mask[k] = w;
        }
        if (valid && MXQ_IN_BOUNDS(y + r * cols + c, 4, y, xy_bytes, err)) y[r * cols + c] = __uint_as_float(out);
    }
}

// MXFP4 quant-dequant of bf16 to bf16 (cols % 32 == 0, 16-byte aligned): a
// thread takes whole 32-element blocks (four 16-byte chunks each), two blocks
// in flight; a CTA takes a window of 2 x 256 blocks.  Every result (codebook
// value x 2^e, or NaN for a non-finite block) is exact in bf16.
constexpr int64_t kBlkWindow = static_cast<int64_t>(kThreads) * 2;
__global__ void __launch_bounds__(kThreads) k_qdq_mxfp4_bf16(const uint16_t *__restrict__ x, uint16_t *y,
                                                             int64_t nblocks, float sf, unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    const uint64_t xy_bytes = static_cast<uint64_t>(nblocks) * 64;  // extent (debug builds)
    (void)xy_bytes; (void)err;
    for (int64_t w0 = static_cast<int64_t>(blockIdx.x) * kBlkWindow; w0 < nblocks;
         w0 += static_cast<int64_t>(gridDim.x) * kBlkWindow) {
        uint4 in[2][4];
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int64_t b = w0 + u * kThreads + threadIdx.x;
#pragma unroll
            for (int j = 0; j < 4; j++)
                in[u][j] = b < nblocks && MXQ_IN_BOUNDS(x + 32 * b + 8 * j, 16, x, xy_bytes, err) ? ldg_nc_v4(x + 32 * b + 8 * j)
                                                                                               : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int64_t b = w0 + u * kThreads + threadIdx.x;
            if (b >= nblocks || !MXQ_IN_BOUNDS(y + 32 * b, 64, y, xy_bytes, err)) continue;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                w[4 * j] = in[u][j].x; w[4 * j + 1] = in[u][j].y; w[4 * j + 2] = in[u][j].z; w[4 * j + 3] = in[u][j].w;
            }
            uint32_t m2 = 0;
#pragma unroll
            for (int k = 0; k < 16; k++) m2 = __vmaxu2(m2, w[k] & 0x7FFF7FFFu);
            const uint32_t a = max(m2 & 0xFFFFu, m2 >> 16) << 16;  // |bf16| bits as fp32 bits
            uint32_t o[16];
            if (a >= 0x7F800000u) {
#pragma unroll
                for (int k = 0; k < 16; k++) o[k] = 0x7FC07FC0u;
            } else {
                const int e = mx4_exp(__uint_as_float(a), sf);
                const float f = mx4_inv_scale(e) * kBf16Nudge, sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
#pragma unroll
                for (int k = 0; k < 16; k++)
                    o[k] = e2m1_qdq_bf16x2(__uint_as_float(w[k] << 16) * f, __uint_as_float(w[k] & 0xFFFF0000u) * f, sc);
            }
#pragma unroll
            for (int j = 0; j < 4; j++) stg_v4(y + 32 * b + 8 * j, make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]));
        }
    }
}

// Packed MXFP4 quant of an [R x C] tensor (fp32 or bf16, leading dim ldx)
// with R and C multiples of 128, so that every scale tile is whole and has no
// padding.  A CTA takes a block of 64 rows x 128 columns: thread t quantizes
// the 32-element block t % 4 of row t / 4 (all of its loads issued first, one
// scale decision per block) into 16 bytes of nibbles (even element in the low
// nibble); the 4 lanes holding a row's 4 blocks put its scale bytes together,
// one 16-byte row-group word of its scale tile, stored as one word.
template <typename InT>
__global__ void __launch_bounds__(kThreads) k_pack_mxfp4(const InT *__restrict__ x, int64_t ldx,
                                                         uint8_t *__restrict__ q, int64_t ldq,
                                                         uint8_t *__restrict__ s, int64_t kb_tiles, float sf,
                                                         unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    // extents (debug builds): R = gridDim.y * 64 rows of C = gridDim.x * 128 columns
    const int64_t R = static_cast<int64_t>(gridDim.y) * 64, C = static_cast<int64_t>(gridDim.x) * 128;
    const uint64_t x_bytes = static_cast<uint64_t>((R - 1) * ldx + C) * sizeof(InT);
    const uint64_t q_bytes = static_cast<uint64_t>(R * ldq), s_bytes = static_cast<uint64_t>(R / 128 * kb_tiles * 512);
    (void)x_bytes; (void)q_bytes; (void)s_bytes; (void)err;
    constexpr int kWords = sizeof(InT) == 4 ? 32 : 16;  // 32-bit words of one block
    const int t = threadIdx.x, lane = t & 31, blk = t & 3;
    const int64_t r = static_cast<int64_t>(blockIdx.y) * 64 + (t >> 2);
    const int64_t c = static_cast<int64_t>(blockIdx.x) * 128 + 32 * blk;
    uint32_t w[kWords];
    const InT *src = x + r * ldx + c;
    const bool src_ok = MXQ_IN_BOUNDS(src, 32 * sizeof(InT), x, x_bytes, err);
#pragma unroll
    for (int j = 0; j < kWords / 8; j++) {
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (src_ok) ldg_nc_v8(reinterpret_cast<const uint32_t *>(src) + 8 * j, lo, hi);
        w[8 * j] = lo.x; w[8 * j + 1] = lo.y; w[8 * j + 2] = lo.z; w[8 * j + 3] = lo.w;
        w[8 * j + 4] = hi.x; w[8 * j + 5] = hi.y; w[8 * j + 6] = hi.z; w[8 * j + 7] = hi.w;
    }
    uint32_t a = 0;
    if (sizeof(InT) == 4) {
#pragma unroll
        for (int k = 0; k < kWords; k++) a = max(a, w[k] & 0x7FFFFFFFu);
    } else {
        uint32_t m2 = 0;
#pragma unroll
        for (int k = 0; k < kWords; k++) m2 = __vmaxu2(m2, w[k] & 0x7FFF7FFFu);
        a = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    }
    const bool nonfinite = a >= 0x7F800000u;
    const int e = nonfinite ? 0 : mx4_exp(__uint_as_float(a), sf);
    const uint32_t sbyte = nonfinite ? 0xFFu : static_cast<uint32_t>(e + 127);
    uint32_t nib[4];  // 8 nibbles each
    const float inv = mx4_inv_scale(e);
    const uint32_t t025 = static_cast<uint32_t>(e + 125) << 23;
#pragma unroll
    for (int g = 0; g < 4; g++) {
        uint32_t v[8];  // fp32 bit patterns of elements 8g .. 8g + 7
#pragma unroll
        for (int k = 0; k < 8; k++)
            v[k] = sizeof(InT) == 4 ? w[8 * g + k] : ((k & 1) ? (w[4 * g + (k >> 1)] & 0xFFFF0000u) : (w[4 * g + (k >> 1)] << 16));
        if (nonfinite) {
            uint32_t p = 0;
#pragma unroll
            for (int k = 0; k < 8; k++) p |= (((v[k] >> 28) & 8u) | 7u) << (4 * k);
            nib[g] = p;
        } else {
            uint32_t b[4];
            if (sizeof(InT) == 2) {  // bf16: the one-multiply nudge
                const float f = inv * kBf16Nudge;
#pragma unroll
                for (int k = 0; k < 4; k++)
                    b[k] = cvt_e2m1x2(__uint_as_float(v[2 * k]) * f, __uint_as_float(v[2 * k + 1]) * f);
            } else {
#pragma unroll
                for (int k = 0; k < 4; k++)
                    b[k] = cvt_e2m1x2(mx4_scaled(v[2 * k], t025, inv), mx4_scaled(v[2 * k + 1], t025, inv));
            }
            nib[g] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
        }
    }
    if (MXQ_IN_BOUNDS(q + r * ldq + c / 2, 16, q, q_bytes, err))
        stg_v4(q + r * ldq + c / 2, make_uint4(nib[0], nib[1], nib[2], nib[3]));
    // the row's 4 scale bytes, from lanes 4i .. 4i + 3
    uint32_t word = sbyte << (8 * blk);
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    uint8_t *sdst = s + ((r >> 7) * kb_tiles + blockIdx.x) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3);
    if (blk == 0 && MXQ_IN_BOUNDS(sdst, 4, s, s_bytes, err)) *reinterpret_cast<uint32_t *>(sdst) = word;
    (void)lane;
}

// Clipped straight-through estimator, backward: gx = gy except +0.0 where the
// forward's saturation mask is set.  Vector path (cols % 32 == 0, 16-byte
// aligned): the QDQ's windows, two 32-byte chunks and their mask words loaded
// per thread before any store; general path: one warp per block.
__global__ void __launch_bounds__(kThreads) k_ste_backward_vec(const float *__restrict__ gy,
                                                               const uint32_t *__restrict__ mask, float *gx,
                                                               int64_t nchunks, unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    const uint64_t g_bytes = static_cast<uint64_t>(nchunks) * 32, m_bytes = static_cast<uint64_t>(nchunks);  // extents
    (void)g_bytes; (void)m_bytes; (void)err;
    const bool al32 = ((reinterpret_cast<uintptr_t>(gy) | reinterpret_cast<uintptr_t>(gx)) & 31) == 0;
    for (int64_t w0 = static_cast<int64_t>(blockIdx.x) * kEwWindow; w0 < nchunks;
         w0 += static_cast<int64_t>(gridDim.x) * kEwWindow) {
        uint4 in[kEwChunks][2];
        uint32_t mw[kEwChunks];
#pragma unroll
        for (int u = 0; u < kEwChunks; u++) {
            const int64_t g = w0 + u * kThreads + threadIdx.x;
            in[u][0] = in[u][1] = make_uint4(0, 0, 0, 0);
            mw[u] = 0;
            if (g < nchunks && MXQ_IN_BOUNDS(gy + 8 * g, 32, gy, g_bytes, err) &&
                MXQ_IN_BOUNDS(mask + g / 4, 4, mask, m_bytes, err)) {
                mw[u] = __ldg(mask + g / 4);
                if (al32) {
                    ldg_nc_v8(gy + 8 * g, in[u][0], in[u][1]);
                } else {
                    in[u][0] = ldg_nc_v4(gy + 8 * g);
                    in[u][1] = ldg_nc_v4(gy + 8 * g + 4);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kEwChunks; u++) {
            const int64_t g = w0 + u * kThreads + threadIdx.x;
            if (g >= nchunks || !MXQ_IN_BOUNDS(gx + 8 * g, 32, gx, g_bytes, err)) continue;
            const uint32_t bits = (mw[u] >> (8 * (g & 3))) & 0xFFu;
            uint4 a = in[u][0], b = in[u][1];
            if (bits) {
                a.x = (bits & 1u) ? 0u : a.x;    a.y = (bits & 2u) ? 0u : a.y;
                a.z = (bits & 4u) ? 0u : a.z;    a.w = (bits & 8u) ? 0u : a.w;
                b.x = (bits & 16u) ? 0u : b.x;   b.y = (bits & 32u) ? 0u : b.y;
                b.z = (bits & 64u) ? 0u : b.z;   b.w = (bits & 128u) ? 0u : b.w;
            }
            if (al32) {
                stg_v8(gx + 8 * g, a, b);
            } else {
                stg_v4(gx + 8 * g, a);
                stg_v4(gx + 8 * g + 4, b);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads) k_ste_backward_gen(const float *__restrict__ gy,
                                                               const uint32_t *__restrict__ mask, float *gx,
                                                               int64_t rows, int64_t cols, unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    const uint64_t g_bytes = static_cast<uint64_t>(rows * cols) * 4;  // extent (debug builds)
    (void)g_bytes; (void)err;
    const int lane = threadIdx.x & 31;
    const int64_t nb = (cols + 31) / 32;
    const int64_t nblocks = rows * nb;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t wstride = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    for (int64_t k = warp0; k < nblocks; k += wstride) {
        const int64_t r = k / nb, c = 32 * (k % nb) + lane;
        if (c >= cols || !MXQ_IN_BOUNDS(gx + r * cols + c, 4, gx, g_bytes, err) ||
            !MXQ_IN_BOUNDS(gy + r * cols + c, 4, gy, g_bytes, err) ||
            !MXQ_IN_BOUNDS(mask + k, 4, mask, static_cast<uint64_t>(nblocks) * 4, err))
            continue;
        const bool sat = (__ldg(mask + k) >> lane) & 1u;
        gx[r * cols + c] = sat ? 0.0f : gy[r * cols + c];
    }
}

// CTAs for the windowed elementwise kernels: one window each, so the hardware
// hands out short CTAs as SMs free up (no persistent loop whose last round
// runs part-empty); capped, with the kernels looping past the cap.
int grid_windows(int64_t nchunks, int64_t window = kEwWindow) {
    const int64_t g = (nchunks + window - 1) / window;
    return static_cast<int>(g < 1 ? 1 : (g > (1 << 20) ? (1 << 20) : g));
}

int grid_for(int64_t work_items, int per_cta) {
    int64_t g = (work_items + per_cta - 1) / per_cta;
    const int64_t cap = 152 * 16;
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

// ---------------------------------------------------------------- launchers
namespace {
// Persistent TMA-staged launch of k_quant_cols_tma; returns false (no launch)
// where x takes no tensor map.
template <bool ROWS, bool GROUPED, bool COLS = true, int FMT = 0>
bool launch_cols_tma(const ColParams &P, int64_t row_tiles, cudaStream_t st, cudaError_t *res);
}  // namespace

cudaError_t launch_quant_rows(const void *x, bool fp32_in, int fmt, int64_t R, int64_t C, int64_t ldx, uint8_t *q,
                              uint8_t *s, cudaStream_t st, float sf) {
    unsigned int *err = nullptr;
    cudaError_t ee = device_error_word(&err);
    if (ee != cudaSuccess) return ee;
    const dim3 grid(static_cast<unsigned>((C + kTile - 1) / kTile), static_cast<unsigned>((R + kTile - 1) / kTile));
    const int64_t kb_tiles = ((C / 32) + 3) / 4;
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    if (!fp32_in && (fmt == 0 || fmt == 2)) {
        // the persistent TMA-staged kernel, row pass only
        ColParams P{};
        P.x = xb; P.R = R; P.C = C; P.ldx = ldx;
        P.q_row = q; P.s_row = s; P.kb_row_tiles = kb_tiles;
        P.sf = sf;
        P.err = err;
        const int64_t row_tiles = (R + kTile - 1) / kTile;
        cudaError_t res = cudaSuccess;
        if (fmt == 0 ? launch_cols_tma<true, false, false, 0>(P, row_tiles, st, &res)
                     : launch_cols_tma<true, false, false, 2>(P, row_tiles, st, &res))
            return res;
    }
    if (fmt == 0) {
        (void)launch_pdl(k_quant_rows<uint16_t, 0>, grid, kThreads, 0, st, xb, R, C, ldx, q, C, s, kb_tiles, sf, err);
    } else if (fmt == 2) {
        (void)launch_pdl(k_quant_rows<uint16_t, 2>, grid, kThreads, 0, st, xb, R, C, ldx, q, C, s, kb_tiles, sf, err);
    } else if (R % kTile == 0 && C % kTile == 0 &&
               ((reinterpret_cast<uintptr_t>(x) | static_cast<uintptr_t>(ldx * (fp32_in ? 4 : 2))) & 31) == 0) {
        // whole scale tiles: 64 x 128 blocks
        const dim3 g2(static_cast<unsigned>(C / kTile), static_cast<unsigned>(R / 64));
        if (fp32_in)
            (void)launch_pdl(k_pack_mxfp4<float>, g2, kThreads, 0, st, static_cast<const float *>(x), ldx, q, C / 2, s, kb_tiles, sf,
                                                          err);
        else
            (void)launch_pdl(k_pack_mxfp4<uint16_t>, g2, kThreads, 0, st, xb, ldx, q, C / 2, s, kb_tiles, sf, err);
    } else if (fp32_in) {
        (void)launch_pdl(k_quant_rows<float, 1>, grid, kThreads, 0, st, static_cast<const float *>(x), R, C, ldx, q, C / 2, s,
                                                          kb_tiles, sf, err);
    } else {
        (void)launch_pdl(k_quant_rows<uint16_t, 1>, grid, kThreads, 0, st, xb, R, C, ldx, q, C / 2, s, kb_tiles, sf, err);
    }
    return cudaGetLastError();
}

namespace {

// Persistent TMA-staged launch of the column quant; returns false (no launch)
// when the input cannot be described by a tensor map -- no rows at all (a
// per-group quant whose groups are all empty writes only padding), or an
// unaligned base or row stride, which the C entry points reject before they
// get here -- so the caller runs the one-tile-per-CTA kernel.
template <bool ROWS, bool GROUPED, bool COLS, int FMT>
bool launch_cols_tma(const ColParams &P, int64_t row_tiles, cudaStream_t st, cudaError_t *res) {
    if ((reinterpret_cast<uintptr_t>(P.x) & 15) || (P.ldx % 8) || P.C >= (1ll << 31) || P.R >= (1ll << 31) ||
        P.R == 0)
        return false;
    CUtensorMap tm;
    if (!encode_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, P.x, static_cast<uint64_t>(P.C),
                        static_cast<uint64_t>(P.R), static_cast<uint64_t>(P.ldx) * 2, kTile, kTile,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
        return false;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) { *res = e; return true; }
    const int smem = QuantRing<GROUPED>::kSlots * static_cast<int>(kTileBytes);
    // per device, once, under a lock (host threads may launch concurrently): the
    // shared-memory attribute (a per-device setting) and the resident CTAs
    static std::mutex init_mu;
    static int64_t resident[64] = {0};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) { *res = e; return true; }
    if (dev < 0 || dev >= 64) { *res = cudaErrorInvalidDevice; return true; }
    int64_t ctas = 0;
    {
        std::lock_guard<std::mutex> lock(init_mu);
        if (resident[dev] == 0) {
            int per_sm = 0, sms = 0;
            if ((e = cudaFuncSetAttribute(k_quant_cols_tma<ROWS, GROUPED, COLS, FMT>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
                (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quant_cols_tma<ROWS, GROUPED, COLS, FMT>,
                                                                   kThreads, smem)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
                *res = e;
                return true;
            }
            resident[dev] = static_cast<int64_t>(per_sm < 1 ? 1 : per_sm) * (sms < 1 ? 1 : sms);
        }
        ctas = resident[dev];
    }
    const int64_t ct_tiles = (P.C + kTile - 1) / kTile;
    const int64_t n_tiles = row_tiles * ct_tiles;
    const int64_t grid = n_tiles < ctas ? n_tiles : ctas;
    // programmatic dependent launch (see pdl_wait in the kernel)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *res = cudaLaunchKernelEx(&cfg, k_quant_cols_tma<ROWS, GROUPED, COLS, FMT>, tm, P, n_tiles, ct_tiles, err);
    return true;
}

}  // namespace

cudaError_t launch_quant_cols(const uint16_t *x, int64_t R, int64_t C, int64_t ldx, uint8_t *q_row, uint8_t *s_row,
                              uint8_t *qT, uint8_t *sT, cudaStream_t st) {
    ColParams P{};
    P.x = x; P.R = R; P.C = C; P.ldx = ldx;
    P.q_row = q_row; P.s_row = s_row; P.kb_row_tiles = ((C / 32) + 3) / 4;
    P.qT = qT; P.sT = sT; P.ldqT = R; P.kb_col_tiles = (((R + 31) / 32) + 3) / 4;
    const int64_t row_tiles = (R + kTile - 1) / kTile;
    cudaError_t res = device_error_word(&P.err);
    if (res != cudaSuccess) return res;
    if (q_row ? launch_cols_tma<true, false>(P, row_tiles, st, &res) : launch_cols_tma<false, false>(P, row_tiles, st, &res))
        return res;
    const dim3 grid(static_cast<unsigned>((C + kTile - 1) / kTile), static_cast<unsigned>(row_tiles));
    if (q_row) (void)launch_pdl(k_quant_cols<true, false>, grid, kThreads, 0, st, P);
    else (void)launch_pdl(k_quant_cols<false, false>, grid, kThreads, 0, st, P);
    return cudaGetLastError();
}

cudaError_t launch_quant_cols_grouped(const uint16_t *x, int64_t T, int64_t C, const int64_t *d_off, int E,
                                      int64_t t_pad, uint8_t *q_row, uint8_t *s_row, uint8_t *qT, uint8_t *sT,
                                      cudaStream_t st, bool row_pad) {
    ColParams P{};
    P.x = x; P.R = T; P.C = C; P.ldx = C;
    P.q_row = q_row; P.s_row = s_row; P.kb_row_tiles = ((C / 32) + 3) / 4;
    P.qT = qT; P.sT = sT; P.ldqT = t_pad; P.kb_col_tiles = (t_pad / 32 + 3) / 4;
    P.offsets = d_off; P.E = E;
    P.row_pad = row_pad && q_row ? 1 : 0;
    cudaError_t res = device_error_word(&P.err);
    if (res != cudaSuccess) return res;
    if (P.row_pad && T == 0) {
        // no rows: every padded row scale is zero
        if ((res = cudaMemsetAsync(s_row, 0, static_cast<size_t>(t_pad / 128 * P.kb_row_tiles * 512), st)) !=
            cudaSuccess)
            return res;
    }
    if (q_row && T > 0) {
        if (launch_cols_tma<true, true>(P, t_pad / kTile, st, &res)) return res;
        // no tensor map for x (only a row count of 2^31 or more gets here, as
        // the entry points check x's alignment): the row quant on its own,
        // then the column quant; the padded row-scale layout needs the
        // combined kernel
        if (P.row_pad) return cudaErrorNotSupported;
        if ((res = launch_quant_rows(x, false, 0, T, C, C, q_row, s_row, st)) != cudaSuccess) return res;
    } else if (launch_cols_tma<false, true>(P, t_pad / kTile, st, &res)) {
        return res;
    }
    const dim3 grid(static_cast<unsigned>((C + kTile - 1) / kTile), static_cast<unsigned>(t_pad / kTile));
    (void)launch_pdl(k_quant_cols<false, true>, grid, kThreads, 0, st, P);
    return cudaGetLastError();
}

cudaError_t launch_qdq_mxfp4(const float *x, float *y, uint32_t *mask, int64_t rows, int64_t cols, float sf,
                             cudaStream_t st) {
    unsigned int *err = nullptr;
    cudaError_t ee = device_error_word(&err);
    if (ee != cudaSuccess) return ee;
    const bool vec = (cols % 32 == 0) && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) == 0;
    if (vec) {
        const int64_t nchunks = rows * cols / 8;
        const int grid = grid_windows(nchunks);
        if (mask) (void)launch_pdl(k_qdq_mxfp4_vec<true>, grid, kThreads, 0, st, x, y, mask, nchunks, sf, err);
        else (void)launch_pdl(k_qdq_mxfp4_vec<false>, grid, kThreads, 0, st, x, y, nullptr, nchunks, sf, err);
    } else {
        const int64_t nblocks = rows * ((cols + 31) / 32);
        const int grid = grid_for(nblocks, kThreads / 32);
        if (mask) (void)launch_pdl(k_qdq_mxfp4_gen<true>, grid, kThreads, 0, st, x, y, mask, rows, cols, sf, err);
        else (void)launch_pdl(k_qdq_mxfp4_gen<false>, grid, kThreads, 0, st, x, y, nullptr, rows, cols, sf, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_qdq_mxfp4_bf16(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols, float sf,
                                  cudaStream_t st) {
    unsigned int *err = nullptr;
    cudaError_t ee = device_error_word(&err);
    if (ee != cudaSuccess) return ee;
    const int64_t nblocks = rows * cols / 32;
    (void)launch_pdl(k_qdq_mxfp4_bf16, grid_windows(nblocks, kBlkWindow), kThreads, 0, st, x, y, nblocks, sf, err);
    return cudaGetLastError();
}

cudaError_t launch_ste_backward(const float *gy, const uint32_t *mask, float *gx, int64_t rows, int64_t cols,
                                cudaStream_t st) {
    unsigned int *err = nullptr;
    cudaError_t ee = device_error_word(&err);
    if (ee != cudaSuccess) return ee;
    const bool vec = (cols % 32 == 0) && ((reinterpret_cast<uintptr_t>(gy) | reinterpret_cast<uintptr_t>(gx)) & 15) == 0;
    if (vec) {
        const int64_t nchunks = rows * cols / 8;
        (void)launch_pdl(k_ste_backward_vec, grid_windows(nchunks), kThreads, 0, st, gy, mask, gx, nchunks, err);
    } else {
        const int64_t nblocks = rows * ((cols + 31) / 32);
        (void)launch_pdl(k_ste_backward_gen, grid_for(nblocks, kThreads / 32), kThreads, 0, st, gy, mask, gx, rows, cols, err);
    }
    return cudaGetLastError();
}

}  // namespace mxq
