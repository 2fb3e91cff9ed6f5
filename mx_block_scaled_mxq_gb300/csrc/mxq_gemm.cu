// mxq_gemm.cu -- block-scaled MXFP8 GEMM on the 5th-generation tensor cores.
//
// C = deq(A) deq(B)^T with E4M3 operands and E8M0 scales per 32-element block
// along K ("低精度训练特性（MXFP8 / HiFloat8）": the forward, input-gradient and
// weight-gradient products of the linear layer and of the experts' grouped
// matmul run on MXFP8 operands, output in bf16).  One kernel serves the dense
// GEMM and both grouped forms:
//   kDense       tiles (m, n) of one problem;
//   kGroupedRows tiles (expert, row tile overlapping the expert's token rows,
//                n); rows outside the expert are computed but not stored
//                (forward and input gradient of the MoE layer);
//   kGroupedK    tiles (expert, m, n) whose contraction runs over the expert's
//                padded token range only (weight gradient of the MoE layer).
//
// Persistent: each CTA (CG = 1) or CTA pair (CG = 2) walks its share of the
// tiles; the stage ring and the accumulator phases run across tiles.
// A CTA has 10 warps; the output tile is (128 * CG) x 256, K steps of 128 bytes:
//   warp 0     TMA producer: A/B code tiles (128B-swizzled) by
//              cp.async.bulk.tensor, 512-byte scale tiles (cp.async.bulk for
//              CG = 1, 2-D TMA for CG = 2);
//   warp 1     allocates 512 TMEM columns; one lane (of the even CTA for
//              CG = 2) copies the scale tiles to TMEM (tcgen05.cp
//              32x128b.warpx4) and issues 4 tcgen05.mma.kind::mxf8f6f4.block_scale
//              (M = 128 * CG, N = 256, K = 32) per stage; tcgen05.commit frees
//              the stage (in both CTAs of a pair);
//   warps 2-9  epilogue, two per TMEM lane sub-partition, each taking 128 of
//              the 256 columns: tcgen05.ld of the fp32 accumulator into
//              registers as bf16 (RNE), release of the accumulator to the MMA
//              warp, then stores that overlap the next tile's mainloop: 32 x 32
//              blocks staged in shared memory and written by TMA
//              (cp.async.bulk.tensor), or, for a warp whose 32 rows straddle an
//              expert boundary, masked 16-byte row stores.
// CG = 2 pairs two SMs on one 256 x 256 tile: each CTA loads 128 rows of A and
// 128 of the 256 rows of B (32 KB per stage, 6 stages), so per SM the operand
// traffic and the shared memory per stage are two thirds of CG = 1's, and the
// deeper ring hides more load latency.  Each CTA holds its own rows' A scales
// and all of B's scales; every load of both CTAs completes on the even CTA's
// stage barrier.
// Every TMA load lands in the shared memory of the CTA that issues it (no
// cluster multicast).
// TMEM: two accumulator banks of 256 columns; a tile in one bank keeps the
// scale slots of stage s in columns [16 s, 16 s + 12) of the other bank
// (A: 4 columns, B: 2 x 4 columns).  Every wait is bounded (mxq_device.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {

// Device error word (bits in mxq_device.cuh), read and cleared by
// read_and_clear_device_error().
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int BN = 256, BK = 128;
// Epilogue warps: two per TMEM lane quadrant, each draining and storing
// kEpiCols of the tile's 256 accumulator columns, so short-contraction tiles
// (the grouped weight gradient's small experts) are drained at twice the rate
// of one warp per quadrant.  Warps 0 and 1 are the producer and the MMA issuer.
constexpr int kEpiWarps = 8;
constexpr int kEpiCols = BN * 4 / kEpiWarps, kEpiChunks = kEpiCols / 32;
constexpr int THREADS = 64 + 32 * kEpiWarps;
// 2 KB store-staging slots per epilogue warp (shared memory holds 16 KB of them)
constexpr int kStoreSlots = 8 / kEpiWarps;
constexpr uint32_t TMEM_COLS = 512, SF_STRIDE = 16;
constexpr int kMaxTableE = 256;  // experts whose group tables are kept in shared memory
// Epilogue stores: true = 32 x 32 blocks staged in shared memory and written
// by TMA stores; false = coalesced 16-byte global stores after an in-register
// transpose.  On GB300 the two are within 1% of each other (dense forward
// 329 vs 327 us; MoE weight gradient 0.98 vs 0.99 ms).
constexpr bool kEpilogueTma = true;

template <int CG>
struct Cfg {
    static constexpr int BM = 128;           // rows of A per CTA (one TMEM lane each)
    static constexpr int TILE_M = 128 * CG;  // rows of one output tile
    static constexpr int B_ROWS = BN / CG;   // rows of B each CTA loads
    static constexpr int STAGES = CG == 1 ? 4 : 6;
    static constexpr uint32_t A_BYTES = BM * BK, B_BYTES = B_ROWS * BK, SFA_BYTES = 512, SFB_BYTES = 1024;
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
    // full / empty per stage; accumulator full / empty / drain, the second
    // accumulator bank's full / empty and both banks' "head drained" barriers
    static constexpr uint32_t NUM_BARS = 2 * STAGES + 7;
    static constexpr uint32_t OFF_MISC = OFF_BAR + 256;
    static constexpr uint32_t OFF_GRP = OFF_MISC + 256;  // group tables (grouped modes, E <= kMaxTableE)
    // epilogue store staging: kEpiWarps x kStoreSlots x (32 rows x 64 bytes), 1024-aligned
    static constexpr uint32_t OFF_STORE = (OFF_GRP + 3 * 8 * (kMaxTableE + 1) + 1023) / 1024 * 1024;
    static constexpr uint32_t SMEM_ALLOC = OFF_STORE + kEpiWarps * kStoreSlots * 2048 + 1024;  // + slack to align the base
    static_assert(NUM_BARS * 8 <= 256, "barrier area");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Division of n < 2^31 by a divisor d fixed for the launch, by a multiply-high
// and a shift (division by invariant integers using multiplication, Granlund
// and Montgomery, 1994).  With l = ceil(log2 d) and m = ceil(2^(31+l) / d):
// m < 2^32, and n * m / 2^(31+l) exceeds n / d by less than n * d / 2^(31+l)
// < 1 / d, so its floor is floor(n / d) for every n < 2^31.  The tile decode
// runs once per tile in three warps; a 64-bit division there costs hundreds of
// cycles.
struct FastDiv {
    uint32_t d, m, s;  // divisor, multiplier, shift l - 1 (unused for d = 1)
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) l++;
    const uint64_t m = ((1ull << (31 + l)) + d - 1) / d;
    return FastDiv{d, static_cast<uint32_t>(m), l > 0 ? l - 1 : 0};
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return f.d == 1 ? n : __umulhi(n, f.m) >> f.s;
}

struct Params {
    GemmMode mode;
    const uint8_t *sa, *sb;
    int64_t sa_kt, sb_kt;              // 512-byte scale tiles per 128-row group
    int64_t b_row_atoms;               // ceil(b_rows / 128)
    __nv_bfloat16 *c;
    int64_t M, N, ldc, K;
    const int64_t *offsets;
    int E;
    int64_t T;                         // grouped modes: token rows, the value off[E] must hold
    int64_t a_row_pad;                 // kGroupedRows: A's scales in the per-group padded layout (t_pad rows), or 0
    int64_t b_row_per_expert, b_k_per_expert, c_expert_stride;
    int m_tiles, n_tiles;  // tile counts (m in units of 128 * CG rows)
    FastDiv fd_m, fd_n, fd_mn;  // division by m_tiles, n_tiles, m_tiles * n_tiles
    int64_t c_expert_rows;      // kGroupedK: output rows per expert (c_expert_stride / ldc)
    int n_fastest;         // kDense tile order: 1 = n fastest (A is the larger operand)
    int tma_store;         // an output tensor map exists: unmasked 32-row boxes are stored with TMA
    int vec_store;         // rows of C are 16-byte aligned (coalesced 16-byte stores)
    const __nv_bfloat16 *bias;  // kDense: bf16 [N] added to every row in fp32, or null
    int64_t total_tiles;   // tile index space (an upper bound for grouped rows)
    uint64_t sa_bytes, sb_bytes, c_bytes;  // buffer extents (checked by debug builds)
};

struct TileInfo {
    int valid, nkb, k_last, b_atoms;
    int64_t a_row0, b_row0, a_k0, b_k0;   // this CTA's TMA coordinates of k-block 0
    int64_t a_ratom, b_ratom, a_katom0, b_katom0;
    int64_t row_lo, row_hi, out_row0, col0, col_hi, c_off;
    int64_t c_row0;  // first row of this expert's output block in the stacked output (kGroupedK), else 0
};

// Instruction descriptors, both operands K-major, N = 256, M = 128 * CG.
// kMXF8 (kind::mxf8f6f4): E4M3 x E4M3, E8M0 scales, scale-factor byte `j` of
// the A and B scale columns.  kBF16 (kind::f16): bf16 x bf16, fp32 accumulator.
template <int CG, int KIND>
__device__ __forceinline__ uint32_t make_idesc(uint32_t j) {
    if constexpr (KIND == kBF16) {
        return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
               (static_cast<uint32_t>(Cfg<CG>::TILE_M >> 4) << 24);
    } else {
        return (j << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
               (static_cast<uint32_t>(Cfg<CG>::TILE_M >> 4) << 24) | (j << 29);
    }
}

// acc[i] += bias[col + i] (fp32) for the columns below col_hi; every lane
// reads the same bias words (a broadcast).
__device__ __forceinline__ void add_bias32(uint32_t (&acc)[32], const __nv_bfloat16 *bias, int64_t col,
                                           int64_t col_hi) {
    const uint16_t *b = reinterpret_cast<const uint16_t *>(bias) + col;
    if (col + 32 <= col_hi) {
#pragma unroll
        for (int v = 0; v < 4; v++) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(b) + v);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                acc[8 * v + 2 * j] = __float_as_uint(__uint_as_float(acc[8 * v + 2 * j]) + __uint_as_float(ws[j] << 16));
                acc[8 * v + 2 * j + 1] =
                    __float_as_uint(__uint_as_float(acc[8 * v + 2 * j + 1]) + __uint_as_float(ws[j] & 0xFFFF0000u));
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; i++)
            if (col + i < col_hi)
                acc[i] = __float_as_uint(__uint_as_float(acc[i]) + __uint_as_float(static_cast<uint32_t>(__ldg(b + i)) << 16));
    }
}

// Work decomposition: which tile this CTA computes (run by all lanes of a warp).
// `rank` is the CTA's position in its pair (0 for CG = 1).
// Group tables a CTA builds once in shared memory (grouped modes with
// E <= kMaxTableE): off[e] = group offsets, pre[e] = exclusive prefix of the
// per-expert tile counts (kGroupedRows) or of the padded group lengths
// (kGroupedK), pst[e] = exclusive prefix of the padded group lengths
// (kGroupedRows with A's scales in the per-group padded layout: group e's
// first scale row).  Tiles are then decoded without touching global memory.
struct GroupTables {
    const int64_t *off, *pre, *pst;
};

// Row tiles of expert e in the grouped forward / dX, rows [o0, o1): with A's
// scales in the per-group padded layout the tiles start at the group's first
// row, so no row is computed twice; otherwise they are the TM-row tiles of
// the matrix that overlap the group.
template <int TM>
__device__ __forceinline__ int64_t expert_row_tiles(const Params &p, int64_t o0, int64_t o1) {
    if (o1 <= o0) return 0;
    return p.a_row_pad ? (o1 - o0 + TM - 1) / TM : (o1 - 1) / TM - o0 / TM + 1;
}

template <int CG>
__device__ void build_group_tables(const Params &p, int64_t *off, int64_t *pre, int64_t *pst, int warp, int lane) {
    constexpr int TM = Cfg<CG>::TILE_M;
    if (warp != 0) return;
    int64_t run = 0, run_p = 0;
    for (int base = 0; base <= p.E; base += 32) {
        const int e = base + lane;
        int64_t o0 = 0, o1 = 0;
        if (e <= p.E) { o0 = p.offsets[e]; off[e] = o0; }
        if (e < p.E) o1 = p.offsets[e + 1];
        int64_t v = 0, w = 0;
        if (e < p.E) {
            w = (o1 - o0 + 127) / 128 * 128;
            v = p.mode == kGroupedRows ? expert_row_tiles<TM>(p, o0, o1) * p.n_tiles : w;
        }
        int64_t incl = v, incl_p = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t u = __shfl_up_sync(0xffffffffu, incl, o), up = __shfl_up_sync(0xffffffffu, incl_p, o);
            if (lane >= o) { incl += u; incl_p += up; }
        }
        if (e <= p.E) { pre[e] = run + incl - v; pst[e] = run_p + incl_p - w; }
        run += __shfl_sync(0xffffffffu, incl, 31);
        run_p += __shfl_sync(0xffffffffu, incl_p, 31);
    }
}

template <int CG>
__device__ TileInfo resolve_tile(const Params &p, int64_t bid, int lane, uint32_t rank, const GroupTables &gt) {
    constexpr int TM = Cfg<CG>::TILE_M, BR = Cfg<CG>::B_ROWS;
    TileInfo t{};
    t.k_last = 4;
    int64_t tile_row0 = 0, bn0 = 0;  // first row of the tile; first row of B for the tile
    int64_t srow0 = -1;              // first scale row of the tile, where it differs from tile_row0
    if (p.mode == kGroupedRows && gt.off != nullptr) {
        // the expert whose tile range [pre[e], pre[e+1]) holds bid (binary search)
        if (bid >= gt.pre[p.E]) { t.valid = 0; return t; }
        int lo = 0, hi = p.E;  // pre[lo] <= bid < pre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (gt.pre[mid] <= bid) lo = mid; else hi = mid;
        }
        const int fe = lo;
        const int64_t fo0 = gt.off[fe], fo1 = gt.off[fe + 1];
        const int64_t mtiles_e = expert_row_tiles<TM>(p, fo0, fo1);
        const int64_t local = bid - gt.pre[fe];
        const uint32_t l32 = static_cast<uint32_t>(local), m32 = static_cast<uint32_t>(mtiles_e);
        const int64_t nt = l32 / m32, j = l32 - static_cast<uint32_t>(nt) * m32;
        t.valid = 1;
        tile_row0 = p.a_row_pad ? fo0 + j * TM : (fo0 / TM + j) * TM;
        if (p.a_row_pad) srow0 = gt.pst[fe] + j * TM;
        bn0 = fe * p.b_row_per_expert + nt * BN;
        t.b_k0 = fe * p.b_k_per_expert; t.b_katom0 = t.b_k0 / BK;
        t.col0 = nt * BN;
        t.row_lo = max(fo0, tile_row0 + 128 * rank);
        t.row_hi = min(fo1, tile_row0 + 128 * rank + 128);
    } else if (p.mode == kGroupedK && gt.off != nullptr) {
        const uint32_t b32 = static_cast<uint32_t>(bid), e32 = fdiv(b32, p.fd_mn);
        const int e = static_cast<int>(e32);
        const uint32_t local = b32 - e32 * p.fd_mn.d, nt32 = fdiv(local, p.fd_m);
        const int64_t nt = nt32, mt = local - nt32 * p.fd_m.d;
        const int64_t pe = gt.pre[e], ne = gt.off[e + 1] - gt.off[e];
        t.valid = 1;
        tile_row0 = mt * TM;
        bn0 = nt * BN;
        t.a_k0 = t.b_k0 = pe; t.a_katom0 = t.b_katom0 = pe / BK;
        t.nkb = static_cast<int>((ne + 127) / 128);
        t.col0 = nt * BN;
        t.row_lo = tile_row0 + 128 * rank;
        t.row_hi = min(p.M, t.row_lo + 128);
        t.c_off = static_cast<int64_t>(e) * p.c_expert_stride;
        t.c_row0 = static_cast<int64_t>(e) * p.c_expert_rows;
    } else if (p.mode == kDense) {
        // raster so that the smaller operand stays in L2 while the larger one
        // streams through once: concurrent CTAs share the larger operand's tile
        const uint32_t b32 = static_cast<uint32_t>(bid);
        const uint32_t q = fdiv(b32, p.n_fastest ? p.fd_n : p.fd_m), r = b32 - q * (p.n_fastest ? p.fd_n.d : p.fd_m.d);
        const int64_t mt = p.n_fastest ? q : r;
        const int64_t nt = p.n_fastest ? r : q;
        t.valid = 1;
        tile_row0 = mt * TM;
        bn0 = nt * BN;
        t.col0 = nt * BN;
        t.row_lo = tile_row0 + 128 * rank;
        t.row_hi = min(p.M, t.row_lo + 128);
    } else if (p.mode == kGroupedRows) {
        // tiles of expert e (expert_row_tiles), times n_tiles; the padded
        // starts P_e of the groups are summed alongside
        int64_t run = 0, run_p = 0;
        int fe = -1;
        int64_t fstart = 0, fo0 = 0, fo1 = 0, fpst = 0;
        for (int base = 0; base < p.E; base += 32) {
            const int e = base + lane;
            int64_t o0 = 0, o1 = 0;
            if (e < p.E) { o0 = p.offsets[e]; o1 = p.offsets[e + 1]; }
            const int64_t cnt = expert_row_tiles<TM>(p, o0, o1) * p.n_tiles, w = (o1 - o0 + 127) / 128 * 128;
            int64_t incl = cnt, incl_p = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t v = __shfl_up_sync(0xffffffffu, incl, o), vp = __shfl_up_sync(0xffffffffu, incl_p, o);
                if (lane >= o) { incl += v; incl_p += vp; }
            }
            const int64_t start = run + incl - cnt, pstart = run_p + incl_p - w;
            const bool mine = cnt > 0 && bid >= start && bid < start + cnt;
            const unsigned bal = __ballot_sync(0xffffffffu, mine);
            if (bal) {
                const int src = __ffs(bal) - 1;
                fe = base + src;
                fstart = __shfl_sync(0xffffffffu, start, src);
                fo0 = __shfl_sync(0xffffffffu, o0, src);
                fo1 = __shfl_sync(0xffffffffu, o1, src);
                fpst = __shfl_sync(0xffffffffu, pstart, src);
                break;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
            run_p += __shfl_sync(0xffffffffu, incl_p, 31);
        }
        if (fe < 0) { t.valid = 0; return t; }
        const int64_t mtiles_e = expert_row_tiles<TM>(p, fo0, fo1);
        const int64_t local = bid - fstart;
        const uint32_t l32 = static_cast<uint32_t>(local), m32 = static_cast<uint32_t>(mtiles_e);
        const int64_t nt = l32 / m32, j = l32 - static_cast<uint32_t>(nt) * m32;
        t.valid = 1;
        tile_row0 = p.a_row_pad ? fo0 + j * TM : (fo0 / TM + j) * TM;
        if (p.a_row_pad) srow0 = fpst + j * TM;
        bn0 = fe * p.b_row_per_expert + nt * BN;
        t.b_k0 = fe * p.b_k_per_expert; t.b_katom0 = t.b_k0 / BK;
        t.col0 = nt * BN;
        t.row_lo = max(fo0, tile_row0 + 128 * rank);
        t.row_hi = min(fo1, tile_row0 + 128 * rank + 128);
    } else {  // kGroupedK
        const uint32_t b32 = static_cast<uint32_t>(bid), e32 = fdiv(b32, p.fd_mn);
        const int e = static_cast<int>(e32);
        const uint32_t local = b32 - e32 * p.fd_mn.d, nt32 = fdiv(local, p.fd_m);
        const int64_t nt = nt32, mt = local - nt32 * p.fd_m.d;
        int64_t pe = 0;  // padded start of group e = sum_{j<e} ceil128(n_j)
        for (int base = 0; base < e; base += 32) {
            const int j = base + lane;
            if (j < e) pe += (p.offsets[j + 1] - p.offsets[j] + 127) / 128 * 128;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) pe += __shfl_xor_sync(0xffffffffu, pe, o);
        const int64_t ne = p.offsets[e + 1] - p.offsets[e];
        t.valid = 1;
        tile_row0 = mt * TM;
        bn0 = nt * BN;
        t.a_k0 = t.b_k0 = pe; t.a_katom0 = t.b_katom0 = pe / BK;
        t.nkb = static_cast<int>((ne + 127) / 128);
        t.col0 = nt * BN;
        t.row_lo = tile_row0 + 128 * rank;
        t.row_hi = min(p.M, t.row_lo + 128);
        t.c_off = static_cast<int64_t>(e) * p.c_expert_stride;
        t.c_row0 = static_cast<int64_t>(e) * p.c_expert_rows;
    }
    t.a_row0 = tile_row0 + 128 * rank;  // this CTA's 128 rows of A (and of the output)
    t.a_ratom = (srow0 >= 0 ? srow0 + 128 * rank : t.a_row0) / 128;
    t.out_row0 = t.a_row0;
    t.b_row0 = bn0 + BR * rank;         // this CTA's share of B's rows
    t.b_ratom = bn0 / 128;              // the tile's B scale tiles (all of them)
    t.col_hi = min(p.N, t.col0 + BN);
    if (p.mode != kGroupedK) {
        t.nkb = static_cast<int>((p.K + BK - 1) / BK);
        t.k_last = static_cast<int>((p.K - static_cast<int64_t>(t.nkb - 1) * BK) / 32);
    }
    if (p.mode == kGroupedRows) {
        t.b_atoms = (t.col0 + 128 < p.N) ? 2 : 1;
    } else {
        const int64_t left = p.b_row_atoms - t.b_ratom;
        t.b_atoms = left >= 2 ? 2 : static_cast<int>(left);
    }
    return t;
}

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Four K = 32 MMAs of one stage and the commit that frees the stage, with a
// non-blocking test of the NEXT stage's barrier issued first and its result
// read last, so the barrier check's latency overlaps the MMA issue instead of
// adding to it.  Returns whether the next stage's data has landed.
template <int CG, int KIND>
__device__ __forceinline__ bool mma4_commit_peek(uint32_t d_tmem, const uint64_t (&ad)[4], const uint64_t (&bd)[4],
                                                 const uint32_t (&id)[4], uint32_t sfa, uint32_t sfb,
                                                 uint32_t accumulate, uint32_t bar_empty_s, uint32_t bar_full_next,
                                                 uint32_t parity_next) {
    uint32_t ready;
    if constexpr (KIND == kBF16) {
        static_assert(CG == 1, "bf16 tiles are single-CTA");
        asm volatile(
            "{\n\t.reg .pred pn, pa, p1;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n\t"
            "setp.ne.b32 pa, %3, 0;\n\t"
            "setp.eq.u32 p1, 0, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%4], %5, %6, %7, pa;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%4], %8, %9, %7, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%4], %10, %11, %7, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%4], %12, %13, %7, p1;\n\t"
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%14];\n\t"
            "selp.u32 %0, 1, 0, pn;\n\t}"
            : "=r"(ready)
            : "r"(bar_full_next), "r"(parity_next), "r"(accumulate), "r"(d_tmem), "l"(ad[0]), "l"(bd[0]), "r"(id[0]),
              "l"(ad[1]), "l"(bd[1]), "l"(ad[2]), "l"(bd[2]), "l"(ad[3]), "l"(bd[3]), "r"(bar_empty_s)
            : "memory");
        (void)sfa;
        (void)sfb;
    } else if constexpr (CG == 2) {
        asm volatile(
            "{\n\t.reg .pred pn, pa, p1;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n\t"
            "setp.ne.b32 pa, %3, 0;\n\t"
            "setp.eq.u32 p1, 0, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %5, %6, %7, [%8], [%9], pa;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %10, %11, %12, [%8], [%9], p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %13, %14, %15, [%8], [%9], p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %16, %17, %18, [%8], [%9], p1;\n\t"
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%19], %20;\n\t"
            "selp.u32 %0, 1, 0, pn;\n\t}"
            : "=r"(ready)
            : "r"(bar_full_next), "r"(parity_next), "r"(accumulate), "r"(d_tmem), "l"(ad[0]), "l"(bd[0]), "r"(id[0]),
              "r"(sfa), "r"(sfb), "l"(ad[1]), "l"(bd[1]), "r"(id[1]), "l"(ad[2]), "l"(bd[2]), "r"(id[2]), "l"(ad[3]),
              "l"(bd[3]), "r"(id[3]), "r"(bar_empty_s), "h"(static_cast<uint16_t>(3))
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred pn, pa, p1;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n\t"
            "setp.ne.b32 pa, %3, 0;\n\t"
            "setp.eq.u32 p1, 0, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %5, %6, %7, [%8], [%9], pa;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %10, %11, %12, [%8], [%9], p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %13, %14, %15, [%8], [%9], p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], %16, %17, %18, [%8], [%9], p1;\n\t"
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%19];\n\t"
            "selp.u32 %0, 1, 0, pn;\n\t}"
            : "=r"(ready)
            : "r"(bar_full_next), "r"(parity_next), "r"(accumulate), "r"(d_tmem), "l"(ad[0]), "l"(bd[0]), "r"(id[0]),
              "r"(sfa), "r"(sfb), "l"(ad[1]), "l"(bd[1]), "r"(id[1]), "l"(ad[2]), "l"(bd[2]), "r"(id[2]), "l"(ad[3]),
              "l"(bd[3]), "r"(id[3]), "r"(bar_empty_s)
            : "memory");
    }
    return ready != 0;
}

// One whole k-block of the single-CTA bf16 path (kind::f16, no scales) in one
// asm block: the next stage's barrier test first, then the four K = 16 MMAs
// and the commit; the test result is read last.
__device__ __forceinline__ bool kblock_bf16_cg1(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t accumulate,
                                                uint32_t bar_empty_s, uint32_t bar_full_next, uint32_t parity_next) {
    constexpr uint32_t kAbHi = (1024u >> 4) | (1u << 14) | (2u << 29);
    constexpr uint32_t kId = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                             (static_cast<uint32_t>(128 >> 4) << 24);
    uint32_t ready;
    asm volatile(
        "{\n\t.reg .pred pn, pa, p1;\n\t.reg .b64 da, db;\n\t.reg .b32 ta, tb;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n\t"
        "setp.ne.b32 pa, %3, 0;\n\t"
        "setp.eq.u32 p1, 0, 0;\n\t"
        "mov.b64 da, {%5, %8};\n\t"
        "mov.b64 db, {%6, %8};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%4], da, db, %9, pa;\n\t"
        "add.u32 ta, %5, 2;\n\t" "add.u32 tb, %6, 2;\n\t"
        "mov.b64 da, {ta, %8};\n\t" "mov.b64 db, {tb, %8};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%4], da, db, %9, p1;\n\t"
        "add.u32 ta, %5, 4;\n\t" "add.u32 tb, %6, 4;\n\t"
        "mov.b64 da, {ta, %8};\n\t" "mov.b64 db, {tb, %8};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%4], da, db, %9, p1;\n\t"
        "add.u32 ta, %5, 6;\n\t" "add.u32 tb, %6, 6;\n\t"
        "mov.b64 da, {ta, %8};\n\t" "mov.b64 db, {tb, %8};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%4], da, db, %9, p1;\n\t"
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
        "selp.u32 %0, 1, 0, pn;\n\t}"
        : "=r"(ready)
        : "r"(bar_full_next), "r"(parity_next), "r"(accumulate), "r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(bar_empty_s),
          "n"(kAbHi), "n"(kId)
        : "memory");
    return ready != 0;
}

// One whole k-block of the single-CTA block-scaled path in one asm block:
// the non-blocking test of the NEXT stage's full barrier is issued first, then
// the three scale-tile copies (A, B rows 0-127, B rows 128-255) into TMEM, the
// four K = 32 MMAs and the commit that frees the stage; the test's result is
// read last, so its latency overlaps all of this stage's tcgen05 issue.
// Descriptors are assembled from per-stage 32-bit low words (start address
// >> 4) and constant high words; +32 bytes of K is +2 in the low word.
// Returns whether the next stage's data has landed.
__device__ __forceinline__ bool kblock_mxf8_cg1(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t sfa_t,
                                                uint32_t sfb_t, uint32_t sa_lo, uint32_t sb_lo, uint32_t accumulate,
                                                uint32_t bar_empty_s, uint32_t bar_full_next, uint32_t parity_next) {
    constexpr uint32_t kAbHi = (1024u >> 4) | (1u << 14) | (2u << 29);  // SBO 1024, version 1, 128-byte swizzle
    constexpr uint32_t kSfHi = (128u >> 4) | (1u << 14);                 // SBO 128, version 1, no swizzle
    constexpr uint32_t kId0 = (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(128 >> 4) << 24);
    uint32_t ready;
#define MXQ_KBLOCK_MXF8_BODY \
    "{\n\t.reg .pred pn, pa, p1;\n\t.reg .b64 da, db, ds;\n\t.reg .b32 ta, tb, tt;\n\t" \
    "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n\t" \
    "mov.b64 ds, {%9, %11};\n\t" \
    "tcgen05.cp.cta_group::1.32x128b.warpx4 [%7], ds;\n\t" \
    "mov.b64 ds, {%10, %11};\n\t" \
    "tcgen05.cp.cta_group::1.32x128b.warpx4 [%8], ds;\n\t" \
    "add.u32 tt, %10, 32;\n\t" \
    "mov.b64 ds, {tt, %11};\n\t" \
    "add.u32 tt, %8, 4;\n\t" \
    "tcgen05.cp.cta_group::1.32x128b.warpx4 [tt], ds;\n\t" \
    "setp.ne.b32 pa, %3, 0;\n\t" \
    "setp.eq.u32 p1, 0, 0;\n\t" \
    "mov.b64 da, {%5, %12};\n\t" \
    "mov.b64 db, {%6, %12};\n\t" \
    "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], da, db, %13, [%7], [%8], pa;\n\t" \
    "add.u32 ta, %5, 2;\n\t" \
    "add.u32 tb, %6, 2;\n\t" \
    "mov.b64 da, {ta, %12};\n\t" \
    "mov.b64 db, {tb, %12};\n\t" \
    "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], da, db, %14, [%7], [%8], p1;\n\t" \
    "add.u32 ta, %5, 4;\n\t" \
    "add.u32 tb, %6, 4;\n\t" \
    "mov.b64 da, {ta, %12};\n\t" \
    "mov.b64 db, {tb, %12};\n\t" \
    "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], da, db, %15, [%7], [%8], p1;\n\t" \
    "add.u32 ta, %5, 6;\n\t" \
    "add.u32 tb, %6, 6;\n\t" \
    "mov.b64 da, {ta, %12};\n\t" \
    "mov.b64 db, {tb, %12};\n\t" \
    "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%4], da, db, %16, [%7], [%8], p1;\n\t"
    asm volatile(MXQ_KBLOCK_MXF8_BODY
                 "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%17];\n\t"
                 "selp.u32 %0, 1, 0, pn;\n\t}"
                 : "=r"(ready)
                 : "r"(bar_full_next), "r"(parity_next), "r"(accumulate), "r"(d_tmem), "r"(a_lo), "r"(b_lo),
                   "r"(sfa_t), "r"(sfb_t), "r"(sa_lo), "r"(sb_lo), "n"(kSfHi), "n"(kAbHi), "n"(kId0),
                   "n"(kId0 | (1u << 4) | (1u << 29)), "n"(kId0 | (2u << 4) | (2u << 29)),
                   "n"(kId0 | (3u << 4) | (3u << 29)), "r"(bar_empty_s)
                 : "memory");
#undef MXQ_KBLOCK_MXF8_BODY
    return ready != 0;
}

template <int CG, int KIND, bool BIAS>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                const __grid_constant__ CUtensorMap tmC, const Params p) {
    using C = Cfg<CG>;
    constexpr bool CLUSTER = CG == 2;             // CTAs work in pairs
    constexpr int STAGES = C::STAGES;
    // the scale-slot columns [0, STAGES * 16) are drained by the epilogue warps
    // of column part 0, in their 64-column step kHeadStep
    constexpr int kHeadStep = (STAGES * SF_STRIDE - 1) / 64;
    static_assert(STAGES * SF_STRIDE <= kEpiCols, "scale slots lie in column part 0");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    pdl_launch_dependents();
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar_full = sbase + C::OFF_BAR, bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_accf = bar_full + 16 * STAGES, bar_acce = bar_accf + 8, bar_drain = bar_accf + 16;
    // Two accumulator banks: tile t accumulates in TMEM columns [256 b, 256 b +
    // 256), b = t % 2, and keeps its scale slots in the first STAGES * 16 columns
    // of the other bank.  The MMA warp starts tile t once tile t - 2 has been
    // drained from bank b and the epilogue has read the head of tile t - 1 (the
    // columns that hold tile t's scale slots; this also means tile t - 1's MMAs
    // are done), so the next tile's MMAs overlap most of the previous tile's
    // drain.  For a CTA pair the bank's release and "head read" barriers live in
    // the even CTA and count the epilogue warps of both CTAs.
    const uint32_t bar_accf1 = bar_accf + 24, bar_acce1 = bar_accf + 32;
    const uint32_t bar_headf0 = bar_accf + 40, bar_headf1 = bar_accf + 48;
    uint32_t rank = 0;
    if constexpr (CLUSTER) rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t first = CLUSTER ? blockIdx.x >> 1 : blockIdx.x;
    const int64_t step = CLUSTER ? gridDim.x >> 1 : gridDim.x;

    // The prologue below touches no global memory (tensor maps are kernel
    // parameters), so it runs before pdl_wait, overlapping the previous
    // kernel's last wave: this CTA only lands on an SM that kernel's CTAs have
    // left, so the tensor memory is free.
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if constexpr (CG == 2) {
            prefetch_tmap(&tmSA);
            prefetch_tmap(&tmSB);
        }
    }
    if (warp == 1) {
        if (lane == 0) {
            for (int s = 0; s < STAGES; s++) {
                mbar_init(bar_full + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, 1);
            }
            mbar_init(bar_accf, 1);
            mbar_init(bar_accf1, 1);
            // one arrival per epilogue warp (of both CTAs of a pair); the head
            // is read by the 4 warps of column part 0
            mbar_init(bar_acce, kEpiWarps * CG);
            mbar_init(bar_acce1, kEpiWarps * CG);
            mbar_init(bar_headf0, 4 * CG);
            mbar_init(bar_headf1, 4 * CG);
            mbar_init(bar_drain, 1);
            fence_mbar_init();
        }
        __syncwarp();
        if constexpr (CG == 2) {
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (CLUSTER) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // no global access before the previous kernel in the stream has completed
    // once any CTA has given up, the rest of the grid does no work (it still
    // leaves through the teardown below, which frees the tensor memory)
    if (threadIdx.x == 0) *abort_flag = *reinterpret_cast<volatile unsigned int *>(&g_device_error) != 0 ? 1 : 0;
    __syncthreads();
    GroupTables gt{nullptr, nullptr, nullptr};
    if (p.mode != kDense) {
        // malformed offsets: no tile is decoded from them, no load or store is issued
        if (warp == 0 && !group_offsets_valid(p.offsets, p.E, p.T, lane) && lane == 0) {
            *abort_flag = 1;
            atomicOr(&g_device_error, kErrBadOffsets);
        }
        __syncthreads();
    }
    if (p.mode != kDense && p.E <= kMaxTableE && !*abort_flag) {
        int64_t *off = reinterpret_cast<int64_t *>(smem + C::OFF_GRP), *pre = off + kMaxTableE + 1;
        int64_t *pst = pre + kMaxTableE + 1;
        build_group_tables<CG>(p, off, pre, pst, warp, lane);
        __syncthreads();
        gt.off = off;
        gt.pre = pre;
        gt.pst = pst;
    }
    // stage barriers and the accumulator-release barriers of the even CTA
    uint32_t lead_full = bar_full, lead_acce = bar_acce, lead_headf0 = bar_headf0;
    if constexpr (CG == 2) {
        lead_full = mapa_shared(bar_full, 0);
        lead_acce = mapa_shared(bar_acce, 0);
        lead_headf0 = mapa_shared(bar_headf0, 0);
    }
    const bool run = *abort_flag == 0;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        uint32_t g = 0;  // k-blocks issued by this CTA (lane 0)
        for (int64_t tile = first; run && tile < p.total_tiles; tile += step) {
            const TileInfo ti = resolve_tile<CG>(p, tile, lane, rank, gt);
            if (!ti.valid) break;  // grouped-row tiles past the real count come last
            int stop = 0;
            if (lane == 0) {
                for (int kb = 0; kb < ti.nkb; kb++, g++) {
                    const uint32_t s = g % STAGES, ph = (g / STAGES) & 1;
                    if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, &g_device_error)) { stop = 1; break; }
                    const uint32_t sa_s = sbase + C::OFF_A + s * C::A_BYTES, sb_s = sbase + C::OFF_B + s * C::B_BYTES;
                    const uint32_t sfa_s = sbase + C::OFF_SFA + s * C::SFA_BYTES;
                    const uint32_t sfb_s = sbase + C::OFF_SFB + s * C::SFB_BYTES;
                    const int ka = static_cast<int>(ti.a_k0 + kb * BK), kb_ = static_cast<int>(ti.b_k0 + kb * BK);
                    if constexpr (KIND == kBF16) {
                        const uint32_t fb = bar_full + 8 * s;
                        mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                        tma_load_2d(sa_s, &tmA, fb, ka, static_cast<int>(ti.a_row0));
                        tma_load_2d(sb_s, &tmB, fb, kb_, static_cast<int>(ti.b_row0));
                        (void)sfa_s;
                        (void)sfb_s;
                    } else if constexpr (CG == 1) {
                        const uint32_t fb = bar_full + 8 * s;
                        mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES + C::SFA_BYTES + 512u * ti.b_atoms);
                        tma_load_2d(sa_s, &tmA, fb, ka, static_cast<int>(ti.a_row0));
                        tma_load_2d(sb_s, &tmB, fb, kb_, static_cast<int>(ti.b_row0));
                        const uint8_t *sa_src = p.sa + (ti.a_ratom * p.sa_kt + ti.a_katom0 + kb) * 512;
                        // (a skipped copy leaves its bytes missing: the stage's wait times out)
                        if (MXQ_IN_BOUNDS(sa_src, 512, p.sa, p.sa_bytes, &g_device_error)) bulk_load(sfa_s, sa_src, 512, fb);
                        for (int h = 0; h < ti.b_atoms; h++) {
                            const uint8_t *sb_src = p.sb + ((ti.b_ratom + h) * p.sb_kt + ti.b_katom0 + kb) * 512;
                            if (MXQ_IN_BOUNDS(sb_src, 512, p.sb, p.sb_bytes, &g_device_error))
                                bulk_load(sfb_s + 512 * h, sb_src, 512, fb);
                        }
                    } else {
                        // both CTAs' loads complete on the even CTA's barrier, which
                        // expects the bytes of both (scale tiles past the buffer are
                        // zero-filled by TMA and still counted)
                        const uint32_t fb = lead_full + 8 * s;
                        if (leader)
                            mbar_arrive_expect_tx(bar_full + 8 * s,
                                                  2 * (C::A_BYTES + C::B_BYTES + C::SFA_BYTES + C::SFB_BYTES));
                        tma_load_2d_pair(sa_s, &tmA, fb, ka, static_cast<int>(ti.a_row0));
                        tma_load_2d_pair(sb_s, &tmB, fb, kb_, static_cast<int>(ti.b_row0));
                        tma_load_2d_pair(sfa_s, &tmSA, fb, 0,
                                         static_cast<int>((ti.a_ratom * p.sa_kt + ti.a_katom0 + kb) * 4));
                        for (int h = 0; h < 2; h++)
                            tma_load_2d_pair(sfb_s + 512 * h, &tmSB, fb, 0,
                                             static_cast<int>(((ti.b_ratom + h) * p.sb_kt + ti.b_katom0 + kb) * 4));
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        if (lane == 0 && *abort_flag) {  // let this CTA's copies land before it exits
            if constexpr (CG == 1) {
                for (uint32_t j = g > STAGES ? g - STAGES : 0; j < g; j++)
                    mbar_wait_drain(bar_full + 8 * (j % STAGES), (j / STAGES) & 1);
            } else {
                spin_ns(2000000);  // the pair's loads complete on the other CTA's barriers
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (CG == 1 || leader) {
            uint32_t g = 0, acc_it = 0;
            bool issued_any = false;
            // descriptor low words (start address >> 4) of stage 0's operand and scale tiles
            const uint32_t a_lo0 = (sbase + C::OFF_A) >> 4, b_lo0 = (sbase + C::OFF_B) >> 4;
            const uint32_t sa_lo0 = (sbase + C::OFF_SFA) >> 4, sb_lo0 = (sbase + C::OFF_SFB) >> 4;
            for (int64_t tile = first; run && tile < p.total_tiles; tile += step) {
                const TileInfo ti = resolve_tile<CG>(p, tile, lane, rank, gt);
                if (!ti.valid) break;
                if (ti.nkb == 0) continue;  // empty group: the epilogue writes zeros
                int stop = 0;
                // accumulator bank and scale-slot base of this tile
                const uint32_t bank = acc_it & 1;
                const uint32_t d_tmem = tmem + 256 * bank;
                const uint32_t sf_base = tmem + 256 * (1 - bank);
                if (lane == 0) {
                    // bank drained of tile t - 2; head of tile t - 1 drained
                    if (acc_it >= 2 && !mbar_wait(bank ? bar_acce1 : bar_acce, ((acc_it - 2) >> 1) & 1, abort_flag,
                                                  &g_device_error))
                        stop = 1;
                    if (!stop && acc_it >= 1 &&
                        !mbar_wait(bank ? bar_headf0 : bar_headf1, ((acc_it - 1) >> 1) & 1, abort_flag, &g_device_error))
                        stop = 1;
                    tc_fence_after();
                    bool ready = false;  // stage g known to have landed (from the previous stage's peek)
                    int kb0 = 0;         // first k-block left to the general loop below
                    if constexpr (CG == 1) {
                        // every k-block but a short last one: one asm block each
                        const int nfull = ti.k_last == 4 ? ti.nkb : ti.nkb - 1;
                        for (; kb0 < nfull; kb0++, g++) {
                            const uint32_t s = g % STAGES, ph = (g / STAGES) & 1;
                            if (!ready && !mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_device_error)) {
                                stop = 1;
                                break;
                            }
                            tc_fence_after();
                            issued_any = true;
                            const uint32_t s1 = (g + 1) % STAGES, ph1 = ((g + 1) / STAGES) & 1;
                            if constexpr (KIND == kBF16) {
                                ready = kblock_bf16_cg1(d_tmem, a_lo0 + s * (C::A_BYTES >> 4),
                                                        b_lo0 + s * (C::B_BYTES >> 4), kb0 != 0 ? 1u : 0u,
                                                        bar_empty + 8 * s, bar_full + 8 * s1, ph1);
                            } else {
                                const uint32_t sf_t = sf_base + s * SF_STRIDE;
                                ready = kblock_mxf8_cg1(d_tmem, a_lo0 + s * (C::A_BYTES >> 4),
                                                        b_lo0 + s * (C::B_BYTES >> 4), sf_t, sf_t + 4,
                                                        sa_lo0 + s * (C::SFA_BYTES >> 4),
                                                        sb_lo0 + s * (C::SFB_BYTES >> 4), kb0 != 0 ? 1u : 0u,
                                                        bar_empty + 8 * s, bar_full + 8 * s1, ph1);
                            }
                        }
                    }
                    for (int kb = kb0; kb < ti.nkb && !stop; kb++, g++) {
                        const uint32_t s = g % STAGES, ph = (g / STAGES) & 1;
                        if (!ready && !mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_device_error)) { stop = 1; break; }
                        tc_fence_after();
                        const uint32_t sfa_t = sf_base + s * SF_STRIDE, sfb_t = sfa_t + 4;
                        const uint64_t dA = smem_desc(sbase + C::OFF_SFA + s * C::SFA_BYTES, 0, 128, 0);
                        const uint64_t dB0 = smem_desc(sbase + C::OFF_SFB + s * C::SFB_BYTES, 0, 128, 0);
                        const uint64_t dB1 = smem_desc(sbase + C::OFF_SFB + s * C::SFB_BYTES + 512, 0, 128, 0);
                        if constexpr (KIND == kBF16) {
                            (void)dA;  // no scales
                            (void)dB0;
                            (void)dB1;
                        } else if constexpr (CG == 2) {
                            tc_cp_32x128b_warpx4_pair(sfa_t, dA);
                            tc_cp_32x128b_warpx4_pair(sfb_t, dB0);
                            tc_cp_32x128b_warpx4_pair(sfb_t + 4, dB1);
                        } else {
                            tc_cp_32x128b_warpx4(sfa_t, dA);
                            tc_cp_32x128b_warpx4(sfb_t, dB0);
                            tc_cp_32x128b_warpx4(sfb_t + 4, dB1);
                        }
                        const int kk = (kb == ti.nkb - 1) ? ti.k_last : 4;
                        issued_any = true;
                        if (kk == 4 && kb + 1 < ti.nkb) {
                            uint64_t ad[4], bd[4];
                            uint32_t id[4];
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                ad[j] = smem_desc(sbase + C::OFF_A + s * C::A_BYTES + 32 * j, 0, 1024, 2);
                                bd[j] = smem_desc(sbase + C::OFF_B + s * C::B_BYTES + 32 * j, 0, 1024, 2);
                                id[j] = make_idesc<CG, KIND>(j);
                            }
                            const uint32_t s1 = (g + 1) % STAGES, ph1 = ((g + 1) / STAGES) & 1;
                            ready = mma4_commit_peek<CG, KIND>(d_tmem, ad, bd, id, sfa_t, sfb_t, kb != 0 ? 1u : 0u,
                                                         bar_empty + 8 * s, bar_full + 8 * s1, ph1);
                            continue;
                        }
                        for (int j = 0; j < kk; j++) {
                            const uint64_t ad = smem_desc(sbase + C::OFF_A + s * C::A_BYTES + 32 * j, 0, 1024, 2);
                            const uint64_t bd = smem_desc(sbase + C::OFF_B + s * C::B_BYTES + 32 * j, 0, 1024, 2);
                            const uint32_t acc = (kb | j) != 0 ? 1u : 0u;
                            if constexpr (KIND == kBF16)
                                tc_mma_bf16(d_tmem, ad, bd, make_idesc<CG, KIND>(j), acc);
                            else if constexpr (CG == 2)
                                tc_mma_mxf8_pair(d_tmem, ad, bd, make_idesc<CG, KIND>(j), sfa_t, sfb_t, acc);
                            else
                                tc_mma_mxf8(d_tmem, ad, bd, make_idesc<CG, KIND>(j), sfa_t, sfb_t, acc);
                        }
                        if constexpr (CG == 2) tc_commit_pair_mc(bar_empty + 8 * s, 3);
                        else tc_commit(bar_empty + 8 * s);
                        ready = false;
                    }
                    if (!stop) {
                        if constexpr (CG == 2) tc_commit_pair_mc(bank ? bar_accf1 : bar_accf, 3);
                        else tc_commit(bank ? bar_accf1 : bar_accf);
                    }
                }
                acc_it++;
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
            }
            if (lane == 0 && issued_any && *abort_flag) {  // no MMA in flight at dealloc
                if constexpr (CG == 2) tc_commit_pair_mc(bar_drain, 1);
                else tc_commit(bar_drain);
                mbar_wait_drain(bar_drain, 0);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        // Drain the accumulator into registers (bf16), release it to the MMA
        // warp, then store: the global stores overlap the next tile's mainloop.
        // Two warps per TMEM lane quadrant: warp `ew` drains rows 32 sub ..
        // 32 sub + 31 (its quadrant) of columns [kEpiCols part, +kEpiCols).
        const int ew = warp - 2, sub = warp & 3, part = ew >> 2;
        uint32_t acc_it = 0;
        const uint32_t st_slots = sbase + C::OFF_STORE + kStoreSlots * 2048 * ew;  // this warp's staging slots
        uint32_t st_count = 0;                                                     // blocks this warp has stored
        for (int64_t tile = first; run && tile < p.total_tiles; tile += step) {
            const TileInfo ti = resolve_tile<CG>(p, tile, lane, rank, gt);
            if (!ti.valid) break;
            const int64_t grow = ti.out_row0 + 32 * sub + lane;
            const bool row_ok = grow >= ti.row_lo && grow < ti.row_hi;
            __nv_bfloat16 *crow = p.c + ti.c_off + grow * p.ldc;
            const int64_t pcol0 = ti.col0 + kEpiCols * part;  // first column of this warp's part
            if (ti.nkb == 0) {  // empty group: its weight gradient is zero
                if (row_ok) {
                    const int64_t pend = min(ti.col_hi, pcol0 + kEpiCols);
                    int64_t col = pcol0;
                    for (; col + 8 <= pend; col += 8)
                        if (MXQ_IN_BOUNDS(crow + col, 16, p.c, p.c_bytes, &g_device_error))
                            *reinterpret_cast<uint4 *>(crow + col) = make_uint4(0, 0, 0, 0);
                    for (; col < pend; col++)
                        if (MXQ_IN_BOUNDS(crow + col, 2, p.c, p.c_bytes, &g_device_error))
                            crow[col] = __float2bfloat16_rn(0.0f);
                }
                continue;
            }
            const uint32_t bank = acc_it & 1;
            if (!mbar_wait(bank ? bar_accf1 : bar_accf, (acc_it >> 1) & 1, abort_flag, &g_device_error)) break;
            tc_fence_after();
            const uint32_t acc_t = tmem + 256 * bank + (static_cast<uint32_t>(32 * sub) << 16);
            // How this warp's 32 x 32 blocks are stored (warp-uniform):
            //  1: 4 x 4 transposes of 16-byte chunks inside each group of 4 lanes
            //     (two xor-shuffle rounds, in place) leave lane 4g + c with chunk
            //     c of rows 4g .. 4g + 3, so each store instruction writes 8 rows
            //     x 64 contiguous bytes; rows outside the tile's output are
            //     masked per lane, a block cut by the last column goes row by row;
            //  2: staged in a 64-byte-swizzled slot (conflict-free 16-byte writes)
            //     and stored by TMA, which takes whole 32-row boxes -- this warp's
            //     rows must all belong to the tile's output (always for dense
            //     problems, where the tensor map clips rows past M and columns
            //     past N; grouped tiles mask rows of other experts);
            //  0: each lane stores its own row.
            const int64_t wrow0 = ti.out_row0 + 32 * sub;
            const int smode = (!kEpilogueTma && p.vec_store) ? 1
                              : (p.tma_store && (p.mode == kDense || (wrow0 >= ti.row_lo && wrow0 + 32 <= ti.row_hi)))
                                  ? 2
                                  : 0;
            const int c4 = lane & 3;
            const int64_t r0 = wrow0 + 4 * (lane >> 2);
            unsigned rmask = 0;
#pragma unroll
            for (int k = 0; k < 4; k++) rmask |= (r0 + k >= ti.row_lo && r0 + k < ti.row_hi ? 1u : 0u) << k;
            auto store_chunk = [&](int lc, uint32_t (&m)[16]) {
                const int64_t col = pcol0 + 32 * lc;
                if (col >= ti.col_hi) return;  // warp-uniform
                if (smode == 1) {
                    if (col + 32 <= ti.col_hi) {  // m: chunk j, word w at m[4 * j + w]
#pragma unroll
                        for (int j = 0; j < 4; j += 2)
#pragma unroll
                            for (int w = 0; w < 4; w++) {
                                const uint32_t snd = (lane & 1) ? m[4 * j + w] : m[4 * j + 4 + w];
                                const uint32_t rcv = __shfl_xor_sync(0xffffffffu, snd, 1);
                                if (lane & 1) m[4 * j + w] = rcv;
                                else m[4 * j + 4 + w] = rcv;
                            }
#pragma unroll
                        for (int j = 0; j < 2; j++)
#pragma unroll
                            for (int w = 0; w < 4; w++) {
                                const uint32_t snd = (lane & 2) ? m[4 * j + w] : m[4 * j + 8 + w];
                                const uint32_t rcv = __shfl_xor_sync(0xffffffffu, snd, 2);
                                if (lane & 2) m[4 * j + w] = rcv;
                                else m[4 * j + 8 + w] = rcv;
                            }
                        uint8_t *wp = reinterpret_cast<uint8_t *>(p.c + ti.c_off + r0 * p.ldc + col + 8 * c4);
#pragma unroll
                        for (int k = 0; k < 4; k++)
                            if ((rmask & (1u << k)) && MXQ_IN_BOUNDS(wp + k * p.ldc * 2, 16, p.c, p.c_bytes, &g_device_error))
                                *reinterpret_cast<uint4 *>(wp + k * p.ldc * 2) =
                                    make_uint4(m[4 * k], m[4 * k + 1], m[4 * k + 2], m[4 * k + 3]);
                        return;
                    }
                } else if (smode == 2) {
                    const uint32_t slot = st_slots + 2048 * (st_count % kStoreSlots);
                    if (st_count >= static_cast<uint32_t>(kStoreSlots)) {  // the slot's previous store has read it
                        if (lane == 0) bulk_wait_read<kStoreSlots - 1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint32_t dst = slot + 64 * lane + 16 * (q ^ ((lane >> 1) & 3));
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(m[4 * q]),
                                     "r"(m[4 * q + 1]), "r"(m[4 * q + 2]), "r"(m[4 * q + 3])
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, slot, static_cast<int>(col), static_cast<int>(ti.c_row0 + wrow0));
                        bulk_commit_group();
                    }
                    st_count++;
                    return;
                }
                if (!row_ok) return;
                if (col + 32 <= ti.col_hi) {
                    uint4 *dst = reinterpret_cast<uint4 *>(crow + col);
                    if (MXQ_IN_BOUNDS(dst, 64, p.c, p.c_bytes, &g_device_error)) {
#pragma unroll
                        for (int i = 0; i < 4; i++) dst[i] = make_uint4(m[4 * i], m[4 * i + 1], m[4 * i + 2], m[4 * i + 3]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        if (col + i < ti.col_hi && MXQ_IN_BOUNDS(crow + col + i, 2, p.c, p.c_bytes, &g_device_error))
                            reinterpret_cast<uint16_t *>(crow)[col + i] = static_cast<uint16_t>(m[i >> 1] >> (16 * (i & 1)));
                }
            };
            // Drain this warp's part: two TMEM loads in flight per wait, rounded
            // to bf16 as they arrive; the accumulator goes back to the MMA warp
            // as soon as the last load has landed, and the stores follow.
            uint32_t pk[kEpiChunks][16];
#pragma unroll
            for (int h = 0; h < kEpiChunks / 2; h++) {
                uint32_t r[2][32];
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    const int ch = kEpiChunks * part + 2 * h + q;
                    if (ti.col0 + 32 * ch < ti.col_hi)  // warp-uniform
                        tmem_ld_32x32b_x32(acc_t + 32 * ch, r[q]);
                }
                tc_wait_ld();
                if (part == 0 && h == kHeadStep) {  // head read: the next tile may put its scales there
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (CG == 2) mbar_arrive_cluster(lead_headf0 + 8 * bank);
                        else mbar_arrive(bar_headf0 + 8 * bank);
                    }
                }
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    const int ch = kEpiChunks * part + 2 * h + q;
                    if (ti.col0 + 32 * ch < ti.col_hi) {
                        if constexpr (BIAS) add_bias32(r[q], p.bias, ti.col0 + 32 * ch, ti.col_hi);
#pragma unroll
                        for (int i = 0; i < 16; i++)
                            pk[2 * h + q][i] = pack_bf16x2(__uint_as_float(r[q][2 * i]), __uint_as_float(r[q][2 * i + 1]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 2) mbar_arrive_cluster(bank ? lead_acce + 24 : lead_acce);
                else mbar_arrive(bank ? bar_acce1 : bar_acce);
            }
            acc_it++;
#pragma unroll
            for (int lc = 0; lc < kEpiChunks; lc++) store_chunk(lc, pk[lc]);
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_all();  // staged stores done before shared memory goes away
    tc_fence_before();
    if constexpr (CLUSTER) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (CG == 2) tmem_dealloc_pair(tmem, TMEM_COLS);
        else tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D K-major fp8 operand [rows x k], box 128 bytes x box_rows, 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const uint8_t *base, int64_t rows, int64_t k, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A swz scale buffer of `bytes` bytes seen as rows of 128 bytes; one box of
// 4 rows is one 512-byte scale tile.
bool make_scale_tmap(CUtensorMap *m, const uint8_t *base, int64_t bytes) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(bytes / 128)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 4};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output [rows x n] with leading dimension ld (elements); 32 x 32 boxes,
// 64-byte swizzle (the staging slots' layout).
bool make_out_tmap(CUtensorMap *m, void *base, int64_t rows, int64_t n, int64_t ld) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t scale_bytes_of(int64_t rows, int64_t k) { return (rows + 127) / 128 * 128 * ((k / 32 + 3) / 4 * 4); }

// CTAs per tile.  Single-CTA tiles are the default: on GB300 the pair tile
// moves a third less operand data per SM and, without its scale copies, runs
// the dense 8192 x 14336 x 4096 product in 305 us against 325 us, but each
// tcgen05.cp.cta_group::2 costs about 50 clocks of MMA issue while MMAs are in
// flight, and its three copies per k-block bring it to 363 us.
// MXQ_GEMM_CTA_GROUP=2 selects pair tiles (read once per process).
int cta_group_for(const GemmProblem &) {
    static int forced = [] {
        const char *v = getenv("MXQ_GEMM_CTA_GROUP");
        return v ? atoi(v) : 0;
    }();
    return forced == 2 ? 2 : 1;
}

template <int CG, int KIND, bool BIAS>
cudaError_t launch_cg(const GemmProblem &g, Params p, cudaStream_t st) {
    using C = Cfg<CG>;
    CUtensorMap tmA, tmB, tmSA, tmSB, tmC;
    const int64_t esz = KIND == kBF16 ? 2 : 1;  // operand bytes per element (tensor maps run over bytes)
    if (!make_tmap(&tmA, g.a, g.a_rows, esz * g.a_k, C::BM) ||
        !make_tmap(&tmB, g.b, g.b_rows, esz * g.b_k, C::B_ROWS))
        return cudaErrorInvalidValue;
    if (CG == 2) {
        if (!make_scale_tmap(&tmSA, g.sa, scale_bytes_of(p.a_row_pad ? p.a_row_pad : g.a_rows, g.a_k)) ||
            !make_scale_tmap(&tmSB, g.sb, scale_bytes_of(g.b_rows, g.b_k)))
            return cudaErrorInvalidValue;
    } else {
        tmSA = tmA;  // unused
        tmSB = tmB;
    }
    constexpr int64_t kUnitRows = C::TILE_M;  // rows per CTA (pair)
    p.m_tiles = static_cast<int>((g.M + kUnitRows - 1) / kUnitRows);
    // output tensor map for the epilogue's TMA stores (all experts' outputs
    // stacked for the grouped weight gradient); without one (ldc not a
    // multiple of 8, or rows past the 32-bit TMA coordinate range) every
    // store is a plain global store
    const int64_t c_rows = g.mode == kGroupedK ? static_cast<int64_t>(g.E) * g.M : g.M;
    p.tma_store = c_rows < (1ll << 31) && make_out_tmap(&tmC, g.c, c_rows, g.N, g.ldc) ? 1 : 0;
    p.vec_store = (g.ldc % 8 == 0 && (reinterpret_cast<uintptr_t>(g.c) & 15) == 0) ? 1 : 0;
    if (!p.tma_store) tmC = tmA;  // unused
    if (g.mode == kDense) p.total_tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    else if (g.mode == kGroupedRows) p.total_tiles = ((g.T + kUnitRows - 1) / kUnitRows + g.E) * p.n_tiles;
    else p.total_tiles = static_cast<int64_t>(g.E) * p.m_tiles * p.n_tiles;
    if (p.total_tiles <= 0) return cudaSuccess;
    if (p.total_tiles >= (1ll << 31)) return cudaErrorInvalidValue;  // the tile decode divides 31-bit indices
    p.fd_m = make_fastdiv(static_cast<uint32_t>(p.m_tiles));
    p.fd_n = make_fastdiv(static_cast<uint32_t>(p.n_tiles));
    p.fd_mn = make_fastdiv(static_cast<uint32_t>(p.m_tiles) * static_cast<uint32_t>(p.n_tiles));
    p.c_expert_rows = g.mode == kGroupedK ? p.c_expert_stride / p.ldc : 0;

    // persistent grid: as many CTAs (CTA pairs) as can be resident at once, one
    // per SM (a CTA needs ~200 KB of shared memory).  Per device, once, under a
    // lock (host threads may launch concurrently): the kernel's shared-memory
    // attribute, which is a per-device setting, then the residency.
    static std::mutex init_mu;
    static int resident[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = st;
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    int units_max = 0;
    {
        std::lock_guard<std::mutex> lock(init_mu);
        if (resident[dev] == 0) {
            e = cudaFuncSetAttribute(k_gemm<CG, KIND, BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
            if (e != cudaSuccess) return e;
            int n = 0;
            if (CG == 2) {
                cfg.gridDim = dim3(2);
                e = cudaOccupancyMaxActiveClusters(&n, k_gemm<CG, KIND, BIAS>, &cfg);
            } else {
                e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            }
            if (e != cudaSuccess) return e;
            resident[dev] = n > 0 ? n : 1;
        }
        units_max = resident[dev];
    }
    const int64_t units = p.total_tiles < units_max ? p.total_tiles : units_max;
    cfg.gridDim = dim3(static_cast<unsigned>(units * CG));
    // programmatic dependent launch (see pdl_wait in the kernel)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs++;
    return cudaLaunchKernelEx(&cfg, k_gemm<CG, KIND, BIAS>, tmA, tmB, tmSA, tmSB, tmC, p);
}

}  // namespace

bool encode_tmap_2d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promo) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t device_error_word(unsigned int **out) {
    static unsigned int *addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

namespace {
// Failure-detection self-test: one thread waits on an mbarrier that nothing
// arrives on, with a bounded wait of `timeout_ns`; the wait gives up, sets
// the timeout bit of the device error word and the kernel returns normally.
__global__ void k_selftest_wait(uint64_t timeout_ns, int *gave_up) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const bool done = mbar_wait_for(b, 0, &abort_flag, &g_device_error, timeout_ns);
    *gave_up = done ? 0 : 1;
}
}  // namespace

namespace {
// Group-offset check on its own: one warp reads off[0..E] (nothing else) and
// sets kErrBadOffsets when they are malformed.
__global__ void k_check_offsets(const int64_t *off, int E, int64_t T) {
    if (!group_offsets_valid(off, E, T, threadIdx.x & 31) && threadIdx.x == 0) atomicOr(&g_device_error, kErrBadOffsets);
}
}  // namespace

cudaError_t launch_check_offsets(const int64_t *d_off, int E, int64_t T, cudaStream_t st) {
    k_check_offsets<<<1, 32, 0, st>>>(d_off, E, T);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(uint64_t timeout_ns, int *d_gave_up, cudaStream_t st) {
    k_selftest_wait<<<1, 32, 0, st>>>(timeout_ns, d_gave_up);
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(unsigned int *word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || *word == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
}

cudaError_t launch_gemm(const GemmProblem &g, cudaStream_t st) {
    Params p{};
    p.mode = g.mode;
    p.sa = g.sa; p.sb = g.sb;
    p.sa_kt = (g.a_k / 32 + 3) / 4;
    p.sb_kt = (g.b_k / 32 + 3) / 4;
    p.b_row_atoms = (g.b_rows + 127) / 128;
    p.c = static_cast<__nv_bfloat16 *>(g.c);
    p.M = g.M; p.N = g.N; p.ldc = g.ldc;
    p.K = g.kind == kBF16 ? 2 * g.K : g.K;  // the mainloop counts contraction bytes
    p.offsets = g.offsets; p.E = g.E; p.T = g.T;
    p.a_row_pad = g.mode == kGroupedRows ? g.a_row_pad : 0;
    p.b_row_per_expert = g.b_row_per_expert;
    p.b_k_per_expert = g.b_k_per_expert;
    p.c_expert_stride = g.c_expert_stride;
    p.bias = g.mode == kDense ? static_cast<const __nv_bfloat16 *>(g.bias) : nullptr;
    p.n_tiles = static_cast<int>((g.N + BN - 1) / BN);
    p.n_fastest = g.mode == kDense && g.a_rows > g.b_rows ? 1 : 0;
    p.sa_bytes = g.kind == kBF16 ? 0 : static_cast<uint64_t>(scale_bytes_of(p.a_row_pad ? p.a_row_pad : g.a_rows, g.a_k));
    p.sb_bytes = g.kind == kBF16 ? 0 : static_cast<uint64_t>(scale_bytes_of(g.b_rows, g.b_k));
    p.c_bytes = 2ull * static_cast<uint64_t>(g.mode == kGroupedK ? static_cast<int64_t>(g.E) * g.M : g.M) *
                static_cast<uint64_t>(g.ldc);
    // bias (dense only) is a separate instance: a per-chunk test in the
    // epilogue measurably slows the launches that have none
    if (g.kind == kBF16) {
        // dense, or the grouped forward (experts' B rows stacked; no contraction offsets)
        if (g.mode == kGroupedK || (g.mode == kGroupedRows && (g.b_k_per_expert != 0 || p.a_row_pad || p.bias)))
            return cudaErrorInvalidValue;
        return p.bias ? launch_cg<1, kBF16, true>(g, p, st) : launch_cg<1, kBF16, false>(g, p, st);
    }
    if (p.bias) return launch_cg<1, kMXF8, true>(g, p, st);
    if (cta_group_for(g) == 2) return launch_cg<2, kMXF8, false>(g, p, st);
    return launch_cg<1, kMXF8, false>(g, p, st);
}

}  // namespace mxq
