// mxq_gemm.cu -- block-scaled MXFP8 GEMM on the 5th-generation tensor cores.
//
// C = deq(A) deq(B)^T with E4M3 operands and E8M0 scales per 32-element block
// along K ("低精度训练特性（MXFP8 / HiFloat8）": the forward, input-gradient and
// weight-gradient products of the linear layer and of the experts' grouped
// matmul run on MXFP8 operands, output in bf16).  One kernel serves the dense
// GEMM and both grouped forms:
//   kDense       tiles (m, n) of one problem;
//   kGroupedRows tiles (expert, 128-row tile overlapping the expert's token
//                rows, n); rows outside the expert are computed but not stored
//                (forward and input gradient of the MoE layer);
//   kGroupedK    tiles (expert, m, n) whose contraction runs over the expert's
//                padded token range only (weight gradient of the MoE layer).
//
// Persistent: one CTA per SM walks tiles blockIdx.x, +gridDim.x, ...
// CTA = 6 warps, tile 128 x 256, K step 128 bytes, 4-stage mbarrier pipeline:
//   warp 0     TMA producer: A/B code tiles (128B-swizzled) by
//              cp.async.bulk.tensor, 512-byte scale tiles by cp.async.bulk;
//   warp 1     allocates 512 TMEM columns; one lane copies the scale tiles to
//              TMEM (tcgen05.cp 32x128b.warpx4) and issues 4
//              tcgen05.mma.kind::mxf8f6f4.block_scale (M128 N256 K32) per stage,
//              then tcgen05.commit frees the stage;
//   warps 2-5  epilogue: tcgen05.ld of the fp32 accumulator (one TMEM lane
//              sub-partition each) into registers as bf16 (RNE), then release
//              the accumulator to the MMA warp before the 16-byte global
//              stores, which overlap the next tile's mainloop.
// TMEM: columns [0, 256) accumulator; [256 + 16 s, +12) scale slots of stage s
// (A: 4 columns, B: 2 x 4 columns).  Every wait is bounded (mxq_device.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <mutex>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {

// Device error word (bits in mxq_device.cuh), read and cleared by
// read_and_clear_device_error().
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4, THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK, B_BYTES = BN * BK, SFA_BYTES = 512, SFB_BYTES = 1024;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
constexpr uint32_t NUM_BARS = 2 * STAGES + 3;
constexpr uint32_t OFF_MISC = OFF_BAR + 128;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 256;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack to align the base to 1024
constexpr uint32_t TMEM_COLS = 512, SF_COL0 = 256, SF_STRIDE = 16;
static_assert(NUM_BARS * 8 <= 128, "barrier area");
static_assert(SF_COL0 + STAGES * SF_STRIDE <= TMEM_COLS, "tmem budget");

struct Params {
    GemmMode mode;
    const uint8_t *sa, *sb;
    int64_t sa_kt, sb_kt;              // 512-byte scale tiles per 128-row group
    int64_t b_row_atoms;               // ceil(b_rows / 128)
    __nv_bfloat16 *c;
    int64_t M, N, ldc, K;
    const int64_t *offsets;
    int E;
    int64_t b_row_per_expert, b_k_per_expert, c_expert_stride;
    int m_tiles, n_tiles;
    int n_fastest;        // kDense tile order: 1 = n fastest (A is the larger operand)
    int64_t total_tiles;  // tile index space (an upper bound for grouped rows)
};

struct TileInfo {
    int valid, nkb, k_last, b_atoms;
    int64_t a_row0, b_row0, a_k0, b_k0;   // TMA coordinates of k-block 0
    int64_t a_ratom, b_ratom, a_katom0, b_katom0;
    int64_t row_lo, row_hi, out_row0, col0, col_hi, c_off;
};

// Instruction descriptor, kind::mxf8f6f4: E4M3 x E4M3, both K-major, N = 256,
// M = 128, E8M0 scales, scale-factor byte `j` of the A and B scale columns.
__device__ __forceinline__ uint32_t make_idesc(uint32_t j) {
    return (j << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(BM >> 4) << 24) | (j << 29);
}

// Work decomposition: which tile this CTA computes (run by all lanes of warp 0).
__device__ TileInfo resolve_tile(const Params &p, int64_t bid, int lane) {
    TileInfo t{};
    t.k_last = 4;
    if (p.mode == kDense) {
        // raster so that the smaller operand stays in L2 while the larger one
        // streams through once: concurrent CTAs share the larger operand's tile
        const int64_t mt = p.n_fastest ? bid / p.n_tiles : bid % p.m_tiles;
        const int64_t nt = p.n_fastest ? bid % p.n_tiles : bid / p.m_tiles;
        t.valid = 1;
        t.a_row0 = mt * BM; t.b_row0 = nt * BN;
        t.a_ratom = mt; t.b_ratom = 2 * nt;
        t.row_lo = t.a_row0; t.row_hi = min(p.M, t.a_row0 + BM); t.out_row0 = t.a_row0;
        t.col0 = nt * BN; t.col_hi = min(p.N, t.col0 + BN);
    } else if (p.mode == kGroupedRows) {
        // tiles of expert e: every 128-row tile overlapping [o_e, o_e+1), times n_tiles
        int64_t run = 0;
        int fe = -1;
        int64_t fstart = 0, fo0 = 0, fo1 = 0;
        for (int base = 0; base < p.E; base += 32) {
            const int e = base + lane;
            int64_t o0 = 0, o1 = 0;
            if (e < p.E) { o0 = p.offsets[e]; o1 = p.offsets[e + 1]; }
            const int64_t cnt = (o1 > o0) ? ((o1 - 1) / BM - o0 / BM + 1) * p.n_tiles : 0;
            int64_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const int64_t start = run + incl - cnt;
            const bool mine = cnt > 0 && bid >= start && bid < start + cnt;
            const unsigned bal = __ballot_sync(0xffffffffu, mine);
            if (bal) {
                const int src = __ffs(bal) - 1;
                fe = base + src;
                fstart = __shfl_sync(0xffffffffu, start, src);
                fo0 = __shfl_sync(0xffffffffu, o0, src);
                fo1 = __shfl_sync(0xffffffffu, o1, src);
                break;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (fe < 0) { t.valid = 0; return t; }
        const int64_t mtiles_e = (fo1 - 1) / BM - fo0 / BM + 1;
        const int64_t local = bid - fstart;
        const int64_t nt = local / mtiles_e, mt = fo0 / BM + local % mtiles_e;
        t.valid = 1;
        t.a_row0 = mt * BM; t.a_ratom = mt;
        t.b_row0 = fe * p.b_row_per_expert + nt * BN; t.b_ratom = t.b_row0 / BM;
        t.b_k0 = fe * p.b_k_per_expert; t.b_katom0 = t.b_k0 / BK;
        t.row_lo = max(fo0, t.a_row0); t.row_hi = min(fo1, t.a_row0 + BM); t.out_row0 = t.a_row0;
        t.col0 = nt * BN; t.col_hi = min(p.N, t.col0 + BN);
    } else {  // kGroupedK
        const int64_t per = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
        const int e = static_cast<int>(bid / per);
        const int64_t local = bid % per, mt = local % p.m_tiles, nt = local / p.m_tiles;
        int64_t pe = 0;  // padded start of group e = sum_{j<e} ceil128(n_j)
        for (int base = 0; base < e; base += 32) {
            const int j = base + lane;
            if (j < e) pe += (p.offsets[j + 1] - p.offsets[j] + 127) / 128 * 128;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) pe += __shfl_xor_sync(0xffffffffu, pe, o);
        const int64_t ne = p.offsets[e + 1] - p.offsets[e];
        t.valid = 1;
        t.a_row0 = mt * BM; t.b_row0 = nt * BN; t.a_ratom = mt; t.b_ratom = 2 * nt;
        t.a_k0 = t.b_k0 = pe; t.a_katom0 = t.b_katom0 = pe / BK;
        t.nkb = static_cast<int>((ne + 127) / 128);
        t.row_lo = t.a_row0; t.row_hi = min(p.M, t.a_row0 + BM); t.out_row0 = t.a_row0;
        t.col0 = nt * BN; t.col_hi = min(p.N, t.col0 + BN);
        t.c_off = static_cast<int64_t>(e) * p.c_expert_stride;
    }
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

__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_mxf8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar_full = sbase + OFF_BAR, bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_accf = bar_full + 16 * STAGES, bar_acce = bar_accf + 8, bar_drain = bar_accf + 16;

    // once any CTA has given up, the rest of the grid does no work
    if (threadIdx.x == 0) *abort_flag = *reinterpret_cast<volatile unsigned int *>(&g_device_error) != 0 ? 1 : 0;
    __syncthreads();
    if (*abort_flag) return;  // before any TMEM allocation

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        if (lane == 0) {
            for (int s = 0; s < STAGES; s++) {
                mbar_init(bar_full + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, 1);
            }
            mbar_init(bar_accf, 1);
            mbar_init(bar_acce, 4);  // one arrival per epilogue warp
            mbar_init(bar_drain, 1);
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Persistent loop: every warp walks the same tile sequence and decodes each
    // tile itself; the stage ring and the accumulator phases run across tiles.
    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        uint32_t g = 0;  // k-blocks issued by this CTA (lane 0)
        for (int64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
            const TileInfo ti = resolve_tile(p, tile, lane);
            if (!ti.valid) break;  // grouped-row tiles past the real count come last
            int stop = 0;
            if (lane == 0) {
                for (int kb = 0; kb < ti.nkb; kb++, g++) {
                    const uint32_t s = g % STAGES, ph = (g / STAGES) & 1;
                    if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, &g_device_error)) { stop = 1; break; }
                    const uint32_t fb = bar_full + 8 * s;
                    mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + SFA_BYTES + 512u * ti.b_atoms);
                    tma_load_2d(sbase + OFF_A + s * A_BYTES, &tmA, fb, static_cast<int>(ti.a_k0 + kb * BK),
                                static_cast<int>(ti.a_row0));
                    tma_load_2d(sbase + OFF_B + s * B_BYTES, &tmB, fb, static_cast<int>(ti.b_k0 + kb * BK),
                                static_cast<int>(ti.b_row0));
                    bulk_load(sbase + OFF_SFA + s * SFA_BYTES,
                              p.sa + (ti.a_ratom * p.sa_kt + ti.a_katom0 + kb) * 512, 512, fb);
                    for (int h = 0; h < ti.b_atoms; h++)
                        bulk_load(sbase + OFF_SFB + s * SFB_BYTES + 512 * h,
                                  p.sb + ((ti.b_ratom + h) * p.sb_kt + ti.b_katom0 + kb) * 512, 512, fb);
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        if (lane == 0 && *abort_flag) {  // let this CTA's copies land before it exits
            for (uint32_t j = g > STAGES ? g - STAGES : 0; j < g; j++)
                mbar_wait_drain(bar_full + 8 * (j % STAGES), (j / STAGES) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        uint32_t g = 0, acc_it = 0;
        bool issued_any = false;
        for (int64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
            const TileInfo ti = resolve_tile(p, tile, lane);
            if (!ti.valid) break;
            if (ti.nkb == 0) continue;  // empty group: the epilogue writes zeros
            int stop = 0;
            if (lane == 0) {
                // the epilogue must have drained the previous accumulator
                if (acc_it > 0 && !mbar_wait(bar_acce, (acc_it - 1) & 1, abort_flag, &g_device_error)) stop = 1;
                tc_fence_after();
                for (int kb = 0; kb < ti.nkb && !stop; kb++, g++) {
                    const uint32_t s = g % STAGES, ph = (g / STAGES) & 1;
                    if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_device_error)) { stop = 1; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + SF_COL0 + s * SF_STRIDE, sfb_t = sfa_t + 4;
                    tc_cp_32x128b_warpx4(sfa_t, smem_desc(sbase + OFF_SFA + s * SFA_BYTES, 0, 128, 0));
                    tc_cp_32x128b_warpx4(sfb_t, smem_desc(sbase + OFF_SFB + s * SFB_BYTES, 0, 128, 0));
                    tc_cp_32x128b_warpx4(sfb_t + 4, smem_desc(sbase + OFF_SFB + s * SFB_BYTES + 512, 0, 128, 0));
                    const int kk = (kb == ti.nkb - 1) ? ti.k_last : 4;
                    for (int j = 0; j < kk; j++) {
                        const uint64_t ad = smem_desc(sbase + OFF_A + s * A_BYTES + 32 * j, 0, 1024, 2);
                        const uint64_t bd = smem_desc(sbase + OFF_B + s * B_BYTES + 32 * j, 0, 1024, 2);
                        tc_mma_mxf8(tmem, ad, bd, make_idesc(static_cast<uint32_t>(j)), sfa_t, sfb_t,
                                    (kb | j) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    tc_commit(bar_empty + 8 * s);
                }
                if (!stop) tc_commit(bar_accf);
            }
            acc_it++;
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        if (lane == 0 && issued_any && *abort_flag) {  // no MMA in flight at dealloc
            tc_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0);
        }
    } else {
        // ---------------------------------------------------- epilogue
        // Drain the accumulator into registers (bf16), release it to the MMA
        // warp, then store: the global stores overlap the next tile's mainloop.
        const int sub = warp & 3;
        uint32_t acc_it = 0;
        for (int64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
            const TileInfo ti = resolve_tile(p, tile, lane);
            if (!ti.valid) break;
            const int64_t grow = ti.out_row0 + 32 * sub + lane;
            const bool row_ok = grow >= ti.row_lo && grow < ti.row_hi;
            __nv_bfloat16 *crow = p.c + ti.c_off + grow * p.ldc;
            if (ti.nkb == 0) {
                if (row_ok)
                    for (int64_t col = ti.col0; col < ti.col_hi; col++) crow[col] = __float2bfloat16_rn(0.0f);
                continue;
            }
            if (!mbar_wait(bar_accf, acc_it & 1, abort_flag, &g_device_error)) break;
            tc_fence_after();
            uint32_t pk[BN / 2];
#pragma unroll
            for (int ch = 0; ch < BN / 32; ch++) {
                if (ti.col0 + 32 * ch < ti.col_hi) {  // warp-uniform
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * sub) << 16) + 32 * ch, r);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        pk[16 * ch + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce);
            acc_it++;
            if (!row_ok) continue;
#pragma unroll
            for (int ch = 0; ch < BN / 32; ch++) {
                const int64_t col = ti.col0 + 32 * ch;
                if (col + 32 <= ti.col_hi) {
                    uint4 *dst = reinterpret_cast<uint4 *>(crow + col);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        dst[i] = make_uint4(pk[16 * ch + 4 * i], pk[16 * ch + 4 * i + 1], pk[16 * ch + 4 * i + 2],
                                            pk[16 * ch + 4 * i + 3]);
                } else if (col < ti.col_hi) {
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        if (col + i < ti.col_hi)
                            reinterpret_cast<uint16_t *>(crow)[col + i] =
                                static_cast<uint16_t>(pk[16 * ch + (i >> 1)] >> (16 * (i & 1)));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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

}  // namespace

cudaError_t read_and_clear_device_error(unsigned int *word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || *word == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
}

cudaError_t launch_gemm(const GemmProblem &g, cudaStream_t st) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(k_gemm_mxf8, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap tmA, tmB;
    if (!make_tmap(&tmA, g.a, g.a_rows, g.a_k, BM) || !make_tmap(&tmB, g.b, g.b_rows, g.b_k, BN))
        return cudaErrorInvalidValue;

    Params p{};
    p.mode = g.mode;
    p.sa = g.sa; p.sb = g.sb;
    p.sa_kt = (g.a_k / 32 + 3) / 4;
    p.sb_kt = (g.b_k / 32 + 3) / 4;
    p.b_row_atoms = (g.b_rows + 127) / 128;
    p.c = static_cast<__nv_bfloat16 *>(g.c);
    p.M = g.M; p.N = g.N; p.ldc = g.ldc; p.K = g.K;
    p.offsets = g.offsets; p.E = g.E;
    p.b_row_per_expert = g.b_row_per_expert;
    p.b_k_per_expert = g.b_k_per_expert;
    p.c_expert_stride = g.c_expert_stride;
    p.m_tiles = static_cast<int>((g.M + BM - 1) / BM);
    p.n_tiles = static_cast<int>((g.N + BN - 1) / BN);
    p.n_fastest = g.mode == kDense && g.a_rows > g.b_rows ? 1 : 0;
    if (g.mode == kDense) p.total_tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    else if (g.mode == kGroupedRows) p.total_tiles = ((g.T + BM - 1) / BM + g.E) * p.n_tiles;
    else p.total_tiles = static_cast<int64_t>(g.E) * p.m_tiles * p.n_tiles;
    if (p.total_tiles <= 0) return cudaSuccess;
    // persistent grid: one CTA per SM (the CTA needs ~200 KB of shared memory)
    static int num_sms[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (num_sms[dev] == 0) {
        e = cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int64_t grid = p.total_tiles < num_sms[dev] ? p.total_tiles : num_sms[dev];
    k_gemm_mxf8<<<static_cast<unsigned>(grid), THREADS, SMEM_ALLOC, st>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace mxq
