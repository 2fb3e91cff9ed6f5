// mxq_internal.h -- kernel launchers shared between the libmxq translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mxq.h"

namespace mxq {

// ---- quantization (mxq_quant.cu) ----
// cols % 32 == 0.  fmt 0: MXFP8 E4M3 codes (bf16 in); 1: packed MXFP4 nibbles; 2: MXFP4 values as E4M3
// codes (bf16 in).  fmt 1 takes bf16 or fp32 in.  sf: the MXFP4 scale factor.
cudaError_t launch_quant_rows(const void *x, bool fp32_in, int fmt, int64_t R, int64_t C, int64_t ldx,
                              uint8_t *q, uint8_t *s, cudaStream_t st, float sf = 6.0f);
// Column MXFP8 quant of bf16 x; q_row/s_row non-null adds the row quant (dual).
cudaError_t launch_quant_cols(const uint16_t *x, int64_t R, int64_t C, int64_t ldx, uint8_t *q_row,
                              uint8_t *s_row, uint8_t *qT, uint8_t *sT, cudaStream_t st);
// Per-group column MXFP8 quant of bf16 x [T x C]; q_row/s_row non-null adds the
// plain row quant of x from the same read (cols % 32 == 0), its scales in
// swz(T, C/32) or, with row_pad, in the per-group padded layout swz(t_pad, C/32).
cudaError_t launch_quant_cols_grouped(const uint16_t *x, int64_t T, int64_t C, const int64_t *d_off, int E,
                                      int64_t t_pad, uint8_t *q_row, uint8_t *s_row, uint8_t *qT, uint8_t *sT,
                                      cudaStream_t st, bool row_pad);
cudaError_t launch_qdq_mxfp4(const float *x, float *y, uint32_t *mask, int64_t rows, int64_t cols, float sf,
                             cudaStream_t st);
// MXFP4 quant-dequant bf16 -> bf16, blocks of 32 along rows; cols % 32 == 0, 16-byte aligned.
cudaError_t launch_qdq_mxfp4_bf16(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols, float sf,
                                  cudaStream_t st);
cudaError_t launch_ste_backward(const float *gy, const uint32_t *mask, float *gx, int64_t rows, int64_t cols,
                                cudaStream_t st);

// ---- GEMM (mxq_gemm.cu) ----
enum GemmMode { kDense = 0, kGroupedRows = 1, kGroupedK = 2 };
// Operand kind: kMXF8 = E4M3 codes with E8M0 block scales (all modes);
// kBF16 = plain bf16 operands, no scales (kDense, and kGroupedRows without
// contraction offsets: the grouped forward).
enum GemmKind { kMXF8 = 0, kBF16 = 1 };

struct GemmProblem {
    GemmMode mode;
    int kind;  // GemmKind; sizes below are in elements for both kinds
    // A: [a_rows x a_k] E4M3 codes, K-major; scales swz(a_rows, a_k/32)
    const uint8_t *a, *sa;
    int64_t a_rows, a_k;
    // B: [b_rows x b_k] E4M3 codes, K-major; scales swz(b_rows, b_k/32)
    const uint8_t *b, *sb;
    int64_t b_rows, b_k;
    // output bf16: M x N per problem (per expert in kGroupedK), leading dim ldc
    void *c;
    int64_t M, N, ldc;
    int64_t K;  // contraction length (kDense / kGroupedRows)
    // grouped
    const int64_t *offsets;   // device, E+1
    int E;
    int64_t b_row_per_expert; // kGroupedRows: B row offset of expert e = e * this
    int64_t b_k_per_expert;   // kGroupedRows: B contraction offset of expert e = e * this
    int64_t c_expert_stride;  // kGroupedK: elements between experts' outputs
    int64_t T;                // kGroupedRows: token rows (= off[E])
    int64_t a_row_pad;        // kGroupedRows: 0, or t_pad when A's scales are in the per-group
                              // padded layout swz(t_pad, a_k/32) (row r of group e at scale row
                              // P_e + r - off[e], P_e = sum over e' < e of ceil128(n_e'))
    const void *bias;         // kDense: optional bf16 [N] added in fp32 before rounding (16-byte aligned)
};
cudaError_t launch_gemm(const GemmProblem &p, cudaStream_t st);
// 2-D tiled tensor map over [outer x inner] elements with the given row
// stride in bytes (false if the driver entry point or the encode fails).
bool encode_tmap_2d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promo);
// Device address of the error word that bounded waits set (current device).
cudaError_t device_error_word(unsigned int **out);
// Self-test of the bounded waits: a kernel whose wait nothing completes gives
// up after timeout_ns, sets the error word and writes 1 to *d_gave_up.
cudaError_t launch_selftest_wait(uint64_t timeout_ns, int *d_gave_up, cudaStream_t st);
// Checks group offsets on the device (one warp reads d_off[0..E] only) and sets
// the bad-offsets bit of the device error word when they are malformed.
cudaError_t launch_check_offsets(const int64_t *d_off, int E, int64_t T, cudaStream_t st);
// Reads the device error word set by bounded waits that gave up, then clears it.
cudaError_t read_and_clear_device_error(unsigned int *word);

// ---- error reporting shared by the C entry points (mxq_api.cu) ----
mxq_status api_fail(mxq_status s, const char *msg);           // records msg, returns s
mxq_status api_check_arch();                                   // MXQ_ERR_ARCH unless sm_103
mxq_status api_cuda_result(cudaError_t e, const char *what);   // MXQ_OK or MXQ_ERR_CUDA

}  // namespace mxq
