/*
 * mxq.h -- C ABI of libmxq: MX block-scaled quantization and block-scaled
 * MXFP8 GEMMs for GB300 (sm_103a).
 *
 * What the operations are (web pages, cited by title and section):
 *  [TT]  "低精度训练特性（MXFP8 / HiFloat8）" (torchtitan-npu feature guide):
 *        section "线性层低精度" MXFP8 mode -- per-block quantization of
 *        activations and weights, block size 32, every 32 elements share one
 *        scale, then a low-precision matmul for the forward, input-gradient and
 *        weight-gradient products, output back in the original precision;
 *        section "MoE 专家层低精度" MXFP8 mode -- the same for the experts'
 *        grouped matmul, with the weight gradient's operands quantized per
 *        group ("grouped dynamic MX quant").
 *  [FB]  "Ascend/MindSpeed pull 3852" (the fb-split PR), change summary:
 *        forward quantizes along one axis only and saves nothing; backward
 *        recomputes the other axis (vs. dual-axis quant whose extra outputs are
 *        saved for backward).
 *  [AMCT] "AMCT FakeQuant 模拟伪量化工具包" article: section 2 (MXFP4 numeric
 *        model), section 3.2-3.3 (the kernel's raw call and its Python
 *        wrapper's padding convention), section 4.2 (config validation).
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers to memory the caller owns and
 *    keeps alive until the work on `stream` has finished.  The library never
 *    allocates device memory; size queries tell the caller how much to give.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument checks run first, on the host, and return an
 *    error before anything is launched; nothing is written on error.
 *  - Pointers must be 16-byte aligned.  Row-major everywhere; `ld*` are
 *    leading dimensions in elements.
 *  - Codes are bytes: E4M3 (OCP FP8, max 448) or, for E2M1, two 4-bit codes
 *    per byte (even element in the low nibble; nibble = sign<<3 | index into
 *    {0, .5, 1, 1.5, 2, 3, 4, 6}).  Scales are E8M0 bytes (2^(byte-127)).
 *  - Scale layout "swz(R, KB)": the logical R x KB scale matrix (KB = number
 *    of 32-element blocks along the contraction axis) with R padded to 128 and
 *    KB to 4, stored as 512-byte tiles of 128 rows x 4 blocks, tile (i, j) at
 *    byte 512*(i*ceil(KB/4) + j), element (r, c) of a tile at
 *    16*(r%32) + 4*(r/32) + c.  This is the layout the tcgen05 block-scaled
 *    MMA reads; the quantizers write padding bytes as 0.
 *  - "K-major": every GEMM operand is [rows x K] with the scale blocks along K;
 *    a column quant writes its codes transposed ([C x R]) so that it too is
 *    K-major.
 *  - Errors: the return value; mxq_last_error_string() gives the reason
 *    (thread-local).  No exception crosses the ABI.  MXQ_ERR_ARCH when the
 *    current device is not compute capability 10.3.
 *  - Host threads: entry points may be called from several host threads at
 *    once, each on its own stream (mxq_linear_fwd_noalloc's shared scratch is
 *    the exception; see there).  The first launch of each kernel on a device
 *    does a one-time setup under a lock: its shared-memory attribute and its
 *    resident-CTA count.  That setup, like every per-device value the library
 *    keeps, belongs to the device's primary context.  After a
 *    cudaDeviceReset, do not call the library on that device again in the
 *    same process.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *mxq_stream_t; /* same type as cudaStream_t */

typedef enum {
    MXQ_OK = 0,
    MXQ_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or enum */
    MXQ_ERR_UNSUPPORTED = 2, /* valid request this library does not implement */
    MXQ_ERR_ARCH = 3,        /* current device is not sm_103 */
    MXQ_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    MXQ_ERR_TIMEOUT = 5      /* a kernel gave up waiting (see mxq_poll_device_error) */
} mxq_status;

typedef enum { MXQ_BF16 = 0, MXQ_F32 = 1 } mxq_dtype;
typedef enum { MXQ_E4M3 = 0, MXQ_E2M1 = 1 } mxq_fmt;
typedef enum { MXQ_SAVE_QUANT = 0, MXQ_RECOMPUTE = 1 } mxq_mode;
typedef enum { MXQ_GG_FWD = 0, MXQ_GG_DX = 1, MXQ_GG_DW = 2 } mxq_gg_kind;

/* ------------------------------------------------------------------ */
/* Size queries (host only, no CUDA calls)                              */
/* ------------------------------------------------------------------ */

/* Bytes of swz(rows, k_blocks): ceil128(rows) * ceil4(k_blocks). */
size_t mxq_scale_bytes(int64_t rows, int64_t k_blocks);

/* Capacity of the padded token axis of a per-group column quant of T rows in
 * E groups: 128 * (ceil(T/128) + E), an upper bound on
 * sum_e ceil128(n_e) for any split of T rows into E groups. */
int64_t mxq_grouped_padded_rows(int64_t T, int E);

/* ------------------------------------------------------------------ */
/* Quantization                                                         */
/* ------------------------------------------------------------------ */

/* Dynamic MX quantization of x[rows x cols] (leading dim ldx).
 * [TT] MXFP8 mode (blocks of 32 sharing one scale; axis -1 or -2 of the
 * dynamic MX quant op) and [FB] (the dual-axis variant returns both axes from
 * one call).
 *  fmt = MXQ_E4M3 (MXFP8): dtype must be MXQ_BF16.  Scale exponent
 *      X = floor(log2 amax) - 8 clamped to [-127,127] (X = -127 for an
 *      all-zero block); code = E4M3(x * 2^-X), round-to-nearest-even,
 *      saturating to +-448.
 *    axis = -1 (or dual_axis): blocks along cols; needs cols % 32 == 0.
 *      q_row [rows x cols] u8, s_row swz(rows, cols/32).
 *    axis = -2 (or dual_axis): blocks along rows (a ragged last block is
 *      zero-padded); q_colT [cols x rows] u8 (transposed, leading dim rows),
 *      s_colT swz(cols, ceil(rows/32)).  Needs cols % 8 == 0.
 *    dual_axis != 0: both outputs from one read of x ([FB]).
 *  fmt = MXQ_E2M1 (MXFP4, [AMCT] section 2 with scale_factor 6): dtype BF16
 *      or F32, axis -1 only, dual_axis 0, cols % 32 == 0.  q_row holds
 *      rows x cols/2 bytes, s_row swz(rows, cols/32), scale byte e + 127 with
 *      e = round(log2(max(amax/6, 2^-30))).
 * Pointers not needed by the chosen axis may be NULL.  ldx % 8 == 0.
 * rows == 0 or cols == 0 is a no-op. */
mxq_status mxq_quantize(const void *x, mxq_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                        int axis, mxq_fmt fmt, int dual_axis,
                        void *q_row, void *s_row, void *q_colT, void *s_colT,
                        mxq_stream_t stream);

/* Per-group column MXFP8 quant for the grouped weight gradient ([TT] MoE
 * MXFP8 mode, "grouped dynamic MX quant"): x bf16 [rows x cols] (leading
 * dim cols), group e = rows [off[e], off[e+1]) with d_offsets a DEVICE array
 * of E+1 int64 (non-decreasing, off[0] = 0, off[E] = rows; checked on the
 * device as described below).  Blocks of 32 rows restart at every group
 * start and a group's last block is zero-padded.  Group e is written at padded column P_e =
 * sum_{j<e} ceil128(n_j) of q_colT [cols x t_pad] (leading dim t_pad) and its
 * scales into s_colT swz(cols, t_pad/32).  Every byte of both outputs is
 * written (padding = 0).  t_pad % 128 == 0 and
 * t_pad >= mxq_grouped_padded_rows(rows, E) guarantees room; cols % 8 == 0;
 * 1 <= E <= 4096. */
mxq_status mxq_quantize_grouped_col(const void *x_bf16, int64_t rows, int64_t cols,
                                    const int64_t *d_offsets, int E, int64_t t_pad,
                                    void *q_colT, void *s_colT, mxq_stream_t stream);

/* Group offsets, as every grouped entry point takes them: E+1 int64 values
 * with off[0] = 0, off[e] <= off[e+1] and off[E] = T (the number of token
 * rows); group e is rows [off[e], off[e+1]) and may be empty.  ([TT] MoE
 * MXFP8 mode: the token counts per expert that the grouped matmul splits its
 * rows by.)
 * Every grouped kernel checks its DEVICE offsets before it reads or writes
 * anything that depends on them.  Malformed offsets make the kernel skip all
 * of its work (its outputs are left unwritten) and set bit 2 of the device
 * error word, which mxq_poll_device_error reports as MXQ_ERR_INVALID_ARG;
 * no access outside the caller's buffers happens.
 * mxq_validate_group_offsets applies the same rule to a HOST copy and returns
 * MXQ_ERR_INVALID_ARG with the first violation in mxq_last_error_string()
 * (no CUDA call).  mxq_check_group_offsets launches, on `stream`, one warp
 * that reads d_offsets[0..E] and nothing else and sets the same bit when they
 * are malformed. */
mxq_status mxq_validate_group_offsets(const int64_t *offsets, int E, int64_t T);
mxq_status mxq_check_group_offsets(const int64_t *d_offsets, int E, int64_t T, mxq_stream_t stream);

/* Grouped dual-axis MXFP8 quant: the per-group column quant above and the
 * plain row quant of the same x from one read of x, as the MoE layer needs
 * them ([TT] MoE MXFP8 mode: the forward and input-gradient matmuls take the
 * row quant of X and dY along the feature dim, the weight-gradient matmul
 * their per-group column quant; [FB] for producing both axes in one pass).
 *  q_row [rows x cols] u8 and s_row swz(rows, cols/32) are exactly what
 *  mxq_quantize(x, MXQ_BF16, rows, cols, cols, -1, MXQ_E4M3, 0, ...) writes,
 *  padding bytes included; q_colT/s_colT exactly what
 *  mxq_quantize_grouped_col writes.  x is dense (leading dim cols).
 *  q_row and s_row are both given (cols % 32 == 0) or both NULL (then this is
 *  mxq_quantize_grouped_col).  Other arguments and errors as for
 *  mxq_quantize_grouped_col. */
mxq_status mxq_quantize_grouped_dual(const void *x_bf16, int64_t rows, int64_t cols,
                                     const int64_t *d_offsets, int E, int64_t t_pad,
                                     void *q_row, void *s_row, void *q_colT, void *s_colT,
                                     mxq_stream_t stream);

/* The same quant with the row scales in the per-group padded layout:
 * s_row is swz(t_pad, cols/32) (DEVICE, written in full), and the row scales
 * of row r of group e sit at scale row P_e + (r - off[e]), where
 * P_e = sum over e' < e of ceil128(off[e'+1] - off[e']) is the group's padded
 * start, the same as in the column quant; every other scale row is zero.
 * q_row is the plain [rows x cols] row quant as above, and q_colT/s_colT as
 * above.  Each group's scale rows start a 512-byte scale tile, so the grouped
 * forward / dX GEMM given this layout (t_pad > 0) tiles each group from its
 * first row and computes no row twice.  q_row and s_row are required;
 * other arguments and errors as for mxq_quantize_grouped_dual. */
mxq_status mxq_quantize_grouped_dual_padded(const void *x_bf16, int64_t rows, int64_t cols,
                                            const int64_t *d_offsets, int E, int64_t t_pad,
                                            void *q_row, void *s_row, void *q_colT, void *s_colT,
                                            mxq_stream_t stream);

/* MXFP4 quant-dequant ([AMCT] sections 2, 3.2-3.3): fp32 x viewed as
 * [rows x cols] with cols the tensor's last dim; blocks of 32 along each row,
 * the last block of a row zero-padded (never spanning two rows);
 * scale = 2^round(log2(max(amax/scale_factor, 2^-30))) (evaluated exactly),
 * elements snapped to {0, +-.5, +-1, +-1.5, +-2, +-3, +-4, +-6} * scale with
 * midpoints rounding away from zero.  y has x's shape; y may equal x.
 * block_size must be 32 (else MXQ_ERR_UNSUPPORTED, as the Ascend kernel and
 * its wrapper require); scale_factor must be finite and > 0 ([AMCT] 4.2) --
 * scale_factor = 6 / inv_scale_factor_scale ([AMCT] 3.3). */
mxq_status mxq_qdq_mxfp4(const float *x, float *y, int64_t rows, int64_t cols,
                         int block_size, float scale_factor, mxq_stream_t stream);

/* MXFP4 quant-dequant of a bf16 tensor to bf16 ([AMCT] section 3.4: the
 * result has the input's dtype): the same rule as mxq_qdq_mxfp4 on the
 * exactly widened values; every result is exact in bf16 (a non-finite block
 * gives NaN).  x, y bf16 [rows x cols], DEVICE, 16-byte aligned, y may equal
 * x; cols % 32 == 0 (else MXQ_ERR_UNSUPPORTED). */
mxq_status mxq_qdq_mxfp4_bf16(const void *x_bf16, void *y_bf16, int64_t rows, int64_t cols,
                              int block_size, float scale_factor, mxq_stream_t stream);

/* Forward of the clipped straight-through estimator ([AMCT] section 4.1,
 * "STE and clipped STE"): y = MXFP4 quant-dequant of x exactly as
 * mxq_qdq_mxfp4, and the saturation mask the backward needs.  An element is
 * saturated when |x| > 6 * (its block's scale), i.e. when the codebook's top
 * value clipped it.  sat_mask (DEVICE, uint32 [rows x ceil(cols/32)], written
 * in full) holds one word per block: bit i of word (r, b) is element
 * (r, 32b + i); bits past the end of a ragged row are 0; a block with a
 * non-finite element has no saturated elements.  Arguments and errors as for
 * mxq_qdq_mxfp4; sat_mask must be non-null and 4-byte aligned. */
mxq_status mxq_mxfp4_ste_forward(const float *x, float *y, uint32_t *sat_mask, int64_t rows,
                                 int64_t cols, int block_size, float scale_factor,
                                 mxq_stream_t stream);

/* Backward of the clipped straight-through estimator ([AMCT] section 4.1):
 * grad_x = grad_y with every element whose sat_mask bit is set replaced by
 * +0.0 and every other element copied bit for bit.  grad_y, grad_x fp32
 * [rows x cols] (DEVICE, 4-byte aligned; grad_x may equal grad_y); sat_mask
 * as written by mxq_mxfp4_ste_forward for the same shape.  The plain STE is
 * the identity and needs no call. */
mxq_status mxq_mxfp4_ste_backward(const float *grad_y, const uint32_t *sat_mask, int64_t rows,
                                  int64_t cols, float *grad_x, mxq_stream_t stream);

/* ------------------------------------------------------------------ */
/* MXFP4 quantization-aware training: linear-layer forward                */
/* ------------------------------------------------------------------ */

/* Workspace of mxq_qat_linear_fwd: W4A4 (quantize_input != 0) holds both
 * quantized operands (codes + scales, each rounded up to 256 bytes); W4A16
 * holds Q(w) in bf16. */
size_t mxq_qat_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int quantize_input);

/* Forward of the MXFP4 QAT linear layer ([AMCT] section 4.3):
 * y = F.linear(Q(x), Q(w), bias) with Q the MXFP4 quant-dequant along K
 * (blocks of 32, scale_factor as in mxq_qdq_mxfp4) and the bias not
 * quantized.  x bf16 [M x K], w bf16 [N x K] (the layer's high-precision
 * master weight, left unchanged), bias bf16 [N] or NULL, y bf16 [M x N]; all
 * DEVICE, 16-byte aligned.  Q(x) and Q(w) are held exactly as E4M3 codes
 * under the MXFP4 E8M0 scales, and the product is accumulated in fp32 on the
 * block-scaled tensor cores; the bias is added in fp32 before the one
 * rounding to bf16.  quantize_input = 0 (W4A16) leaves x unquantized: Q(w)
 * is formed in bf16 (exact) and the product runs on the bf16 tensor cores.
 * M, N, K positive multiples of 32; workspace >=
 * mxq_qat_linear_workspace_bytes(M, N, K, quantize_input). */
mxq_status mxq_qat_linear_fwd(const void *x_bf16, const void *w_bf16, const void *bias_bf16,
                              int64_t M, int64_t N, int64_t K, int quantize_input,
                              float scale_factor, void *y_bf16, void *workspace,
                              size_t ws_bytes, mxq_stream_t stream);

/* The MXFP4 QAT forward of an MoE expert layer ([AMCT] section 4.3 applies
 * the fake-quant linear to each expert's matmul): for each group e of the
 * routed rows (d_offsets as for mxq_grouped_gemm),
 *   y[off[e]:off[e+1]] = Q(x[off[e]:off[e+1]]) Q(W_e)^T    (quantize_input = 1, W4A4)
 *   y[off[e]:off[e+1]] = x[off[e]:off[e+1]] Q(W_e)^T       (quantize_input = 0, W4A16)
 * with Q the MXFP4 quant-dequant of mxq_qdq_mxfp4 along K.  x bf16 [T x K],
 * w bf16 [E x N x K] (expert e's weight is rows [e*N, (e+1)*N) of the
 * stacked [E*N x K]), y bf16 [T x N], all DEVICE and 16-byte aligned.
 * W4A4 holds both operands' MXFP4 values exactly as E4M3 codes under their
 * E8M0 scales and runs the block-scaled grouped GEMM; W4A16 forms Q(W) in
 * bf16 (exact) and runs the grouped GEMM on the bf16 tensor cores.  An empty
 * group has no rows to write; T = 0 is a no-op.  N % 128 == 0, K % 32 == 0;
 * workspace >= mxq_qat_grouped_fwd_workspace_bytes(T, E, N, K,
 * quantize_input), 16-byte aligned.  Malformed offsets as for the grouped
 * GEMM. */
size_t mxq_qat_grouped_fwd_workspace_bytes(int64_t T, int E, int64_t N, int64_t K, int quantize_input);
mxq_status mxq_qat_grouped_fwd(const void *x_bf16, const void *w_bf16, const int64_t *d_offsets, int E,
                               int64_t T, int64_t N, int64_t K, int quantize_input, float scale_factor,
                               void *y_bf16, void *workspace, size_t ws_bytes, mxq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Block-scaled MXFP8 GEMMs ([TT] MXFP8 mode; output in bf16, fp32 accumulate) */
/* ------------------------------------------------------------------ */

/* C[M x N] (bf16, leading dim ldc) = deq(A) deq(B)^T with A [M x K] E4M3
 * codes + swz(M, K/32) scales and B [N x K] E4M3 codes + swz(N, K/32).
 * K % 32 == 0, K > 0, ldc >= N, ldc % 8 == 0.  M or N == 0 is a no-op. */
mxq_status mxq_gemm(const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb,
                    int64_t M, int64_t N, int64_t K, void *c_bf16, int64_t ldc,
                    mxq_stream_t stream);

/* Grouped (MoE) block-scaled GEMM over E experts ([TT] MoE MXFP8 mode),
 * group offsets d_offsets (DEVICE, E+1 int64, as for
 * mxq_quantize_grouped_col), T = off[E] token rows.
 *  MXQ_GG_FWD: out[T x N] rows of group e = deq(A_e) deq(B_e)^T, A [T x K]
 *      row-quantized (swz(T, K/32)), B [E*N x K] row-quantized as one matrix
 *      (swz(E*N, K/32)); expert e's weight is rows [e*N, (e+1)*N).
 *      N % 128 == 0.
 *  MXQ_GG_DX: out[T x K] rows of group e = deq(A_e) deq(B_e)^T, A = dY
 *      [T x N] row-quantized (swz(T, N/32)), B = the column quant of the
 *      stacked weights [E*N x K] ([FB] op_dx: the weight re-quantized along the
 *      other axis): codes [K x E*N], swz(K, E*N/32); expert e contracts over
 *      columns [e*N, (e+1)*N).  N % 128 == 0.  (K here is the output width.)
 *  MXQ_GG_DW: out[E x N x K]: out_e = deq(A_e) deq(B_e)^T contracted over the
 *      rows of group e only, A = per-group column quant of dY (codes
 *      [N x t_pad], swz(N, t_pad/32)), B = per-group column quant of X (codes
 *      [K x t_pad], swz(K, t_pad/32)); a group with no rows gives zeros.
 * K % 32 == 0 (FWD/DX), ldc is the output's row length (N for FWD/DW, K for
 * DX).
 * t_pad: for MXQ_GG_DW the padded length of the column quants (a multiple of
 * 128, >= mxq_grouped_padded_rows(T, E)).  For MXQ_GG_FWD / MXQ_GG_DX, 0
 * means A's scales are swz(T, .) as written by mxq_quantize or
 * mxq_quantize_grouped_dual: the row tiles are the matrix's 128-row tiles,
 * and one that straddles a group boundary is computed once per group it
 * touches; t_pad > 0 (same rule as for DW) means A's scales are in the
 * per-group padded layout of mxq_quantize_grouped_dual_padded (swz(t_pad, .)):
 * each group is tiled from its own first row.  Both give the same output bit
 * for bit. */
mxq_status mxq_grouped_gemm(mxq_gg_kind kind, const uint8_t *a, const uint8_t *sa,
                            const uint8_t *b, const uint8_t *sb, const int64_t *d_offsets, int E,
                            int64_t T, int64_t N, int64_t K, int64_t t_pad, void *out_bf16,
                            mxq_stream_t stream);

/* ------------------------------------------------------------------ */
/* MXFP8 linear layer: Y = X W^T, dX = dY W, dW = dY^T X                */
/* ------------------------------------------------------------------ */
/* [TT] MXFP8 mode; [FB] for the two modes:
 *  MXQ_SAVE_QUANT: forward dual-quantizes X and W and keeps their column
 *      quants in ctx for the backward.
 *  MXQ_RECOMPUTE: forward row-quantizes only and keeps nothing; backward
 *      re-quantizes X and W along the other axis from the bf16 originals.
 * Both modes give bitwise-identical Y, dX and dW.
 * x bf16 [M x K], w bf16 [N x K], dy bf16 [M x N]; y bf16 [M x N],
 * dx bf16 [M x K], dw bf16 [N x K].  M, N, K multiples of 32, K,N > 0.
 * ctx (mxq_linear_ctx_bytes) carries state from fwd to bwd_dx to bwd_dw of
 * the same step and must not be reused by another step in between; bwd_dx
 * stores dY's column quant there for bwd_dw.  workspace
 * (mxq_linear_workspace_bytes) is scratch for one call. */
size_t mxq_linear_ctx_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode);
/* Bytes of ctx that live from the forward to the backward (the memory the
 * recompute mode saves): (M*K + N*K) codes + their scales for SAVE, 0 for
 * RECOMPUTE. */
size_t mxq_linear_saved_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode);
size_t mxq_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode);

mxq_status mxq_linear_fwd(const void *x, const void *w, int64_t M, int64_t N, int64_t K,
                          mxq_mode mode, void *ctx, void *y, void *workspace, size_t ws_bytes,
                          mxq_stream_t stream);
mxq_status mxq_linear_bwd_dx(const void *dy, const void *w, int64_t M, int64_t N, int64_t K,
                             mxq_mode mode, void *ctx, void *dx, void *workspace, size_t ws_bytes,
                             mxq_stream_t stream);
mxq_status mxq_linear_bwd_dw(const void *dy, const void *x, int64_t M, int64_t N, int64_t K,
                             mxq_mode mode, void *ctx, void *dw, void *workspace, size_t ws_bytes,
                             mxq_stream_t stream);

/* ---- MoE expert layer, the same two modes ([TT] MoE MXFP8 mode; [FB]'s
 * weights are the experts' [E,K,N], so its forward weight quant along axis
 * -2 and its dX recompute along axis -1 are our row and column quants of the
 * stacked [E*N x K]).  x bf16 [T x K] routed rows grouped by d_offsets
 * (DEVICE, E+1, as for mxq_grouped_gemm), w bf16 [E x N x K] (expert e's
 * weight is rows [e*N, (e+1)*N) of the stacked [E*N x K]), dy bf16 [T x N];
 * y [T x N], dx [T x K], dw [E x N x K] bf16.  For group e:
 *   y_e = X_e W_e^T,  dX_e = dY_e W_e,  dW_e = dY_e^T X_e (zero for an empty group),
 * all MXFP8 with fp32 accumulation (the grouped GEMM kinds FWD, DX, DW).
 *  MXQ_SAVE_QUANT: the forward quantizes X (row quant and per-group column
 *      quant from one read) and W (row and column quant from one read) and
 *      keeps the column quants in ctx for the backward.
 *  MXQ_RECOMPUTE: the forward row-quantizes only and keeps nothing; the
 *      backward re-quantizes W along E*N and X per group from the bf16
 *      originals.
 * In both, bwd_dx quantizes dY once (row quant and per-group column quant)
 * and leaves the column quant in ctx for bwd_dw.  The two modes give
 * bitwise-identical y, dx and dw.  T > 0, 1 <= E <= 4096, N a positive
 * multiple of 128, K of 32; ctx (mxq_grouped_linear_ctx_bytes) carries state
 * from fwd to bwd_dx to bwd_dw of one step; workspace
 * (mxq_grouped_linear_workspace_bytes) is scratch for one call; all DEVICE,
 * 16-byte aligned.  Malformed offsets as for mxq_grouped_gemm. */
size_t mxq_grouped_linear_ctx_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode);
/* Bytes of ctx that live from the forward to the backward: the column quants
 * of X (per group, [K x t_pad]) and of W ([K x E*N]) with their scales for
 * SAVE, 0 for RECOMPUTE. */
size_t mxq_grouped_linear_saved_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode);
size_t mxq_grouped_linear_workspace_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode);
mxq_status mxq_grouped_linear_fwd(const void *x, const void *w, const int64_t *d_offsets, int E,
                                  int64_t T, int64_t N, int64_t K, mxq_mode mode, void *ctx, void *y,
                                  void *workspace, size_t ws_bytes, mxq_stream_t stream);
mxq_status mxq_grouped_linear_bwd_dx(const void *dy, const void *w, const int64_t *d_offsets, int E,
                                     int64_t T, int64_t N, int64_t K, mxq_mode mode, void *ctx, void *dx,
                                     void *workspace, size_t ws_bytes, mxq_stream_t stream);
mxq_status mxq_grouped_linear_bwd_dw(const void *dy, const void *x, const int64_t *d_offsets, int E,
                                     int64_t T, int64_t N, int64_t K, mxq_mode mode, void *ctx, void *dw,
                                     void *workspace, size_t ws_bytes, mxq_stream_t stream);

/* ---- Quantized-weight reuse ([FB]: the reuse flags of the MXFP8 matmul
 * path) ----
 * Within one optimizer step W does not change, so its quantization can be
 * made once and reused by every micro-batch's forward and input gradient:
 * mxq_linear_quantize_weight reads W once and writes row(W) and colT(W)
 * into a caller-owned cache (mxq_linear_weight_cache_bytes); the _wq entry
 * points then take W's quantization from the cache instead of from W.
 * Results are bitwise identical to mxq_linear_fwd / mxq_linear_bwd_dx (the
 * quantization is deterministic); the cache is valid until W changes.
 * `mode` then applies to X only (SAVE keeps colT(X) in ctx, RECOMPUTE
 * re-quantizes it in mxq_linear_bwd_dw, which serves both paths).  ctx of
 * the _wq path is mxq_linear_wq_ctx_bytes (no copy of colT(W)); workspace
 * needs at most mxq_linear_workspace_bytes. */
size_t mxq_linear_weight_cache_bytes(int64_t N, int64_t K);
size_t mxq_linear_wq_ctx_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode);
mxq_status mxq_linear_quantize_weight(const void *w, int64_t N, int64_t K, void *wcache,
                                      size_t cache_bytes, mxq_stream_t stream);
mxq_status mxq_linear_fwd_wq(const void *x, const void *wcache, int64_t M, int64_t N, int64_t K,
                             mxq_mode mode, void *ctx, void *y, void *workspace, size_t ws_bytes,
                             mxq_stream_t stream);
mxq_status mxq_linear_bwd_dx_wq(const void *dy, const void *wcache, int64_t M, int64_t N, int64_t K,
                                mxq_mode mode, void *ctx, void *dx, void *workspace,
                                size_t ws_bytes, mxq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Linear forward without caller-provided scratch                       */
/* ------------------------------------------------------------------ */

/* Device memory the library holds for mxq_linear_fwd_noalloc: 64 MiB on every
 * GPU that loads the library, kept until the process exits. */
#define MXQ_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* Y = X W^T of the MXFP8 linear layer -- the same y as mxq_linear_fwd -- for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * of this entry point.
 *
 * Who needs it: mxq_linear_fwd wants a caller-provided workspace for the
 * quantized operands.  A plug-in running inside a host framework that owns
 * the device memory pool and does not let plug-ins call cudaMalloc, or a
 * service that reserves its memory once at start-up and must not allocate
 * afterwards, has no workspace to give; this entry point uses scratch that
 * lives inside the library instead.
 *
 * x bf16 [M x K], w bf16 [N x K], y bf16 [M x N]: device pointers the caller
 * owns, 16-byte aligned.  M, N, K positive multiples of 32, and the row quants
 * of X and W (M*K + N*K code bytes plus their scale tiles, each rounded up to
 * 256 bytes) must fit in MXQ_NOALLOC_SCRATCH_BYTES -- otherwise
 * MXQ_ERR_INVALID_ARG, with the sizes in mxq_last_error_string().  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 * The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for the life
 * of the process: make that first call before any stream capture.  A
 * cudaDeviceReset (or anything else that destroys the device's primary
 * context) invalidates the kept address: after one, do not call this entry
 * point on that device again in the same process.  All calls share the one scratch array, which
 * keeps the last call's contents; each call rewrites everything it reads, so
 * nothing needs clearing.  Calls whose GPU work can overlap (on different
 * streams, or from different host threads) race on the array and corrupt
 * each other's results: issue them on one stream or otherwise serialize
 * them. */
mxq_status mxq_linear_fwd_noalloc(const void *x, const void *w, int64_t M, int64_t N, int64_t K, void *y,
                                  mxq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Diagnostics                                                          */
/* ------------------------------------------------------------------ */

/* Reason for the last non-OK status returned on this thread ("" if none). */
const char *mxq_last_error_string(void);

/* Synchronizes the current device, then reads and clears the device-side
 * error word (a variable inside the library, whose device address is looked
 * up once per device and kept, so it too is invalid after a cudaDeviceReset)
 * that kernels set when they give up (bit 0: an mbarrier wait
 * timed out; bit 1: a tensor-memory allocation failed; bit 2: a grouped
 * kernel found its group offsets malformed and did no work; bit 3: the debug
 * build of the library, compiled with MXQ_DEBUG, found a computed address
 * outside its buffer and skipped that access).  Returns MXQ_ERR_CUDA if bit 3
 * was set, else MXQ_ERR_INVALID_ARG if bit 2 was set, else MXQ_ERR_TIMEOUT if
 * any bit was set (*word receives the bits), MXQ_OK otherwise.  word may be
 * NULL. */
mxq_status mxq_poll_device_error(uint32_t *word);

/* Failure-detection self-test (no counterpart on the pages): launches one
 * kernel whose thread waits, with the same bounded-wait code every kernel of
 * this library uses, on an mbarrier that nothing arrives on.  After
 * timeout_ms (1..10000) the wait gives up, sets bit 0 of the device error
 * word and writes 1 to *d_gave_up (DEVICE int); the kernel then returns
 * normally, so the context stays usable.  mxq_poll_device_error reports and
 * clears the bit.  While the bit is set, GEMM launches skip their work. */
mxq_status mxq_selftest_wait_timeout(uint32_t timeout_ms, int *d_gave_up, mxq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MXQ_H */
