// mxq_api.cu -- the C ABI of libmxq (declared in include/mxq.h): argument
// validation, arch check, dispatch to the kernels, and the linear layer's
// saved-quant / recompute orchestration.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

thread_local std::string g_last_error;

mxq_status fail(mxq_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

mxq_status ok() {
    g_last_error.clear();
    return MXQ_OK;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;

mxq_status check_arch() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MXQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    static std::atomic<int> cc[kMaxDevices] = {};  // major*10+minor, 0 = unknown (racing threads store the same value)
    if (dev < 0 || dev >= kMaxDevices) return fail(MXQ_ERR_CUDA, "device index %d out of range", dev);
    int v = cc[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return fail(MXQ_ERR_CUDA, "cannot query compute capability of device %d", dev);
        v = major * 10 + minor;
        cc[dev].store(v, std::memory_order_relaxed);
    }
    if (v != 103)
        return fail(MXQ_ERR_ARCH, "libmxq is built for sm_103a (GB300); device %d is sm_%d", dev, v);
    return MXQ_OK;
}

mxq_status cuda_result(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(MXQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
inline size_t scale_bytes(int64_t rows, int64_t kb) {
    return static_cast<size_t>(ceil_div(rows, 128) * 128) * static_cast<size_t>(ceil_div(kb, 4) * 4);
}
// codes + scales of a K-major operand [rows x k]
inline size_t operand_bytes(int64_t rows, int64_t k) {
    return round256(static_cast<size_t>(rows) * static_cast<size_t>(k)) + round256(scale_bytes(rows, ceil_div(k, 32)));
}

struct Operand {
    uint8_t *q, *s;
};
inline Operand carve(uint8_t *&p, int64_t rows, int64_t k) {
    Operand o;
    o.q = p;
    p += round256(static_cast<size_t>(rows) * static_cast<size_t>(k));
    o.s = p;
    p += round256(scale_bytes(rows, ceil_div(k, 32)));
    return o;
}

mxq_status dense_gemm(const Operand &A, const Operand &B, int64_t M, int64_t N, int64_t K, void *c, int64_t ldc,
                      cudaStream_t st, const void *bias = nullptr) {
    if (M == 0 || N == 0) return ok();
    mxq::GemmProblem g{};
    g.mode = mxq::kDense;
    g.a = A.q; g.sa = A.s; g.a_rows = M; g.a_k = K;
    g.b = B.q; g.sb = B.s; g.b_rows = N; g.b_k = K;
    g.c = c; g.M = M; g.N = N; g.ldc = ldc; g.K = K;
    g.bias = bias;
    return cuda_result(mxq::launch_gemm(g, st), "mxq gemm launch");
}

// ---- linear-layer memory plan ----
// ctx:  SAVE: [colT(X): K x M][colT(dY): N x M][colT(W): K x N];  RECOMPUTE: [colT(dY)]
//       (the backward dW reads only the prefix [colT(X)][colT(dY)], which the
//       cached-weight entry points share; they keep colT(W) in the cache)
// ws :  fwd [row(X)][row(W)];  bwd_dx [row(dY)][colT(W) if RECOMPUTE];  bwd_dw [colT(X) if RECOMPUTE]
// weight cache: [row(W): N x K][colT(W): K x N]
size_t saved_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    return mode == MXQ_SAVE_QUANT ? operand_bytes(K, M) + operand_bytes(K, N) : 0;
}
size_t ctx_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    return saved_bytes(M, N, K, mode) + operand_bytes(N, M);
}
size_t wq_ctx_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    return (mode == MXQ_SAVE_QUANT ? operand_bytes(K, M) : 0) + operand_bytes(N, M);
}
size_t ws_fwd(int64_t M, int64_t N, int64_t K) { return operand_bytes(M, K) + operand_bytes(N, K); }
size_t ws_dx(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    return operand_bytes(M, N) + (mode == MXQ_RECOMPUTE ? operand_bytes(K, N) : 0);
}
size_t ws_dw(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    return mode == MXQ_RECOMPUTE ? operand_bytes(K, M) : 0;
}

// ---- grouped (MoE expert) linear-layer memory plan ----
// x [T x K] routed rows grouped by the offsets, the stacked expert weights
// w [E*N x K], dy [T x N]; t_pad = mxq_grouped_padded_rows(T, E); gcolT = the
// per-group column quant [C x t_pad]; prow = a row quant whose scales are in
// the per-group padded layout ([T x C] codes, swz(t_pad, C/32) scales).
// ctx:  SAVE: [gcolT(X): K x t_pad][gcolT(dY): N x t_pad][colT(W): K x E*N];  RECOMPUTE: [gcolT(dY)]
// ws :  fwd [prow(X)][row(W)];  bwd_dx [prow(dY)][colT(W) if RECOMPUTE];  bwd_dw [gcolT(X) if RECOMPUTE]
inline size_t prow_bytes(int64_t T, int64_t t_pad, int64_t k) {
    return round256(static_cast<size_t>(T) * static_cast<size_t>(k)) + round256(scale_bytes(t_pad, ceil_div(k, 32)));
}
inline Operand carve_prow(uint8_t *&p, int64_t T, int64_t t_pad, int64_t k) {
    Operand o;
    o.q = p;
    p += round256(static_cast<size_t>(T) * static_cast<size_t>(k));
    o.s = p;
    p += round256(scale_bytes(t_pad, ceil_div(k, 32)));
    return o;
}
size_t g_saved_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    const int64_t tp = mxq_grouped_padded_rows(T, E);
    return mode == MXQ_SAVE_QUANT ? operand_bytes(K, tp) + operand_bytes(K, static_cast<int64_t>(E) * N) : 0;
}
size_t g_ctx_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    return g_saved_bytes(T, E, N, K, mode) + operand_bytes(N, mxq_grouped_padded_rows(T, E));
}
size_t g_ws_fwd(int64_t T, int E, int64_t N, int64_t K) {
    return prow_bytes(T, mxq_grouped_padded_rows(T, E), K) + operand_bytes(static_cast<int64_t>(E) * N, K);
}
size_t g_ws_dx(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    return prow_bytes(T, mxq_grouped_padded_rows(T, E), N) +
           (mode == MXQ_RECOMPUTE ? operand_bytes(K, static_cast<int64_t>(E) * N) : 0);
}
size_t g_ws_dw(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    return mode == MXQ_RECOMPUTE ? operand_bytes(K, mxq_grouped_padded_rows(T, E)) : 0;
}

mxq_status check_grouped_linear(const void *a, const void *b, const int64_t *d_offsets, int E, int64_t T, int64_t N,
                                int64_t K, mxq_mode mode, void *ctx, void *out, void *ws, size_t ws_bytes,
                                size_t ws_need) {
    if (!a || !b || !ctx || !out) return fail(MXQ_ERR_INVALID_ARG, "null tensor pointer");
    if (!al16(a) || !al16(b) || !al16(ctx) || !al16(out) || (ws && !al16(ws)))
        return fail(MXQ_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!d_offsets || (reinterpret_cast<uintptr_t>(d_offsets) & 7))
        return fail(MXQ_ERR_INVALID_ARG, "d_offsets must be a non-null 8-byte aligned device pointer");
    if (mode != MXQ_SAVE_QUANT && mode != MXQ_RECOMPUTE) return fail(MXQ_ERR_INVALID_ARG, "bad mode %d", (int)mode);
    if (E < 1 || E > 4096) return fail(MXQ_ERR_INVALID_ARG, "E must be in [1, 4096]");
    if (T <= 0 || N <= 0 || K <= 0 || N % 128 || K % 32)
        return fail(MXQ_ERR_INVALID_ARG, "T > 0, N a positive multiple of 128, K of 32 (got %lld, %lld, %lld)",
                    (long long)T, (long long)N, (long long)K);
    if (T > (1ll << 31) || K > (1ll << 31) || static_cast<int64_t>(E) * N > (1ll << 31) ||
        mxq_grouped_padded_rows(T, E) / 128 > 65535)
        return fail(MXQ_ERR_UNSUPPORTED, "dimension above the supported range");
    if (ws_need > 0 && (!ws || ws_bytes < ws_need))
        return fail(MXQ_ERR_INVALID_ARG, "workspace too small: need %zu bytes, got %zu", ws_need, ws ? ws_bytes : 0);
    return MXQ_OK;
}

// The grouped GEMM problem of one MoE matmul (arguments already checked).
//  FWD: out[T x N] rows of group e = A rows . B_e^T, A [T x K], B [E*N x K] (expert e's rows [eN, (e+1)N)).
//  DX:  out[T x K] rows of group e = A rows . B_e^T, A [T x N], B = colT(W) [K x E*N] (expert e's columns).
//  DW:  out[E x N x K], per-group contraction over the padded column quants [N x t_pad], [K x t_pad].
//  t_pad for FWD/DX: 0 = A's scales swz(T, .), else the per-group padded layout swz(t_pad, .).
mxq::GemmProblem grouped_problem(mxq_gg_kind kind, const uint8_t *a, const uint8_t *sa, const uint8_t *b,
                                 const uint8_t *sb, const int64_t *d_offsets, int E, int64_t T, int64_t N, int64_t K,
                                 int64_t t_pad, void *out_bf16) {
    mxq::GemmProblem g{};
    g.offsets = d_offsets;
    g.E = E;
    g.c = out_bf16;
    g.T = T;
    g.a = a; g.sa = sa; g.b = b; g.sb = sb;
    if (kind == MXQ_GG_FWD || kind == MXQ_GG_DX) {
        g.mode = mxq::kGroupedRows;
        g.a_row_pad = t_pad;
        if (kind == MXQ_GG_FWD) {  // out[T x N] = X[T x K] . W_e[N x K]^T
            g.a_rows = T; g.a_k = K;
            g.b_rows = static_cast<int64_t>(E) * N; g.b_k = K;
            g.M = T; g.N = N; g.ldc = N; g.K = K;
            g.b_row_per_expert = N; g.b_k_per_expert = 0;
        } else {  // out[T x K] = dY[T x N] . colT(W)_e[K x N]^T
            g.a_rows = T; g.a_k = N;
            g.b_rows = K; g.b_k = static_cast<int64_t>(E) * N;
            g.M = T; g.N = K; g.ldc = K; g.K = N;
            g.b_row_per_expert = 0; g.b_k_per_expert = N;
        }
    } else {
        g.mode = mxq::kGroupedK;
        g.a_rows = N; g.a_k = t_pad;
        g.b_rows = K; g.b_k = t_pad;
        g.M = N; g.N = K; g.ldc = K;
        g.c_expert_stride = N * K;
    }
    return g;
}

mxq_status check_linear(const void *a, const void *b, int64_t M, int64_t N, int64_t K, mxq_mode mode, void *ctx,
                        void *out, void *ws, size_t ws_bytes, size_t ws_need) {
    if (!a || !b || !ctx || !out) return fail(MXQ_ERR_INVALID_ARG, "null tensor pointer");
    if (!al16(a) || !al16(b) || !al16(ctx) || !al16(out) || (ws && !al16(ws)))
        return fail(MXQ_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (mode != MXQ_SAVE_QUANT && mode != MXQ_RECOMPUTE) return fail(MXQ_ERR_INVALID_ARG, "bad mode %d", (int)mode);
    if (M <= 0 || N <= 0 || K <= 0 || M % 32 || N % 32 || K % 32)
        return fail(MXQ_ERR_INVALID_ARG, "M, N, K must be positive multiples of 32 (got %lld, %lld, %lld)",
                    (long long)M, (long long)N, (long long)K);
    if (M > (1ll << 31) || N > (1ll << 31) || K > (1ll << 31))
        return fail(MXQ_ERR_UNSUPPORTED, "dimension above 2^31");
    if (ws_need > 0 && (!ws || ws_bytes < ws_need))
        return fail(MXQ_ERR_INVALID_ARG, "workspace too small: need %zu bytes, got %zu", ws_need, ws ? ws_bytes : 0);
    return MXQ_OK;
}

}  // namespace

// Error reporting and the arch check for entry points defined in other
// translation units (same behaviour as the helpers above).
namespace mxq {
mxq_status api_fail(mxq_status s, const char *msg) { return fail(s, "%s", msg); }
mxq_status api_check_arch() { return check_arch(); }
mxq_status api_cuda_result(cudaError_t e, const char *what) { return cuda_result(e, what); }
}  // namespace mxq

extern "C" {

const char *mxq_last_error_string(void) { return g_last_error.c_str(); }

size_t mxq_scale_bytes(int64_t rows, int64_t k_blocks) {
    if (rows <= 0 || k_blocks <= 0) return 0;
    return scale_bytes(rows, k_blocks);
}

int64_t mxq_grouped_padded_rows(int64_t T, int E) {
    if (T < 0 || E < 0) return 0;
    return 128 * (ceil_div(T, 128) + E);
}

mxq_status mxq_selftest_wait_timeout(uint32_t timeout_ms, int *d_gave_up, mxq_stream_t stream) {
    if (!d_gave_up || (reinterpret_cast<uintptr_t>(d_gave_up) & 3))
        return fail(MXQ_ERR_INVALID_ARG, "d_gave_up must be a non-null int pointer");
    if (timeout_ms == 0 || timeout_ms > 10000) return fail(MXQ_ERR_INVALID_ARG, "timeout_ms must be in [1, 10000]");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(mxq::launch_selftest_wait(static_cast<uint64_t>(timeout_ms) * 1000000ull, d_gave_up,
                                                 reinterpret_cast<cudaStream_t>(stream)),
                       "mxq_selftest_wait_timeout launch");
}

mxq_status mxq_poll_device_error(uint32_t *word) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(MXQ_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    unsigned int w = 0;
    e = mxq::read_and_clear_device_error(&w);
    if (e != cudaSuccess) return fail(MXQ_ERR_CUDA, "read device error word: %s", cudaGetErrorString(e));
    if (word) *word = w;
    if (w & 8u)
        return fail(MXQ_ERR_CUDA,
                    "a bounds check of the debug build found an access outside its buffer and skipped it "
                    "(device error bits 0x%x)",
                    w);
    if (w & 4u)
        return fail(MXQ_ERR_INVALID_ARG,
                    "a grouped kernel found its group offsets malformed (they must rise from off[0] = 0 to "
                    "off[E] = T without decreasing) and skipped its work (device error bits 0x%x)",
                    w);
    if (w) return fail(MXQ_ERR_TIMEOUT, "a kernel reported device error bits 0x%x", w);
    return ok();
}

mxq_status mxq_validate_group_offsets(const int64_t *offsets, int E, int64_t T) {
    if (!offsets) return fail(MXQ_ERR_INVALID_ARG, "offsets is null");
    if (E < 1 || E > 4096) return fail(MXQ_ERR_INVALID_ARG, "E must be in [1, 4096]");
    if (T < 0) return fail(MXQ_ERR_INVALID_ARG, "T must be >= 0");
    if (offsets[0] != 0) return fail(MXQ_ERR_INVALID_ARG, "off[0] = %lld, must be 0", (long long)offsets[0]);
    for (int e = 0; e < E; e++)
        if (offsets[e + 1] < offsets[e])
            return fail(MXQ_ERR_INVALID_ARG, "off[%d] = %lld < off[%d] = %lld: offsets must not decrease", e + 1,
                        (long long)offsets[e + 1], e, (long long)offsets[e]);
    if (offsets[E] != T)
        return fail(MXQ_ERR_INVALID_ARG, "off[E] = %lld, must equal T = %lld", (long long)offsets[E], (long long)T);
    return ok();
}

mxq_status mxq_check_group_offsets(const int64_t *d_offsets, int E, int64_t T, mxq_stream_t stream) {
    if (!d_offsets || (reinterpret_cast<uintptr_t>(d_offsets) & 7))
        return fail(MXQ_ERR_INVALID_ARG, "d_offsets must be a non-null 8-byte aligned device pointer");
    if (E < 1 || E > 4096) return fail(MXQ_ERR_INVALID_ARG, "E must be in [1, 4096]");
    if (T < 0) return fail(MXQ_ERR_INVALID_ARG, "T must be >= 0");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(mxq::launch_check_offsets(d_offsets, E, T, reinterpret_cast<cudaStream_t>(stream)),
                       "mxq_check_group_offsets launch");
}

mxq_status mxq_quantize(const void *x, mxq_dtype dtype, int64_t rows, int64_t cols, int64_t ldx, int axis,
                        mxq_fmt fmt, int dual_axis, void *q_row, void *s_row, void *q_colT, void *s_colT,
                        mxq_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (dtype != MXQ_BF16 && dtype != MXQ_F32) return fail(MXQ_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if (fmt != MXQ_E4M3 && fmt != MXQ_E2M1) return fail(MXQ_ERR_INVALID_ARG, "bad fmt %d", (int)fmt);
    if (!dual_axis && axis != -1 && axis != -2) return fail(MXQ_ERR_INVALID_ARG, "axis must be -1 or -2");
    const bool want_row = dual_axis || axis == -1, want_col = dual_axis || axis == -2;
    if (fmt == MXQ_E2M1 && (want_col || dual_axis))
        return fail(MXQ_ERR_UNSUPPORTED, "E2M1 quantization is along the last axis only");
    if (fmt == MXQ_E4M3 && dtype != MXQ_BF16) return fail(MXQ_ERR_UNSUPPORTED, "MXFP8 quantization takes bf16 input");
    if (ldx < cols || ldx % 8) return fail(MXQ_ERR_INVALID_ARG, "ldx must be >= cols and a multiple of 8");
    if (want_row && cols % 32) return fail(MXQ_ERR_INVALID_ARG, "cols must be a multiple of 32 along the block axis");
    if (want_col && cols % 8) return fail(MXQ_ERR_INVALID_ARG, "column quant needs cols % 8 == 0");
    if (rows > (1ll << 31) || cols > (1ll << 31) || ceil_div(rows, 128) > 65535)
        return fail(MXQ_ERR_UNSUPPORTED, "tensor too large for one launch");
    if (rows == 0 || cols == 0) return ok();
    if (!x || !al16(x)) return fail(MXQ_ERR_INVALID_ARG, "x must be a non-null 16-byte aligned pointer");
    if (want_row && (!q_row || !s_row || !al16(q_row) || !al16(s_row)))
        return fail(MXQ_ERR_INVALID_ARG, "q_row/s_row must be non-null 16-byte aligned pointers");
    if (want_col && (!q_colT || !s_colT || !al16(q_colT) || !al16(s_colT)))
        return fail(MXQ_ERR_INVALID_ARG, "q_colT/s_colT must be non-null 16-byte aligned pointers");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (want_col) {
        e = mxq::launch_quant_cols(static_cast<const uint16_t *>(x), rows, cols, ldx,
                                   want_row ? static_cast<uint8_t *>(q_row) : nullptr,
                                   want_row ? static_cast<uint8_t *>(s_row) : nullptr, static_cast<uint8_t *>(q_colT),
                                   static_cast<uint8_t *>(s_colT), st);
    } else {
        e = mxq::launch_quant_rows(x, dtype == MXQ_F32, fmt == MXQ_E2M1 ? 1 : 0, rows, cols, ldx,
                                   static_cast<uint8_t *>(q_row), static_cast<uint8_t *>(s_row), st);
    }
    return cuda_result(e, "mxq_quantize launch");
}

namespace {
mxq_status grouped_dual(const void *x_bf16, int64_t rows, int64_t cols, const int64_t *d_offsets, int E,
                        int64_t t_pad, void *q_row, void *s_row, void *q_colT, void *s_colT, mxq_stream_t stream,
                        bool row_pad) {
    if (rows < 0 || cols < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (E < 1 || E > 4096) return fail(MXQ_ERR_INVALID_ARG, "E must be in [1, 4096]");
    if (cols % 8) return fail(MXQ_ERR_INVALID_ARG, "cols must be a multiple of 8");
    const bool want_row = q_row != nullptr || s_row != nullptr;
    if (want_row && cols % 32) return fail(MXQ_ERR_INVALID_ARG, "cols must be a multiple of 32 for the row quant");
    if (t_pad < 0 || t_pad % 128 || t_pad < mxq_grouped_padded_rows(rows, E))
        return fail(MXQ_ERR_INVALID_ARG, "t_pad must be a multiple of 128 and >= mxq_grouped_padded_rows(rows, E) = %lld",
                    (long long)mxq_grouped_padded_rows(rows, E));
    if (t_pad / 128 > 65535 || cols > (1ll << 31)) return fail(MXQ_ERR_UNSUPPORTED, "tensor too large for one launch");
    if (cols == 0) return ok();
    if (!d_offsets || (reinterpret_cast<uintptr_t>(d_offsets) & 7))
        return fail(MXQ_ERR_INVALID_ARG, "d_offsets must be a non-null 8-byte aligned device pointer");
    if ((rows > 0 && (!x_bf16 || !al16(x_bf16))) || !q_colT || !s_colT || !al16(q_colT) || !al16(s_colT))
        return fail(MXQ_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned");
    if (want_row && (!q_row || !s_row || !al16(q_row) || !al16(s_row)))
        return fail(MXQ_ERR_INVALID_ARG, "q_row/s_row must both be non-null and 16-byte aligned");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(mxq::launch_quant_cols_grouped(static_cast<const uint16_t *>(x_bf16), rows, cols, d_offsets, E,
                                                      t_pad, static_cast<uint8_t *>(q_row),
                                                      static_cast<uint8_t *>(s_row), static_cast<uint8_t *>(q_colT),
                                                      static_cast<uint8_t *>(s_colT),
                                                      reinterpret_cast<cudaStream_t>(stream), row_pad),
                       "mxq_quantize_grouped_dual launch");
}
}  // namespace

mxq_status mxq_quantize_grouped_dual(const void *x_bf16, int64_t rows, int64_t cols, const int64_t *d_offsets,
                                     int E, int64_t t_pad, void *q_row, void *s_row, void *q_colT, void *s_colT,
                                     mxq_stream_t stream) {
    return grouped_dual(x_bf16, rows, cols, d_offsets, E, t_pad, q_row, s_row, q_colT, s_colT, stream, false);
}

mxq_status mxq_quantize_grouped_dual_padded(const void *x_bf16, int64_t rows, int64_t cols,
                                            const int64_t *d_offsets, int E, int64_t t_pad, void *q_row,
                                            void *s_row, void *q_colT, void *s_colT, mxq_stream_t stream) {
    if (!q_row || !s_row) return fail(MXQ_ERR_INVALID_ARG, "q_row and s_row are required");
    return grouped_dual(x_bf16, rows, cols, d_offsets, E, t_pad, q_row, s_row, q_colT, s_colT, stream, true);
}

mxq_status mxq_quantize_grouped_col(const void *x_bf16, int64_t rows, int64_t cols, const int64_t *d_offsets, int E,
                                    int64_t t_pad, void *q_colT, void *s_colT, mxq_stream_t stream) {
    return mxq_quantize_grouped_dual(x_bf16, rows, cols, d_offsets, E, t_pad, nullptr, nullptr, q_colT, s_colT,
                                     stream);
}

mxq_status mxq_qdq_mxfp4(const float *x, float *y, int64_t rows, int64_t cols, int block_size, float scale_factor,
                         mxq_stream_t stream) {
    if (block_size != 32) return fail(MXQ_ERR_UNSUPPORTED, "block_size must be 32 (got %d)", block_size);
    if (!(scale_factor > 0.0f) || !(scale_factor <= 3.402823466e38f))
        return fail(MXQ_ERR_INVALID_ARG, "scale_factor must be finite and > 0");
    if (rows < 0 || cols < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (rows == 0 || cols == 0) return ok();
    if (!x || !y || (reinterpret_cast<uintptr_t>(x) & 3) || (reinterpret_cast<uintptr_t>(y) & 3))
        return fail(MXQ_ERR_INVALID_ARG, "x and y must be non-null fp32 pointers");
    if (rows > (1ll << 40) / (cols > 0 ? cols : 1)) return fail(MXQ_ERR_UNSUPPORTED, "tensor too large");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(
        mxq::launch_qdq_mxfp4(x, y, nullptr, rows, cols, scale_factor, reinterpret_cast<cudaStream_t>(stream)),
        "mxq_qdq_mxfp4 launch");
}

mxq_status mxq_qdq_mxfp4_bf16(const void *x, void *y, int64_t rows, int64_t cols, int block_size, float scale_factor,
                              mxq_stream_t stream) {
    if (block_size != 32) return fail(MXQ_ERR_UNSUPPORTED, "block_size must be 32 (got %d)", block_size);
    if (!(scale_factor > 0.0f) || !(scale_factor <= 3.402823466e38f))
        return fail(MXQ_ERR_INVALID_ARG, "scale_factor must be finite and > 0");
    if (rows < 0 || cols < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (rows == 0 || cols == 0) return ok();
    if (!x || !y || !al16(x) || !al16(y)) return fail(MXQ_ERR_INVALID_ARG, "x and y must be 16-byte aligned bf16 pointers");
    if (cols % 32) return fail(MXQ_ERR_UNSUPPORTED, "bf16 quant-dequant needs cols %% 32 == 0 (got %lld)", (long long)cols);
    if (rows > (1ll << 40) / cols) return fail(MXQ_ERR_UNSUPPORTED, "tensor too large");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(mxq::launch_qdq_mxfp4_bf16(static_cast<const uint16_t *>(x), static_cast<uint16_t *>(y), rows,
                                                  cols, scale_factor, reinterpret_cast<cudaStream_t>(stream)),
                       "mxq_qdq_mxfp4_bf16 launch");
}

mxq_status mxq_mxfp4_ste_forward(const float *x, float *y, uint32_t *sat_mask, int64_t rows, int64_t cols,
                                 int block_size, float scale_factor, mxq_stream_t stream) {
    if (block_size != 32) return fail(MXQ_ERR_UNSUPPORTED, "block_size must be 32 (got %d)", block_size);
    if (!(scale_factor > 0.0f) || !(scale_factor <= 3.402823466e38f))
        return fail(MXQ_ERR_INVALID_ARG, "scale_factor must be finite and > 0");
    if (rows < 0 || cols < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (rows == 0 || cols == 0) return ok();
    if (!x || !y || (reinterpret_cast<uintptr_t>(x) & 3) || (reinterpret_cast<uintptr_t>(y) & 3))
        return fail(MXQ_ERR_INVALID_ARG, "x and y must be non-null fp32 pointers");
    if (!sat_mask || (reinterpret_cast<uintptr_t>(sat_mask) & 3))
        return fail(MXQ_ERR_INVALID_ARG, "sat_mask must be a non-null uint32 pointer");
    if (rows > (1ll << 40) / cols) return fail(MXQ_ERR_UNSUPPORTED, "tensor too large");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(
        mxq::launch_qdq_mxfp4(x, y, sat_mask, rows, cols, scale_factor, reinterpret_cast<cudaStream_t>(stream)),
        "mxq_mxfp4_ste_forward launch");
}

mxq_status mxq_mxfp4_ste_backward(const float *grad_y, const uint32_t *sat_mask, int64_t rows, int64_t cols,
                                  float *grad_x, mxq_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (rows == 0 || cols == 0) return ok();
    if (!grad_y || !grad_x || (reinterpret_cast<uintptr_t>(grad_y) & 3) || (reinterpret_cast<uintptr_t>(grad_x) & 3))
        return fail(MXQ_ERR_INVALID_ARG, "grad_y and grad_x must be non-null fp32 pointers");
    if (!sat_mask || (reinterpret_cast<uintptr_t>(sat_mask) & 3))
        return fail(MXQ_ERR_INVALID_ARG, "sat_mask must be a non-null uint32 pointer");
    if (rows > (1ll << 40) / cols) return fail(MXQ_ERR_UNSUPPORTED, "tensor too large");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(
        mxq::launch_ste_backward(grad_y, sat_mask, grad_x, rows, cols, reinterpret_cast<cudaStream_t>(stream)),
        "mxq_mxfp4_ste_backward launch");
}

mxq_status mxq_gemm(const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb, int64_t M, int64_t N,
                    int64_t K, void *c_bf16, int64_t ldc, mxq_stream_t stream) {
    if (M < 0 || N < 0) return fail(MXQ_ERR_INVALID_ARG, "negative size");
    if (K <= 0 || K % 32) return fail(MXQ_ERR_INVALID_ARG, "K must be a positive multiple of 32 (got %lld)", (long long)K);
    if (ldc < N || ldc % 8) return fail(MXQ_ERR_INVALID_ARG, "ldc must be >= N and a multiple of 8");
    if (M > (1ll << 31) || N > (1ll << 31) || K > (1ll << 31)) return fail(MXQ_ERR_UNSUPPORTED, "dimension above 2^31");
    if (M == 0 || N == 0) return ok();
    if (!a || !sa || !b || !sb || !c_bf16 || !al16(a) || !al16(sa) || !al16(b) || !al16(sb) || !al16(c_bf16))
        return fail(MXQ_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned");
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    Operand A{const_cast<uint8_t *>(a), const_cast<uint8_t *>(sa)}, B{const_cast<uint8_t *>(b), const_cast<uint8_t *>(sb)};
    return dense_gemm(A, B, M, N, K, c_bf16, ldc, reinterpret_cast<cudaStream_t>(stream));
}

mxq_status mxq_grouped_gemm(mxq_gg_kind kind, const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb,
                            const int64_t *d_offsets, int E, int64_t T, int64_t N, int64_t K, int64_t t_pad,
                            void *out_bf16, mxq_stream_t stream) {
    if (kind != MXQ_GG_FWD && kind != MXQ_GG_DX && kind != MXQ_GG_DW) return fail(MXQ_ERR_INVALID_ARG, "bad kind");
    if (E < 1 || E > 4096) return fail(MXQ_ERR_INVALID_ARG, "E must be in [1, 4096]");
    if (T < 0 || N <= 0 || K <= 0) return fail(MXQ_ERR_INVALID_ARG, "bad sizes");
    if (N > (1ll << 31) || K > (1ll << 31) || T > (1ll << 31) || static_cast<int64_t>(E) * N > (1ll << 31))
        return fail(MXQ_ERR_UNSUPPORTED, "dimension above 2^31");
    if (!d_offsets || (reinterpret_cast<uintptr_t>(d_offsets) & 7))
        return fail(MXQ_ERR_INVALID_ARG, "d_offsets must be a non-null 8-byte aligned device pointer");
    if (!a || !sa || !b || !sb || !out_bf16 || !al16(a) || !al16(sa) || !al16(b) || !al16(sb) || !al16(out_bf16))
        return fail(MXQ_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned");
    if (kind == MXQ_GG_FWD || kind == MXQ_GG_DX) {
        if (N % 128) return fail(MXQ_ERR_INVALID_ARG, "N must be a multiple of 128 for the grouped forward/dX");
        if (K % 32) return fail(MXQ_ERR_INVALID_ARG, "K must be a multiple of 32");
        if (t_pad != 0 && (t_pad < 0 || t_pad % 128 || t_pad < mxq_grouped_padded_rows(T, E)))
            return fail(MXQ_ERR_INVALID_ARG,
                        "t_pad must be 0 or a multiple of 128 and >= mxq_grouped_padded_rows(T, E) = %lld",
                        (long long)mxq_grouped_padded_rows(T, E));
        if (t_pad > (1ll << 31)) return fail(MXQ_ERR_UNSUPPORTED, "t_pad above 2^31");
        if (T == 0) return ok();
    } else {
        if (t_pad <= 0 || t_pad % 128 || t_pad < mxq_grouped_padded_rows(T, E))
            return fail(MXQ_ERR_INVALID_ARG, "t_pad must be a multiple of 128 and >= mxq_grouped_padded_rows(T, E)");
        if (t_pad > (1ll << 31)) return fail(MXQ_ERR_UNSUPPORTED, "t_pad above 2^31");
    }
    const mxq::GemmProblem g = grouped_problem(kind, a, sa, b, sb, d_offsets, E, T, N, K, t_pad, out_bf16);
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    return cuda_result(mxq::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)), "mxq_grouped_gemm launch");
}

size_t mxq_linear_ctx_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return ctx_bytes(M, N, K, mode);
}
size_t mxq_linear_saved_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return saved_bytes(M, N, K, mode);
}
size_t mxq_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    size_t w = ws_fwd(M, N, K);
    if (ws_dx(M, N, K, mode) > w) w = ws_dx(M, N, K, mode);
    if (ws_dw(M, N, K, mode) > w) w = ws_dw(M, N, K, mode);
    return w;
}

mxq_status mxq_linear_fwd(const void *x, const void *w, int64_t M, int64_t N, int64_t K, mxq_mode mode, void *ctx,
                          void *y, void *workspace, size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_linear(x, w, M, N, K, mode, ctx, y, workspace, ws_bytes, ws_fwd(M, N, K));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const Operand xq = carve(wp, M, K), wq = carve(wp, N, K);
    cudaError_t e;
    if (mode == MXQ_SAVE_QUANT) {
        uint8_t *cp = static_cast<uint8_t *>(ctx);
        const Operand xT = carve(cp, K, M);
        (void)carve(cp, N, M);  // colT(dY), written by bwd_dx
        const Operand wT = carve(cp, K, N);
        e = mxq::launch_quant_cols(static_cast<const uint16_t *>(x), M, K, K, xq.q, xq.s, xT.q, xT.s, st);
        if (e == cudaSuccess)
            e = mxq::launch_quant_cols(static_cast<const uint16_t *>(w), N, K, K, wq.q, wq.s, wT.q, wT.s, st);
    } else {
        e = mxq::launch_quant_rows(x, false, 0, M, K, K, xq.q, xq.s, st);
        if (e == cudaSuccess) e = mxq::launch_quant_rows(w, false, 0, N, K, K, wq.q, wq.s, st);
    }
    if (e != cudaSuccess) return cuda_result(e, "mxq_linear_fwd quant launch");
    return dense_gemm(xq, wq, M, N, K, y, N, st);
}

mxq_status mxq_linear_bwd_dx(const void *dy, const void *w, int64_t M, int64_t N, int64_t K, mxq_mode mode, void *ctx,
                             void *dx, void *workspace, size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_linear(dy, w, M, N, K, mode, ctx, dx, workspace, ws_bytes, ws_dx(M, N, K, mode));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *cp = static_cast<uint8_t *>(ctx);
    if (mode == MXQ_SAVE_QUANT) (void)carve(cp, K, M);
    const Operand dyT = carve(cp, N, M);
    Operand wT{};
    if (mode == MXQ_SAVE_QUANT) wT = carve(cp, K, N);
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const Operand dyq = carve(wp, M, N);
    cudaError_t e = mxq::launch_quant_cols(static_cast<const uint16_t *>(dy), M, N, N, dyq.q, dyq.s, dyT.q, dyT.s, st);
    if (e == cudaSuccess && mode == MXQ_RECOMPUTE) {
        wT = carve(wp, K, N);
        e = mxq::launch_quant_cols(static_cast<const uint16_t *>(w), N, K, K, nullptr, nullptr, wT.q, wT.s, st);
    }
    if (e != cudaSuccess) return cuda_result(e, "mxq_linear_bwd_dx quant launch");
    return dense_gemm(dyq, wT, M, K, N, dx, K, st);
}

mxq_status mxq_linear_bwd_dw(const void *dy, const void *x, int64_t M, int64_t N, int64_t K, mxq_mode mode, void *ctx,
                             void *dw, void *workspace, size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_linear(dy, x, M, N, K, mode, ctx, dw, workspace, ws_bytes, ws_dw(M, N, K, mode));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *cp = static_cast<uint8_t *>(ctx);
    Operand xT{};
    if (mode == MXQ_SAVE_QUANT) xT = carve(cp, K, M);
    const Operand dyT = carve(cp, N, M);
    if (mode == MXQ_RECOMPUTE) {
        uint8_t *wp = static_cast<uint8_t *>(workspace);
        xT = carve(wp, K, M);
        cudaError_t e = mxq::launch_quant_cols(static_cast<const uint16_t *>(x), M, K, K, nullptr, nullptr, xT.q, xT.s, st);
        if (e != cudaSuccess) return cuda_result(e, "mxq_linear_bwd_dw quant launch");
    }
    return dense_gemm(dyT, xT, N, K, M, dw, K, st);
}

size_t mxq_linear_weight_cache_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return operand_bytes(N, K) + operand_bytes(K, N);
}
size_t mxq_linear_wq_ctx_bytes(int64_t M, int64_t N, int64_t K, mxq_mode mode) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return wq_ctx_bytes(M, N, K, mode);
}

mxq_status mxq_linear_quantize_weight(const void *w, int64_t N, int64_t K, void *wcache, size_t cache_bytes,
                                      mxq_stream_t stream) {
    if (!w || !wcache) return fail(MXQ_ERR_INVALID_ARG, "null tensor pointer");
    if (!al16(w) || !al16(wcache)) return fail(MXQ_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (N <= 0 || K <= 0 || N % 32 || K % 32)
        return fail(MXQ_ERR_INVALID_ARG, "N, K must be positive multiples of 32 (got %lld, %lld)", (long long)N,
                    (long long)K);
    if (N > (1ll << 31) || K > (1ll << 31)) return fail(MXQ_ERR_UNSUPPORTED, "dimension above 2^31");
    if (cache_bytes < mxq_linear_weight_cache_bytes(N, K))
        return fail(MXQ_ERR_INVALID_ARG, "weight cache too small: need %zu bytes, got %zu",
                    mxq_linear_weight_cache_bytes(N, K), cache_bytes);
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    uint8_t *cp = static_cast<uint8_t *>(wcache);
    const Operand wq = carve(cp, N, K), wT = carve(cp, K, N);
    return cuda_result(mxq::launch_quant_cols(static_cast<const uint16_t *>(w), N, K, K, wq.q, wq.s, wT.q, wT.s,
                                              reinterpret_cast<cudaStream_t>(stream)),
                       "mxq_linear_quantize_weight launch");
}

mxq_status mxq_linear_fwd_wq(const void *x, const void *wcache, int64_t M, int64_t N, int64_t K, mxq_mode mode,
                             void *ctx, void *y, void *workspace, size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_linear(x, wcache, M, N, K, mode, ctx, y, workspace, ws_bytes, operand_bytes(M, K));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const Operand xq = carve(wp, M, K);
    uint8_t *cc = static_cast<uint8_t *>(const_cast<void *>(wcache));
    const Operand wq = carve(cc, N, K);
    cudaError_t e;
    if (mode == MXQ_SAVE_QUANT) {
        uint8_t *cp = static_cast<uint8_t *>(ctx);
        const Operand xT = carve(cp, K, M);
        e = mxq::launch_quant_cols(static_cast<const uint16_t *>(x), M, K, K, xq.q, xq.s, xT.q, xT.s, st);
    } else {
        e = mxq::launch_quant_rows(x, false, 0, M, K, K, xq.q, xq.s, st);
    }
    if (e != cudaSuccess) return cuda_result(e, "mxq_linear_fwd_wq quant launch");
    return dense_gemm(xq, wq, M, N, K, y, N, st);
}

mxq_status mxq_linear_bwd_dx_wq(const void *dy, const void *wcache, int64_t M, int64_t N, int64_t K, mxq_mode mode,
                                void *ctx, void *dx, void *workspace, size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_linear(dy, wcache, M, N, K, mode, ctx, dx, workspace, ws_bytes, operand_bytes(M, N));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *cp = static_cast<uint8_t *>(ctx);
    if (mode == MXQ_SAVE_QUANT) (void)carve(cp, K, M);
    const Operand dyT = carve(cp, N, M);
    uint8_t *cc = static_cast<uint8_t *>(const_cast<void *>(wcache));
    (void)carve(cc, N, K);
    const Operand wT = carve(cc, K, N);
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const Operand dyq = carve(wp, M, N);
    cudaError_t e = mxq::launch_quant_cols(static_cast<const uint16_t *>(dy), M, N, N, dyq.q, dyq.s, dyT.q, dyT.s, st);
    if (e != cudaSuccess) return cuda_result(e, "mxq_linear_bwd_dx_wq quant launch");
    return dense_gemm(dyq, wT, M, K, N, dx, K, st);
}

size_t mxq_qat_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int quantize_input) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    // W4A4: both operands as E4M3 codes + scales; W4A16: Q(W) in bf16
    return quantize_input ? operand_bytes(M, K) + operand_bytes(N, K)
                          : round256(2 * static_cast<size_t>(N) * static_cast<size_t>(K));
}

mxq_status mxq_qat_linear_fwd(const void *x, const void *w, const void *bias, int64_t M, int64_t N, int64_t K,
                              int quantize_input, float scale_factor, void *y, void *workspace, size_t ws_bytes,
                              mxq_stream_t stream) {
    if (!x || !w || !y) return fail(MXQ_ERR_INVALID_ARG, "null tensor pointer");
    if (!al16(x) || !al16(w) || !al16(y) || (bias && !al16(bias)) || (workspace && !al16(workspace)))
        return fail(MXQ_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!(scale_factor > 0.0f) || !(scale_factor <= 3.402823466e38f))
        return fail(MXQ_ERR_INVALID_ARG, "scale_factor must be finite and > 0");
    if (M <= 0 || N <= 0 || K <= 0 || M % 32 || N % 32 || K % 32)
        return fail(MXQ_ERR_INVALID_ARG, "M, N, K must be positive multiples of 32 (got %lld, %lld, %lld)",
                    (long long)M, (long long)N, (long long)K);
    if (M > (1ll << 31) || N > (1ll << 31) || K > (1ll << 31))
        return fail(MXQ_ERR_UNSUPPORTED, "dimension above 2^31");
    const size_t need = mxq_qat_linear_workspace_bytes(M, N, K, quantize_input);
    if (!workspace || ws_bytes < need)
        return fail(MXQ_ERR_INVALID_ARG, "workspace too small: need %zu bytes, got %zu", need,
                    workspace ? ws_bytes : 0);
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    if (!quantize_input) {
        // W4A16: Q(W) in bf16 (exact), then the bf16 tensor-core product with x
        uint16_t *qw = reinterpret_cast<uint16_t *>(wp);
        cudaError_t e = mxq::launch_qdq_mxfp4_bf16(static_cast<const uint16_t *>(w), qw, N, K, scale_factor, st);
        if (e != cudaSuccess) return cuda_result(e, "mxq_qat_linear_fwd quant launch");
        mxq::GemmProblem g{};
        g.mode = mxq::kDense;
        g.kind = mxq::kBF16;
        g.a = static_cast<const uint8_t *>(x); g.a_rows = M; g.a_k = K;
        g.b = reinterpret_cast<const uint8_t *>(qw); g.b_rows = N; g.b_k = K;
        g.c = y; g.M = M; g.N = N; g.ldc = N; g.K = K;
        g.bias = bias;
        return cuda_result(mxq::launch_gemm(g, st), "mxq_qat_linear_fwd gemm launch");
    }
    const Operand xq = carve(wp, M, K), wq = carve(wp, N, K);
    // MXFP4 quant-dequant of both operands, held exactly as E4M3 codes under
    // the MXFP4 E8M0 scales, then the block-scaled product plus bias
    cudaError_t e = mxq::launch_quant_rows(x, false, 2, M, K, K, xq.q, xq.s, st, scale_factor);
    if (e == cudaSuccess) e = mxq::launch_quant_rows(w, false, 2, N, K, K, wq.q, wq.s, st, scale_factor);
    if (e != cudaSuccess) return cuda_result(e, "mxq_qat_linear_fwd quant launch");
    return dense_gemm(xq, wq, M, N, K, y, N, st, bias);
}

size_t mxq_qat_grouped_fwd_workspace_bytes(int64_t T, int E, int64_t N, int64_t K, int quantize_input) {
    if (T < 0 || E <= 0 || N <= 0 || K <= 0) return 0;
    const int64_t wrows = static_cast<int64_t>(E) * N;
    return quantize_input ? (T > 0 ? operand_bytes(T, K) : 0) + operand_bytes(wrows, K)
                          : round256(2 * static_cast<size_t>(wrows) * static_cast<size_t>(K));
}

mxq_status mxq_qat_grouped_fwd(const void *x, const void *w, const int64_t *d_offsets, int E, int64_t T, int64_t N,
                               int64_t K, int quantize_input, float scale_factor, void *y, void *workspace,
                               size_t ws_bytes, mxq_stream_t stream) {
    if (E < 1 || E > 4096) return fail(MXQ_ERR_INVALID_ARG, "E must be in [1, 4096]");
    if (T < 0 || N <= 0 || K <= 0 || N % 128 || K % 32)
        return fail(MXQ_ERR_INVALID_ARG, "T >= 0, N a positive multiple of 128, K of 32 (got %lld, %lld, %lld)",
                    (long long)T, (long long)N, (long long)K);
    if (!(scale_factor > 0.0f) || !(scale_factor <= 3.402823466e38f))
        return fail(MXQ_ERR_INVALID_ARG, "scale_factor must be finite and > 0");
    if (K > (1ll << 31) || T > (1ll << 31) || static_cast<int64_t>(E) * N > (1ll << 31))
        return fail(MXQ_ERR_UNSUPPORTED, "dimension above 2^31");
    if (!w || !al16(w) || (T > 0 && (!x || !y || !al16(x) || !al16(y))))
        return fail(MXQ_ERR_INVALID_ARG, "tensor pointers must be non-null and 16-byte aligned");
    if (!d_offsets || (reinterpret_cast<uintptr_t>(d_offsets) & 7))
        return fail(MXQ_ERR_INVALID_ARG, "d_offsets must be a non-null 8-byte aligned device pointer");
    const size_t need = mxq_qat_grouped_fwd_workspace_bytes(T, E, N, K, quantize_input);
    if (!workspace || !al16(workspace) || ws_bytes < need)
        return fail(MXQ_ERR_INVALID_ARG, "workspace too small or unaligned: need %zu bytes, got %zu", need,
                    workspace ? ws_bytes : 0);
    if (T == 0) return ok();
    mxq_status s = check_arch();
    if (s != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t wrows = static_cast<int64_t>(E) * N;
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    mxq::GemmProblem g{};
    g.mode = mxq::kGroupedRows;
    g.offsets = d_offsets; g.E = E; g.T = T;
    g.M = T; g.N = N; g.ldc = N; g.K = K;
    g.a_rows = T; g.a_k = K;
    g.b_rows = wrows; g.b_k = K;
    g.b_row_per_expert = N; g.b_k_per_expert = 0;
    g.c = y;
    if (!quantize_input) {
        // W4A16: Q(W_e) in bf16 (exact), then the bf16 grouped tensor-core product
        uint16_t *qw = reinterpret_cast<uint16_t *>(wp);
        cudaError_t e = mxq::launch_qdq_mxfp4_bf16(static_cast<const uint16_t *>(w), qw, wrows, K, scale_factor, st);
        if (e != cudaSuccess) return cuda_result(e, "mxq_qat_grouped_fwd quant launch");
        g.kind = mxq::kBF16;
        g.a = static_cast<const uint8_t *>(x);
        g.b = reinterpret_cast<const uint8_t *>(qw);
        return cuda_result(mxq::launch_gemm(g, st), "mxq_qat_grouped_fwd gemm launch");
    }
    // W4A4: both operands' MXFP4 quant-dequant held exactly as E4M3 codes under
    // their E8M0 scales (rows of x are independent, so one row quant of all T
    // rows serves every group), then the block-scaled grouped product
    const Operand xq = carve(wp, T, K), wq = carve(wp, wrows, K);
    cudaError_t e = mxq::launch_quant_rows(x, false, 2, T, K, K, xq.q, xq.s, st, scale_factor);
    if (e == cudaSuccess) e = mxq::launch_quant_rows(w, false, 2, wrows, K, K, wq.q, wq.s, st, scale_factor);
    if (e != cudaSuccess) return cuda_result(e, "mxq_qat_grouped_fwd quant launch");
    g.kind = mxq::kMXF8;
    g.a = xq.q; g.sa = xq.s;
    g.b = wq.q; g.sb = wq.s;
    return cuda_result(mxq::launch_gemm(g, st), "mxq_qat_grouped_fwd gemm launch");
}


// ---- grouped (MoE expert) linear layer, SAVE vs RECOMPUTE ----
size_t mxq_grouped_linear_ctx_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    if (T <= 0 || E <= 0 || N <= 0 || K <= 0) return 0;
    return g_ctx_bytes(T, E, N, K, mode);
}
size_t mxq_grouped_linear_saved_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    if (T <= 0 || E <= 0 || N <= 0 || K <= 0) return 0;
    return g_saved_bytes(T, E, N, K, mode);
}
size_t mxq_grouped_linear_workspace_bytes(int64_t T, int E, int64_t N, int64_t K, mxq_mode mode) {
    if (T <= 0 || E <= 0 || N <= 0 || K <= 0) return 0;
    size_t w = g_ws_fwd(T, E, N, K);
    if (g_ws_dx(T, E, N, K, mode) > w) w = g_ws_dx(T, E, N, K, mode);
    if (g_ws_dw(T, E, N, K, mode) > w) w = g_ws_dw(T, E, N, K, mode);
    return w;
}

mxq_status mxq_grouped_linear_fwd(const void *x, const void *w, const int64_t *d_offsets, int E, int64_t T, int64_t N,
                                  int64_t K, mxq_mode mode, void *ctx, void *y, void *workspace, size_t ws_bytes,
                                  mxq_stream_t stream) {
    mxq_status s = check_grouped_linear(x, w, d_offsets, E, T, N, K, mode, ctx, y, workspace, ws_bytes,
                                        g_ws_fwd(T, E, N, K));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t tp = mxq_grouped_padded_rows(T, E), wrows = static_cast<int64_t>(E) * N;
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const Operand xq = carve_prow(wp, T, tp, K), wq = carve(wp, wrows, K);
    cudaError_t e;
    int64_t a_pad = 0;
    if (mode == MXQ_SAVE_QUANT) {
        // X: row quant (padded row scales) and per-group column quant from one
        // read; W: row quant and column quant along E*N from one read
        uint8_t *cp = static_cast<uint8_t *>(ctx);
        const Operand xT = carve(cp, K, tp);
        (void)carve(cp, N, tp);  // gcolT(dY), written by bwd_dx
        const Operand wT = carve(cp, K, wrows);
        e = mxq::launch_quant_cols_grouped(static_cast<const uint16_t *>(x), T, K, d_offsets, E, tp, xq.q, xq.s, xT.q,
                                           xT.s, st, true);
        if (e == cudaSuccess)
            e = mxq::launch_quant_cols(static_cast<const uint16_t *>(w), wrows, K, K, wq.q, wq.s, wT.q, wT.s, st);
        a_pad = tp;
    } else {
        e = mxq::launch_quant_rows(x, false, 0, T, K, K, xq.q, xq.s, st);
        if (e == cudaSuccess) e = mxq::launch_quant_rows(w, false, 0, wrows, K, K, wq.q, wq.s, st);
    }
    if (e != cudaSuccess) return cuda_result(e, "mxq_grouped_linear_fwd quant launch");
    const mxq::GemmProblem g = grouped_problem(MXQ_GG_FWD, xq.q, xq.s, wq.q, wq.s, d_offsets, E, T, N, K, a_pad, y);
    return cuda_result(mxq::launch_gemm(g, st), "mxq_grouped_linear_fwd gemm launch");
}

mxq_status mxq_grouped_linear_bwd_dx(const void *dy, const void *w, const int64_t *d_offsets, int E, int64_t T,
                                     int64_t N, int64_t K, mxq_mode mode, void *ctx, void *dx, void *workspace,
                                     size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_grouped_linear(dy, w, d_offsets, E, T, N, K, mode, ctx, dx, workspace, ws_bytes,
                                        g_ws_dx(T, E, N, K, mode));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t tp = mxq_grouped_padded_rows(T, E), wrows = static_cast<int64_t>(E) * N;
    uint8_t *cp = static_cast<uint8_t *>(ctx);
    if (mode == MXQ_SAVE_QUANT) (void)carve(cp, K, tp);
    const Operand dyT = carve(cp, N, tp);
    Operand wT{};
    if (mode == MXQ_SAVE_QUANT) wT = carve(cp, K, wrows);
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const Operand dyq = carve_prow(wp, T, tp, N);
    // dY: row quant (padded row scales, this call's A) and per-group column
    // quant (bwd_dw's A, kept in ctx) from one read
    cudaError_t e = mxq::launch_quant_cols_grouped(static_cast<const uint16_t *>(dy), T, N, d_offsets, E, tp, dyq.q,
                                                   dyq.s, dyT.q, dyT.s, st, true);
    if (e == cudaSuccess && mode == MXQ_RECOMPUTE) {
        wT = carve(wp, K, wrows);
        e = mxq::launch_quant_cols(static_cast<const uint16_t *>(w), wrows, K, K, nullptr, nullptr, wT.q, wT.s, st);
    }
    if (e != cudaSuccess) return cuda_result(e, "mxq_grouped_linear_bwd_dx quant launch");
    const mxq::GemmProblem g = grouped_problem(MXQ_GG_DX, dyq.q, dyq.s, wT.q, wT.s, d_offsets, E, T, N, K, tp, dx);
    return cuda_result(mxq::launch_gemm(g, st), "mxq_grouped_linear_bwd_dx gemm launch");
}

mxq_status mxq_grouped_linear_bwd_dw(const void *dy, const void *x, const int64_t *d_offsets, int E, int64_t T,
                                     int64_t N, int64_t K, mxq_mode mode, void *ctx, void *dw, void *workspace,
                                     size_t ws_bytes, mxq_stream_t stream) {
    mxq_status s = check_grouped_linear(dy, x, d_offsets, E, T, N, K, mode, ctx, dw, workspace, ws_bytes,
                                        g_ws_dw(T, E, N, K, mode));
    if (s != MXQ_OK) return s;
    if ((s = check_arch()) != MXQ_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t tp = mxq_grouped_padded_rows(T, E);
    uint8_t *cp = static_cast<uint8_t *>(ctx);
    Operand xT{};
    if (mode == MXQ_SAVE_QUANT) xT = carve(cp, K, tp);
    const Operand dyT = carve(cp, N, tp);
    if (mode == MXQ_RECOMPUTE) {
        uint8_t *wp = static_cast<uint8_t *>(workspace);
        xT = carve(wp, K, tp);
        const cudaError_t e = mxq::launch_quant_cols_grouped(static_cast<const uint16_t *>(x), T, K, d_offsets, E, tp,
                                                             nullptr, nullptr, xT.q, xT.s, st, false);
        if (e != cudaSuccess) return cuda_result(e, "mxq_grouped_linear_bwd_dw quant launch");
    }
    const mxq::GemmProblem g = grouped_problem(MXQ_GG_DW, dyT.q, dyT.s, xT.q, xT.s, d_offsets, E, T, N, K, tp, dw);
    return cuda_result(mxq::launch_gemm(g, st), "mxq_grouped_linear_bwd_dw gemm launch");
}

}  // extern "C"
