// mxq_noalloc.cu -- the MXFP8 linear-layer forward for callers that cannot
// allocate device memory.
//
// Every other entry point takes its scratch space (here: the row-quantized X
// and W) from memory the caller passes in.  Some callers have no such memory to
// give: a plug-in running inside a host framework that owns the whole device
// memory pool and does not let plug-ins call cudaMalloc, or a service that
// reserves its memory once at start-up and must not allocate afterwards
// (cudaMalloc can stall the device and can fail once the pool is reserved).
// mxq_linear_fwd_noalloc serves them with scratch that lives inside the
// library: a fixed device array, MXQ_NOALLOC_SCRATCH_BYTES large, that every
// GPU which loads the library holds until the process exits.
//
// The array's name is only a host-side stand-in for host code; its device
// address is looked up once per device with cudaGetSymbolAddress (on the
// first call made with that device current) and passed to the kernels.  The
// kept address belongs to the device's primary context: a cudaDeviceReset
// makes it stale (the header tells callers not to use this entry point on
// that device afterwards).
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

constexpr size_t kScratchBytes = MXQ_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
uint8_t *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_noalloc_scratch on the current device.
cudaError_t scratch_address(int dev, uint8_t **out) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
// codes + swz scales of a K-major operand [rows x k], each padded to 256 bytes
inline size_t operand_bytes(int64_t rows, int64_t k) {
    const size_t scales = static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((k / 32 + 3) / 4 * 4);
    return round256(static_cast<size_t>(rows) * static_cast<size_t>(k)) + round256(scales);
}

}  // namespace

extern "C" mxq_status mxq_linear_fwd_noalloc(const void *x, const void *w, int64_t M, int64_t N, int64_t K, void *y,
                                             mxq_stream_t stream) {
    if (!x || !w || !y) return mxq::api_fail(MXQ_ERR_INVALID_ARG, "null tensor pointer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return mxq::api_fail(MXQ_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (M <= 0 || N <= 0 || K <= 0 || M % 32 || N % 32 || K % 32)
        return mxq::api_fail(MXQ_ERR_INVALID_ARG, "M, N, K must be positive multiples of 32");
    if (M > (1ll << 31) || N > (1ll << 31) || K > (1ll << 31))
        return mxq::api_fail(MXQ_ERR_INVALID_ARG, "dimension above 2^31");
    const size_t a_bytes = operand_bytes(M, K), need = a_bytes + operand_bytes(N, K);
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "mxq_linear_fwd_noalloc: the quantized operands need %zu bytes but the built-in scratch holds %zu "
                 "(MXQ_NOALLOC_SCRATCH_BYTES); use mxq_linear_fwd with a workspace for this size",
                 need, kScratchBytes);
        return mxq::api_fail(MXQ_ERR_INVALID_ARG, msg);
    }
    mxq_status s = mxq::api_check_arch();
    if (s != MXQ_OK) return s;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return mxq::api_cuda_result(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return mxq::api_fail(MXQ_ERR_CUDA, "device index out of range");
    uint8_t *base = nullptr;
    e = scratch_address(dev, &base);
    if (e != cudaSuccess) return mxq::api_cuda_result(e, "cudaGetSymbolAddress of the no-alloc scratch");

    // Scratch layout: [row(X) codes | scales][row(W) codes | scales].  The quant
    // kernels write every byte of these regions (scale padding included), so
    // nothing left over from an earlier call is ever read.
    uint8_t *xq = base, *xs = base + round256(static_cast<size_t>(M) * K);
    uint8_t *wq = base + a_bytes, *ws = wq + round256(static_cast<size_t>(N) * K);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    e = mxq::launch_quant_rows(x, false, 0, M, K, K, xq, xs, st);
    if (e == cudaSuccess) e = mxq::launch_quant_rows(w, false, 0, N, K, K, wq, ws, st);
    if (e != cudaSuccess) return mxq::api_cuda_result(e, "mxq_linear_fwd_noalloc quant launch");
    mxq::GemmProblem g{};
    g.mode = mxq::kDense;
    g.a = xq; g.sa = xs; g.a_rows = M; g.a_k = K;
    g.b = wq; g.sb = ws; g.b_rows = N; g.b_k = K;
    g.c = y; g.M = M; g.N = N; g.ldc = N; g.K = K;
    return mxq::api_cuda_result(mxq::launch_gemm(g, st), "mxq_linear_fwd_noalloc gemm launch");
}
