/*
 * The C ABI used from plain C, with no Python or torch in the process: the
 * caller allocates device memory with the CUDA runtime, quantizes X and W
 * along K with mxq_quantize, multiplies them with mxq_gemm and checks the
 * result against the exact product.
 *
 * Operands take values in {-1, 0, 1} with at least one nonzero per 32-block,
 * so every block's scale exponent is floor(log2 1) - 8 = -8, every code is
 * exact (|x| * 2^8 = 256 <= 448), and every dot product over K = 64 is an
 * integer of magnitude <= 64, exact in fp32 and in bf16: the GEMM output must
 * equal the integer product bit for bit.
 *
 * Prints "ok" and returns 0 on success; prints the first mismatch or the
 * failing call's status and message and returns 1 otherwise.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mxq.h"

enum { M = 256, N = 384, K = 64 };

static uint16_t bf16_of(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16); /* exact for the small integers used here */
}

static float float_of_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* a deterministic value in {-1, 0, 1}; element 0 of every 32-block is 1 */
static int val(uint32_t seed, int r, int c) {
    if (c % 32 == 0) return 1;
    uint32_t h = seed ^ (uint32_t)(r * 7919 + c * 104729);
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    h ^= h >> 15;
    return (int)(h % 3u) - 1;
}

#define CK(call)                                                                              \
    do {                                                                                      \
        cudaError_t e_ = (call);                                                              \
        if (e_ != cudaSuccess) {                                                              \
            printf("CUDA error %d at line %d\n", (int)e_, __LINE__);                          \
            return 1;                                                                         \
        }                                                                                     \
    } while (0)
#define MK(call)                                                                              \
    do {                                                                                      \
        mxq_status s_ = (call);                                                               \
        if (s_ != MXQ_OK) {                                                                   \
            printf("mxq status %d at line %d: %s\n", (int)s_, __LINE__, mxq_last_error_string()); \
            return 1;                                                                         \
        }                                                                                     \
    } while (0)

int main(void) {
    static uint16_t hx[M * K], hw[N * K], hy[M * N];
    static int ix[M * K], iw[N * K];
    for (int r = 0; r < M; r++)
        for (int c = 0; c < K; c++) {
            ix[r * K + c] = val(1u, r, c);
            hx[r * K + c] = bf16_of((float)ix[r * K + c]);
        }
    for (int r = 0; r < N; r++)
        for (int c = 0; c < K; c++) {
            iw[r * K + c] = val(2u, r, c);
            hw[r * K + c] = bf16_of((float)iw[r * K + c]);
        }

    void *dx, *dw, *dy, *qx, *sx, *qw, *sw;
    const size_t sxb = mxq_scale_bytes(M, K / 32), swb = mxq_scale_bytes(N, K / 32);
    CK(cudaMalloc(&dx, sizeof hx));
    CK(cudaMalloc(&dw, sizeof hw));
    CK(cudaMalloc(&dy, sizeof hy));
    CK(cudaMalloc(&qx, (size_t)M * K));
    CK(cudaMalloc(&qw, (size_t)N * K));
    CK(cudaMalloc(&sx, sxb));
    CK(cudaMalloc(&sw, swb));
    CK(cudaMemcpy(dx, hx, sizeof hx, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dw, hw, sizeof hw, cudaMemcpyHostToDevice));

    MK(mxq_quantize(dx, MXQ_BF16, M, K, K, -1, MXQ_E4M3, 0, qx, sx, NULL, NULL, NULL));
    MK(mxq_quantize(dw, MXQ_BF16, N, K, K, -1, MXQ_E4M3, 0, qw, sw, NULL, NULL, NULL));
    MK(mxq_gemm((const uint8_t *)qx, (const uint8_t *)sx, (const uint8_t *)qw, (const uint8_t *)sw, M, N, K, dy, N,
                NULL));
    CK(cudaDeviceSynchronize());
    uint32_t word = 0;
    MK(mxq_poll_device_error(&word));
    CK(cudaMemcpy(hy, dy, sizeof hy, cudaMemcpyDeviceToHost));

    for (int r = 0; r < M; r++)
        for (int c = 0; c < N; c++) {
            int ref = 0;
            for (int k = 0; k < K; k++) ref += ix[r * K + k] * iw[c * K + k];
            const float got = float_of_bf16(hy[r * N + c]);
            if (got != (float)ref) {
                printf("mismatch at (%d, %d): got %g, expected %d\n", r, c, got, ref);
                return 1;
            }
        }
    cudaFree(dx);
    cudaFree(dw);
    cudaFree(dy);
    cudaFree(qx);
    cudaFree(qw);
    cudaFree(sx);
    cudaFree(sw);
    printf("ok\n");
    return 0;
}
