// Centroid sums for Lloyd refinement of the codebook [FibQuant §2.2, refinement: Lloyd iterations
// on draws of the block source minimise the MSE of the finite codebook]. The assignment step of an
// iteration is the encoder itself (the nearest codeword of every block of every training row); this
// kernel forms, for every codeword n,
//   sums[n] = sum of the blocks u_b assigned to n,   counts[n] = their number,
// with u = Pi x / nu recomputed from the encoded rows. Rows whose norm is 0 (zero or non-finite
// input) carry no direction and are skipped.
//
// One thread per row (grid-stride). The rotation is staged in shared memory and read as broadcasts
// (every lane of a warp needs the same element at the same step). When the codebook's sums fit, each
// CTA accumulates into a shared-memory copy and adds it to the caller's fp64 totals with one atomic
// per entry; otherwise (k = d) the blocks go straight to the fp64 totals.
#include "fq_bits.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 256;

template <int D, int K, bool PRIV>
__global__ void __launch_bounds__(kThreads)
centroid_sums(const __half *__restrict__ x, int64_t M, const float *__restrict__ nu,
              const uint32_t *__restrict__ codes, const float *__restrict__ Pi, int N, int B,
              double *__restrict__ sums, double *__restrict__ counts) {
    extern __shared__ float smem[];
    float *Ps = smem;                        // [D x D]
    float *ps = Ps + D * D;                  // [N x K] private sums (PRIV)
    uint32_t *pc = reinterpret_cast<uint32_t *>(ps + (PRIV ? N * K : 0));   // [N] private counts
    for (int i = threadIdx.x; i < D * D; i += blockDim.x) Ps[i] = Pi[i];
    if constexpr (PRIV) {
        for (int i = threadIdx.x; i < N * K; i += blockDim.x) ps[i] = 0.f;
        for (int i = threadIdx.x; i < N; i += blockDim.x) pc[i] = 0u;
    }
    __syncthreads();

    constexpr int NB = D / K;
    const int R = NB * B;
    for (int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; m < M; m += (int64_t)gridDim.x * blockDim.x) {
        const float v = __ldg(nu + m);
        if (!(v > 0.f) || !isfinite(v)) continue;
        const float inv = 1.0f / v;
        __half2 xr[D / 2];
        const uint4 *src = reinterpret_cast<const uint4 *>(x + m * D);
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
            const uint4 w = __ldg(src + q);
            const __half2 *h = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
            for (int t = 0; t < 4; ++t) xr[4 * q + t] = h[t];
        }
        BitReader rd(codes, m * (int64_t)R);
        for (int b = 0; b < NB; ++b) {
            const uint32_t n = rd.get(B);
            float u[K];
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const float *prow = Ps + (b * K + j) * D;
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < D / 2; ++i) {
                    const float2 f = __half22float2(xr[i]);
                    acc = fmaf(prow[2 * i], f.x, acc);
                    acc = fmaf(prow[2 * i + 1], f.y, acc);
                }
                u[j] = acc * inv;
            }
            if constexpr (PRIV) {
#pragma unroll
                for (int j = 0; j < K; ++j) atomicAdd(ps + n * K + j, u[j]);
                atomicAdd(pc + n, 1u);
            } else {
#pragma unroll
                for (int j = 0; j < K; ++j) atomicAdd(sums + (size_t)n * K + j, (double)u[j]);
                atomicAdd(counts + n, 1.0);
            }
        }
    }
    if constexpr (PRIV) {
        __syncthreads();
        for (int i = threadIdx.x; i < N * K; i += blockDim.x)
            if (ps[i] != 0.f) atomicAdd(sums + i, (double)ps[i]);
        for (int i = threadIdx.x; i < N; i += blockDim.x)
            if (pc[i]) atomicAdd(counts + i, (double)pc[i]);
    }
}

template <int D, int K>
cudaError_t launch_dk(const fq_ctx *ctx, const __half *x, int64_t M, const float *nu, const uint32_t *codes,
                      double *sums, double *counts, cudaStream_t s) {
    const size_t base = sizeof(float) * (size_t)D * D;
    const size_t priv = sizeof(float) * (size_t)ctx->N * (K + 1);
    const bool use_priv = K < D && base + priv <= (size_t)ctx->smem_optin;
    int64_t grid = (M + kThreads - 1) / kThreads;
    if (grid > 2 * (int64_t)ctx->num_sms) grid = 2 * (int64_t)ctx->num_sms;
    if (grid < 1) grid = 1;
    if (use_priv) {
        if constexpr (K < D) {
            cudaError_t e = cudaFuncSetAttribute(centroid_sums<D, K, true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(base + priv));
            if (e != cudaSuccess) return e;
            centroid_sums<D, K, true><<<(unsigned)grid, kThreads, base + priv, s>>>(x, M, nu, codes, ctx->Pi, ctx->N,
                                                                                  ctx->B, sums, counts);
        }
    } else {
        cudaError_t e = cudaFuncSetAttribute(centroid_sums<D, K, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)base);
        if (e != cudaSuccess) return e;
        centroid_sums<D, K, false><<<(unsigned)grid, kThreads, base, s>>>(x, M, nu, codes, ctx->Pi, ctx->N, ctx->B,
                                                                        sums, counts);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_centroid_sums(const fq_ctx *ctx, const __half *x, int64_t M, const float *nu,
                                 const uint32_t *codes, double *sums, double *counts, cudaStream_t s) {
#define CALL(D, K) launch_dk<D, K>(ctx, x, M, nu, codes, sums, counts, s)
    if (ctx->d == 64) {
        if (ctx->k == 1) return CALL(64, 1);
        if (ctx->k == 2) return CALL(64, 2);
        if (ctx->k == 4) return CALL(64, 4);
        if (ctx->k == 8) return CALL(64, 8);
        if (ctx->k == 64) return CALL(64, 64);
    } else if (ctx->d == 96) {
        if (ctx->k == 1) return CALL(96, 1);
        if (ctx->k == 2) return CALL(96, 2);
        if (ctx->k == 3) return CALL(96, 3);
        if (ctx->k == 4) return CALL(96, 4);
        if (ctx->k == 8) return CALL(96, 8);
    } else if (ctx->d == 128) {
        if (ctx->k == 1) return CALL(128, 1);
        if (ctx->k == 2) return CALL(128, 2);
        if (ctx->k == 4) return CALL(128, 4);
        if (ctx->k == 8) return CALL(128, 8);
    }
#undef CALL
    return cudaErrorInvalidValue;
}

}  // namespace fq
