// Block encoder for k <= 8 [FibQuant §2.3, encoder]: nu = ||x||, u = Pi x / nu, d/k blocks of
// size k, nearest codeword of each block, fixed-address bit packing.
//
// Portable CUDA-core form: one thread per vector, the codebook and the rotation staged in
// shared memory (every thread of a warp reads the same rotation or codeword entry at the same
// time, which the shared-memory crossbar broadcasts), the vector held in registers.
#include <math.h>

#include "fq_bits.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 128;

template <int D>
__device__ __forceinline__ void load_row_f32(const __half *__restrict__ x, int64_t r, float (&xr)[D]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(x + r * D);
#pragma unroll
    for (int q = 0; q < D / 8; ++q) {
        uint4 v = __ldg(src + q);
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            float2 f = __half22float2(h[t]);
            xr[8 * q + 2 * t] = f.x;
            xr[8 * q + 2 * t + 1] = f.y;
        }
    }
}

template <int D, int K>
__global__ void __launch_bounds__(kThreads)
encode_blocks_simple(const __half *__restrict__ x, int64_t M, RowMap map,
                     const float *__restrict__ Pi, const float *__restrict__ C, int N, int B,
                     float *__restrict__ nu_out, uint32_t *__restrict__ codes,
                     uint32_t *__restrict__ flags) {
    extern __shared__ float smem[];
    float *Cs = smem;            // [N x K]
    float *Ps = smem + N * K;    // [D x D]
    for (int i = threadIdx.x; i < N * K; i += blockDim.x) Cs[i] = C[i];
    for (int i = threadIdx.x; i < D * D; i += blockDim.x) Ps[i] = Pi[i];
    __syncthreads();

    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= M) return;
    constexpr int NB = D / K;
    const int R = NB * B;

    float xr[D];
    load_row_f32<D>(x, r, xr);
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < D; ++j) ss = fmaf(xr[j], xr[j], ss);
    const int64_t orow = map(r);
    BitWriter wr(codes, orow * (int64_t)R);
    // fp16 inputs are bounded by 65504, so ss is finite unless an element is Inf or NaN.
    if (!isfinite(ss)) {
        atomicOr(flags, (uint32_t)FQ_FLAG_NONFINITE);
        nu_out[orow] = 0.f;
        for (int b = 0; b < NB; ++b) wr.put(0u, B);
        wr.flush();
        return;
    }
    const float nu = sqrtf(ss);
    nu_out[orow] = nu;
    const float inv = nu > 0.f ? 1.0f / nu : 0.f;

    for (int b = 0; b < NB; ++b) {
        float u[K];
#pragma unroll
        for (int t = 0; t < K; ++t) {
            const float *prow = Ps + (b * K + t) * D;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < D; ++j) acc = fmaf(prow[j], xr[j], acc);
            u[t] = acc * inv;
        }
        float best = INFINITY;
        int bi = 0;
        for (int n = 0; n < N; ++n) {
            const float *c = Cs + n * K;
            float dd = 0.f;
#pragma unroll
            for (int t = 0; t < K; ++t) {
                float e = u[t] - c[t];
                dd = fmaf(e, e, dd);
            }
            if (dd < best) {
                best = dd;
                bi = n;
            }
        }
        wr.put(nu > 0.f ? (uint32_t)bi : 0u, B);
    }
    wr.flush();
}

template <int D, int K>
size_t smem_bytes(const fq_ctx *ctx) {
    return sizeof(float) * ((size_t)ctx->N * K + (size_t)D * D);
}

template <int D, int K>
cudaError_t launch_dk(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                      uint32_t *codes, cudaStream_t s) {
    const int64_t grid = (M + kThreads - 1) / kThreads;
    encode_blocks_simple<D, K><<<(unsigned)grid, kThreads, smem_bytes<D, K>(ctx), s>>>(
        x, M, map, ctx->Pi, ctx->C, ctx->N, ctx->B, nu, codes, ctx->flags);
    return cudaGetLastError();
}

template <int D, int K>
cudaError_t prep_dk(const fq_ctx *ctx) {
    return cudaFuncSetAttribute(encode_blocks_simple<D, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<D, K>(ctx));
}

}  // namespace

cudaError_t launch_encode_blocks(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map,
                                 float *nu, uint32_t *codes, cudaStream_t s) {
#define CALL(D, K) launch_dk<D, K>(ctx, x, M, map, nu, codes, s)
    if (ctx->d == 64) {
        if (ctx->k == 1) return CALL(64, 1);
        if (ctx->k == 2) return CALL(64, 2);
        if (ctx->k == 4) return CALL(64, 4);
        if (ctx->k == 8) return CALL(64, 8);
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

cudaError_t prepare_encode_blocks(const fq_ctx *ctx) {
#define CALL(D, K) prep_dk<D, K>(ctx)
    if (ctx->d == 64) {
        if (ctx->k == 1) return CALL(64, 1);
        if (ctx->k == 2) return CALL(64, 2);
        if (ctx->k == 4) return CALL(64, 4);
        if (ctx->k == 8) return CALL(64, 8);
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
