// Block decoder for k <= 8 [FibQuant §2.3, decoder], full and random-access (gather):
// read the record at its fixed address, unpack the d/k indices, fetch and concatenate the
// codewords, apply Pi^T, scale by nu.
//
// Portable CUDA-core form: one thread per output vector, codebook and rotation in shared
// memory; the rotation row that all threads of a warp need at a given step is the same, so
// its reads are broadcasts.
#include "fq_bits.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 128;

template <int D>
__device__ __forceinline__ void store_row(__half *out, int64_t j, const float (&v)[D], float s) {
    uint4 *dst = reinterpret_cast<uint4 *>(out + j * D);
#pragma unroll
    for (int q = 0; q < D / 8; ++q) {
        uint4 w;
        __half2 *h = reinterpret_cast<__half2 *>(&w);
#pragma unroll
        for (int t = 0; t < 4; ++t) h[t] = __floats2half2_rn(v[8 * q + 2 * t] * s, v[8 * q + 2 * t + 1] * s);
        dst[q] = w;
    }
}

template <int D>
__device__ __forceinline__ void store_row(float *out, int64_t j, const float (&v)[D], float s) {
    float4 *dst = reinterpret_cast<float4 *>(out + j * D);
#pragma unroll
    for (int q = 0; q < D / 4; ++q)
        dst[q] = make_float4(v[4 * q] * s, v[4 * q + 1] * s, v[4 * q + 2] * s, v[4 * q + 3] * s);
}

template <int D, int K, typename OutT>
__global__ void __launch_bounds__(kThreads)
decode_blocks_simple(const float *__restrict__ nu, const uint32_t *__restrict__ codes, int64_t M,
                     const int64_t *__restrict__ idx, int64_t n, const float *__restrict__ Pi,
                     const float *__restrict__ C, int N, int B, OutT *__restrict__ out,
                     uint32_t *__restrict__ flags) {
    extern __shared__ float smem[];
    float *Cs = smem;            // [N x K]
    float *Ps = smem + N * K;    // [D x D]
    for (int i = threadIdx.x; i < N * K; i += blockDim.x) Cs[i] = C[i];
    for (int i = threadIdx.x; i < D * D; i += blockDim.x) Ps[i] = Pi[i];
    __syncthreads();

    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    constexpr int NB = D / K;
    const int R = NB * B;
    const int64_t row = idx ? __ldg(idx + j) : j;
    float acc[D];
#pragma unroll
    for (int q = 0; q < D; ++q) acc[q] = 0.f;
    if (row < 0 || row >= M) {
        atomicOr(flags, (uint32_t)FQ_FLAG_RANGE);
        store_row<D>(out, j, acc, 0.f);
        return;
    }
    BitReader rd(codes, row * (int64_t)R);
    for (int b = 0; b < NB; ++b) {
        const uint32_t i = rd.get(B);
        const float *c = Cs + i * K;
#pragma unroll
        for (int t = 0; t < K; ++t) {
            const float ct = c[t];
            const float *prow = Ps + (b * K + t) * D;
#pragma unroll
            for (int q = 0; q < D; ++q) acc[q] = fmaf(ct, prow[q], acc[q]);
        }
    }
    store_row<D>(out, j, acc, __ldg(nu + row));
}

template <int D, int K>
size_t smem_bytes(const fq_ctx *ctx) {
    return sizeof(float) * ((size_t)ctx->N * K + (size_t)D * D);
}

template <int D, int K>
cudaError_t launch_dk(const fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                      const int64_t *idx, int64_t n, void *out, bool out_f32, cudaStream_t s) {
    const int64_t grid = (n + kThreads - 1) / kThreads;
    if (out_f32)
        decode_blocks_simple<D, K, float><<<(unsigned)grid, kThreads, smem_bytes<D, K>(ctx), s>>>(
            nu, codes, M, idx, n, ctx->Pi, ctx->C, ctx->N, ctx->B, (float *)out, ctx->flags);
    else
        decode_blocks_simple<D, K, __half><<<(unsigned)grid, kThreads, smem_bytes<D, K>(ctx), s>>>(
            nu, codes, M, idx, n, ctx->Pi, ctx->C, ctx->N, ctx->B, (__half *)out, ctx->flags);
    return cudaGetLastError();
}

template <int D, int K>
cudaError_t prep_dk(const fq_ctx *ctx) {
    const int bytes = (int)smem_bytes<D, K>(ctx);
    cudaError_t e = cudaFuncSetAttribute(decode_blocks_simple<D, K, float>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_blocks_simple<D, K, __half>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_decode_blocks(const fq_ctx *ctx, const float *nu, const uint32_t *codes,
                                 int64_t M, const int64_t *idx, int64_t n, void *out,
                                 bool out_f32, cudaStream_t s) {
#define CALL(D, K) launch_dk<D, K>(ctx, nu, codes, M, idx, n, out, out_f32, s)
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

cudaError_t prepare_decode_blocks(const fq_ctx *ctx) {
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
