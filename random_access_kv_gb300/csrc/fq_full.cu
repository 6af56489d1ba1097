// Full-vector code k = d [FibQuant §4.2: one index per vector, all bits spent on angular
// packing; §3.3: sub-one-bit rates such as b = 12/64 = 0.1875].
//
// With one block the nearest codeword to u = Pi x / nu is
//   argmin_n |u - c_n|^2 = argmin_n  nu |c_n|^2 - 2 x . (Pi^T c_n)      (nu > 0)
// so the rotation folds into a rotated codebook Crot = C Pi (row n = Pi^T c_n, built on the host
// in double precision) and the search becomes a contraction of x with Crot plus an argmin.
// Decoding is x_hat = nu Pi^T c_i = nu Crot[i].
//
// Portable CUDA-core form: one thread per vector, Crot streamed through shared memory in
// chunks that every thread of the block scans (broadcast reads).
#include <math.h>

#include "fq_bits.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 64;   // codewords per shared-memory chunk

template <int D>
__global__ void __launch_bounds__(kThreads)
encode_full_simple(const __half *__restrict__ x, int64_t M, RowMap map,
                   const float *__restrict__ Crot, const float *__restrict__ cc, int N, int B,
                   float *__restrict__ nu_out, uint32_t *__restrict__ codes,
                   uint32_t *__restrict__ flags) {
    __shared__ float Cs[kChunk * D];
    __shared__ float hs[kChunk];
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = r < M;
    float xr[D];
    float ss = 0.f;
    if (live) {
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
#pragma unroll
        for (int j = 0; j < D; ++j) ss = fmaf(xr[j], xr[j], ss);
    } else {
#pragma unroll
        for (int j = 0; j < D; ++j) xr[j] = 0.f;
    }
    const bool finite = isfinite(ss);
    const float nu = finite ? sqrtf(ss) : 0.f;
    float best = INFINITY;
    int bi = 0;
    for (int n0 = 0; n0 < N; n0 += kChunk) {
        __syncthreads();
        for (int i = threadIdx.x; i < kChunk * D; i += blockDim.x) Cs[i] = __ldg(Crot + (size_t)n0 * D + i);
        if (threadIdx.x < kChunk) hs[threadIdx.x] = __ldg(cc + n0 + threadIdx.x);
        __syncthreads();
        for (int n = 0; n < kChunk; ++n) {
            const float *c = Cs + n * D;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < D; ++j) dot = fmaf(xr[j], c[j], dot);
            const float score = fmaf(-2.f, dot, nu * hs[n]);
            if (score < best) {
                best = score;
                bi = n0 + n;
            }
        }
    }
    if (!live) return;
    const int64_t orow = map(r);
    if (!finite) atomicOr(flags, (uint32_t)FQ_FLAG_NONFINITE);
    nu_out[orow] = nu;
    BitWriter wr(codes, orow * (int64_t)B);
    wr.put(nu > 0.f ? (uint32_t)bi : 0u, B);
    wr.flush();
}

// x_hat = nu C_rot[i] for k = d. One warp per 32 output rows: each lane reads its row's index and
// norm, then the warp writes the rows one after another, lane l covering columns 2l and 2l + 1, so
// that every table read (256 B) and every row store (128 B fp16) is a single coalesced access.
template <typename OutT>
__global__ void __launch_bounds__(kThreads)
decode_full(const float *__restrict__ nu, const uint32_t *__restrict__ codes, int64_t M,
            const int64_t *__restrict__ idx, int64_t n, const float *__restrict__ Crot, int B,
            OutT *__restrict__ out, uint32_t *__restrict__ flags) {
    constexpr int D = 64;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t tile = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; tile * 32 < n; tile += nwarps) {
        const int64_t j = tile * 32 + lane;
        float s = 0.f;
        uint32_t i = 0;
        if (j < n) {
            const int64_t row = idx ? __ldg(idx + j) : j;
            if (row < 0 || row >= M) {
                atomicOr(flags, (uint32_t)FQ_FLAG_RANGE);
            } else {
                BitReader rd(codes, row * (int64_t)B);
                i = rd.get(B);
                s = __ldg(nu + row);
            }
        }
        const int rows = n - tile * 32 < 32 ? (int)(n - tile * 32) : 32;
#pragma unroll 8
        for (int r = 0; r < 32; ++r) {
            const uint32_t ir = __shfl_sync(0xffffffffu, i, r);
            const float sr = __shfl_sync(0xffffffffu, s, r);
            if (r < rows) {
                const float2 c = __ldg(reinterpret_cast<const float2 *>(Crot + (size_t)ir * D) + lane);
                OutT *dst = out + (tile * 32 + r) * D;
                if constexpr (sizeof(OutT) == 2)
                    reinterpret_cast<__half2 *>(dst)[lane] = __floats2half2_rn(c.x * sr, c.y * sr);
                else
                    reinterpret_cast<float2 *>(dst)[lane] = make_float2(c.x * sr, c.y * sr);
            }
        }
    }
}

}  // namespace

cudaError_t launch_encode_full(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map,
                               float *nu, uint32_t *codes, cudaStream_t s) {
    if (ctx->d != 64) return cudaErrorInvalidValue;
    const int64_t grid = (M + kThreads - 1) / kThreads;
    encode_full_simple<64><<<(unsigned)grid, kThreads, 0, s>>>(x, M, map, ctx->Crot, ctx->cc, ctx->N,
                                                               ctx->B, nu, codes, ctx->flags);
    return cudaGetLastError();
}

cudaError_t launch_decode_full(const fq_ctx *ctx, const float *nu, const uint32_t *codes,
                               int64_t M, const int64_t *idx, int64_t n, void *out,
                               bool out_f32, cudaStream_t s) {
    if (ctx->d != 64) return cudaErrorInvalidValue;
    int64_t grid = ((n + 31) / 32 + kThreads / 32 - 1) / (kThreads / 32);
    if (grid > 8 * (int64_t)ctx->num_sms) grid = 8 * (int64_t)ctx->num_sms;
    if (out_f32)
        decode_full<float><<<(unsigned)grid, kThreads, 0, s>>>(nu, codes, M, idx, n, ctx->Crot, ctx->B, (float *)out,
                                                               ctx->flags);
    else
        decode_full<__half><<<(unsigned)grid, kThreads, 0, s>>>(nu, codes, M, idx, n, ctx->Crot, ctx->B,
                                                                (__half *)out, ctx->flags);
    return cudaGetLastError();
}

cudaError_t prepare_full(const fq_ctx *) { return cudaSuccess; }

}  // namespace fq
