// Tensor-core full-vector encoder, k = d = 64 [FibQuant §4.2: one index per vector, all bits on
// angular packing; §3.3: sub-one-bit rates, b = log2(N)/64].
//
// With a single block the nearest codeword to u = Pi x / nu is
//     argmin_n |u - c_n|^2 = argmin_n  |c_n|^2 - 2 x.(Pi^T c_n) / nu        (nu > 0),
// a contraction of x with the rotated codebook Crot = C Pi (row n = Pi^T c_n) followed by an
// argmin over n. The contraction runs on the tensor pipe:
//   A = the x tile (fp16, exact), TMA-loaded in the 128-byte swizzle layout;
//   B = -2 * 2^12 * Crot carried as two fp16 halves (hi, lo), streamed in 128-codeword tiles
//       through a 4-stage shared-memory ring by a producer warp (TMA);
//   D = fp32 accumulator in TMEM, 128 lanes x 128 columns per row group.
// Four row groups of 128 threads (one vector per thread) share every codebook tile. After each
// tile a group reads its scores back, s_n = |c_n|^2 + acc_n * 2^-12 / nu, and keeps the running
// minimum: per 16-column chunk a min-tree, and only when a chunk improves on the best so far a
// search for its lowest index holding that value (ties go to the lowest n).
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <vector>

#include "fq_bits.cuh"
#include "fq_internal.h"
#include "fq_sm100.cuh"

namespace fq {

namespace {

using namespace sm100;

constexpr int kD = 64;
constexpr int kRows = 128;            // rows per group tile (= TMEM lanes)
constexpr int kNG = 4;                // row groups per CTA
constexpr int kNT = 128;              // codewords per B tile (MMA N)
constexpr int kStages = 4;
constexpr float kBScale = 4096.f;     // 2^12 on Crot
constexpr int kXBytes = kRows * kD * 2;          // 16 KB
constexpr int kBHalf = kNT * kD * 2;             // 16 KB
constexpr int kMaxN = 4096;

struct FLayout {
    static constexpr int oX = 0;
    static constexpr int oB = oX + kNG * kXBytes;
    static constexpr int oH = oB + kStages * 2 * kBHalf;
    static constexpr int oBar = oH + kMaxN * 4;
    // bars: full[kStages], empty[kStages], xload[kNG], mma[kNG]
    static constexpr int kBars = 2 * kStages + 2 * kNG;
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;
};

struct FullParams {
    int64_t M;
    RowMap map;
    int N, B;
    const float *h;          // [N] |c_n|^2
    float *nu;
    uint32_t *codes;
    uint32_t *flags;
};

__global__ void __launch_bounds__(kNG * 128 + 32, 1)
encode_full_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bhi_map,
               const __grid_constant__ CUtensorMap blo_map, const FullParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + FLayout::oBar);
    uint64_t *full = bars, *empty = bars + kStages, *xload = bars + 2 * kStages, *mmab = bars + 2 * kStages + kNG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + FLayout::oTmem);
    float *hs = reinterpret_cast<float *>(sm + FLayout::oH);

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int64_t ntiles = (p.M + kNG * kRows - 1) / (kNG * kRows);     // CTA tiles of 512 rows
    const int nbt = p.N / kNT;                                            // codebook tiles

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kNG);
        }
        for (int g = 0; g < kNG; ++g) {
            mbar_init(xload + g, 1);
            mbar_init(mmab + g, 1);
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    for (int i = tid; i < p.N; i += blockDim.x) hs[i] = p.h[i];
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kNG * 4) {
        // Producer warp: streams codebook tiles through the ring, for every CTA tile in turn.
        if ((tid & 31) == 0) {
            prefetch_tensormap(&bhi_map);
            prefetch_tensormap(&blo_map);
            uint32_t k = 0;
            bool ok = true;
            for (int64_t ct = blockIdx.x; ct < ntiles && ok; ct += gridDim.x) {
                for (int bt = 0; bt < nbt && ok; ++bt, ++k) {
                    const uint32_t s = k % kStages, round = k / kStages;
                    if (round > 0) ok = mbar_wait(empty + s, (round - 1) & 1);
                    if (!ok) break;
                    uint8_t *dst = sm + FLayout::oB + s * 2 * kBHalf;
                    mbar_arrive_expect_tx(full + s, 2u * kBHalf);
                    tma_load_2d(dst, &bhi_map, 0, bt * kNT, full + s);
                    tma_load_2d(dst + kBHalf, &blo_map, 0, bt * kNT, full + s);
                }
            }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
        }
    } else {
        const int g = warp / 4;
        const int t = tid % 128;
        const int wq = (tid / 32) % 4;
        uint8_t *xt = sm + FLayout::oX + g * kXBytes;
        const uint32_t tmem_acc = tmem_base + (uint32_t)(g * kNT);
        const uint32_t idesc = idesc_f16_f32(128, kNT);
        uint32_t k = 0;            // codebook tiles consumed so far (ring position)
        uint32_t xphase = 0, mphase = 0;
        bool ok = true;
        for (int64_t ct = blockIdx.x; ct < ntiles && ok; ct += gridDim.x) {
            const int64_t row0 = ct * (kNG * kRows) + g * kRows;
            if (t == 0) {
                mbar_arrive_expect_tx(xload + g, (uint32_t)kXBytes);
                tma_load_2d(xt, &xmap, 0, (int)row0, xload + g);
            }
            ok = named_sync_and(1 + g, 128, mbar_wait(xload + g, xphase));
            xphase ^= 1;
            if (!ok) break;
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = *reinterpret_cast<const uint4 *>(xt + t * 128 + ((c ^ (t & 7)) << 4));
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __half22float2(h2[q]);
                    ss = fmaf(f.x, f.x, ss);
                    ss = fmaf(f.y, f.y, ss);
                }
            }
            const bool finite = isfinite(ss);
            const float nu = finite ? sqrtf(ss) : 0.f;
            const float rs = nu > 0.f ? (1.0f / kBScale) / nu : 0.f;
            float best = INFINITY;
            uint32_t bi = 0;
            for (int bt = 0; bt < nbt; ++bt, ++k) {
                const uint32_t s = k % kStages;
                if (t == 0) {
                    // The group's previous epilogue finished reading TMEM (barrier below).
                    ok = mbar_wait(full + s, (k / kStages) & 1);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t xa = smem_addr(xt);
                        const uint32_t bh = smem_addr(sm + FLayout::oB + s * 2 * kBHalf), bl = bh + kBHalf;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
#pragma unroll
                            for (int kk = 0; kk < kD / 16; ++kk)
                                mma_f16(tmem_acc, sdesc_sw128(xa + kk * 32), sdesc_sw128((half ? bl : bh) + kk * 32),
                                        idesc, (half | kk) ? 1u : 0u);
                        }
                        mma_commit(mmab + g);
                        mma_commit(empty + s);
                    }
                }
                ok = named_sync_and(1 + g, 128, ok && mbar_wait(mmab + g, mphase));
                mphase ^= 1;
                if (!ok) break;
                tc_fence_after();
                // Two halves of 64 columns: four 32-column loads in flight per wait.
#pragma unroll
                for (int hh = 0; hh < kNT / 64; ++hh) {
                    uint32_t r[2][32];
                    tmem_ld32_nowait(tmem_acc + ((uint32_t)(32 * wq) << 16) + (uint32_t)(64 * hh), r[0]);
                    tmem_ld32_nowait(tmem_acc + ((uint32_t)(32 * wq) << 16) + (uint32_t)(64 * hh + 32), r[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t *a = &r[c / 2][16 * (c % 2)];
                        const int n0 = bt * kNT + hh * 64 + c * 16;
                        const float4 *h4 = reinterpret_cast<const float4 *>(hs + n0);
                        float sc[16];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 hv = h4[q];
                            sc[4 * q + 0] = fmaf(__uint_as_float(a[4 * q + 0]), rs, hv.x);
                            sc[4 * q + 1] = fmaf(__uint_as_float(a[4 * q + 1]), rs, hv.y);
                            sc[4 * q + 2] = fmaf(__uint_as_float(a[4 * q + 2]), rs, hv.z);
                            sc[4 * q + 3] = fmaf(__uint_as_float(a[4 * q + 3]), rs, hv.w);
                        }
                        const float cmin = min16(sc);
                        if (cmin < best) {
                            best = cmin;
                            uint32_t j = 15;
#pragma unroll
                            for (int q = 15; q >= 0; --q)
                                if (sc[q] == cmin) j = (uint32_t)q;
                            bi = (uint32_t)n0 + j;
                        }
                    }
                }
                tc_fence_before();
                named_sync(1 + g, 128);
            }
            if (!ok) break;
            const int64_t r = row0 + t;
            if (r < p.M) {
                const int64_t orow = p.map(r);
                p.nu[orow] = nu;
                if (!finite) atomicOr(p.flags, (uint32_t)FQ_FLAG_NONFINITE);
                BitWriter wr(p.codes, orow * (int64_t)p.B);
                wr.put(nu > 0.f ? bi : 0u, p.B);
                wr.flush();
            }
        }
        if (!ok && t == 0) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base, 512);
}

bool make_map(CUtensorMap *tm, const void *base, int64_t rows) {
    return encode_rows_tensor_map(tm, base, rows, kD);
}

}  // namespace

bool full_tc_supported(const fq_ctx *ctx) {
    CUtensorMap probe;
    return ctx->k == ctx->d && ctx->d == kD && ctx->N >= kNT && ctx->N <= kMaxN && ctx->N % kNT == 0 &&
           make_map(&probe, ctx->Pi, 128);
}

cudaError_t prepare_full_tc(fq_ctx *ctx) {
    const int N = ctx->N;
    std::vector<float> R((size_t)N * kD);
    cudaError_t e = cudaMemcpy(R.data(), ctx->Crot, R.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    // Row-major fp16 halves of -2 * 2^12 * Crot (TMA applies the swizzle when loading).
    std::vector<uint16_t> hl((size_t)2 * N * kD);
    for (size_t i = 0; i < (size_t)N * kD; ++i) {
        const float v = -2.0f * kBScale * R[i];
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        memcpy(&hl[i], &hi, 2);
        memcpy(&hl[(size_t)N * kD + i], &lo, 2);
    }
    e = cudaMalloc((void **)&ctx->crot_split, hl.size() * 2);
    if (e == cudaSuccess) e = cudaMemcpy(ctx->crot_split, hl.data(), hl.size() * 2, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(encode_full_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, FLayout::kBytes);
}

cudaError_t launch_encode_full_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                  uint32_t *codes, cudaStream_t s) {
    CUtensorMap xm, bh, bl;
    if (!make_map(&xm, x, M)) return cudaErrorInvalidValue;
    if (!make_map(&bh, ctx->crot_split, ctx->N)) return cudaErrorInvalidValue;
    if (!make_map(&bl, ctx->crot_split + (size_t)ctx->N * kD, ctx->N)) return cudaErrorInvalidValue;
    FullParams p;
    p.M = M;
    p.map = map;
    p.N = ctx->N;
    p.B = ctx->B;
    p.h = ctx->cc;
    p.nu = nu;
    p.codes = codes;
    p.flags = ctx->flags;
    const int64_t ntiles = (M + kNG * kRows - 1) / (kNG * kRows);
    int64_t grid = ntiles < ctx->num_sms ? ntiles : ctx->num_sms;
    encode_full_tc<<<(unsigned)grid, kNG * 128 + 32, FLayout::kBytes, s>>>(xm, bh, bl, p);
    return cudaGetLastError();
}

}  // namespace fq
