// Tensor-core full-vector encoder, k = d = 64 [FibQuant §4.2: one index per vector, all bits on
// angular packing; §3.3: sub-one-bit rates, b = log2(N)/64].
//
// With a single block the nearest codeword to u = Pi x / nu is
//     argmin_n |u - c_n|^2,   nu |u - c_n|^2 = nu (|c_n|^2 + 1) - 2 x.(Pi^T c_n)      (nu > 0, |u| = 1),
// a contraction of x with the rotated codebook Crot = C Pi (row n = Pi^T c_n) followed by an
// argmin over n. The contraction runs on the tensor pipe and yields 2^12 nu |u - c_n|^2 directly:
//   A = the x tile (fp16, exact; TMA, 128-byte swizzle), plus a 16-column block per row with
//       nu split into three bf16 parts;
//   B = -2 * 2^12 * Crot as two fp16 halves (hi, lo; TMA, 128-byte swizzle), plus a 16-column
//       block per codeword with 2^12 (|c_n|^2 + 1) split into three bf16 parts, so that one bf16
//       MMA of K = 16 adds the six leading products of the splits (about 24 bits);
//   D = fp32 accumulator in TMEM: per 128-codeword tile, 4 + 4 fp16 MMAs (hi, lo) and the bf16 one.
// Persistent CTAs of 4 row groups x 128 rows share every codebook tile, streamed through a shared-
// memory ring by a loader warp. Two MMA warps issue (each for two row groups, descriptors built once);
// one TMEM buffer of 128 columns per group. 8 consumer warps (two per lane quarter, each serving two
// groups) read each score item with tcgen05.ld.red (each 16-column chunk's minimum comes with the
// load), release the buffer, and fold: the scores are non-negative distances (up to rounding), so
// their bits order like integers; each score takes its column within its chunk in its 4 low
// mantissa bits (a relative change below 2^-19), a tree of 15 integer minima gives the chunk's
// (score, column), and one compare and two selects keep the row's best (chunk, key). Ties go to the
// lowest column, then to the earliest chunk: the lowest n. A chunk whose minimum is above every
// lane's best (by the same key order) cannot change any row's best and is skipped whole; after the
// first codebook tiles most chunks are.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <vector>

#include "fq_bits.cuh"
#include "fq_internal.h"
#include "fq_sm100.cuh"
#include "fq_tmem_red.cuh"

namespace fq {

namespace {

using namespace sm100;

constexpr int kD = 64;
constexpr int kRows = 128;            // rows per group tile (= TMEM lanes)
constexpr int kNG = 4;                // row groups per CTA tile
constexpr int kNT = 128;              // codewords per B tile (MMA N) = TMEM columns per group
constexpr int kStages = 4;
constexpr int kMaxN = 4096;
constexpr float kBScale = 4096.f;     // 2^12 on Crot and on |c|^2 + 1
constexpr int kXBytes = kRows * kD * 2;          // 16 KB: one group's x tile
constexpr int kExBytes = kRows * 16 * 2;         // 4 KB: one group's nu block / one tile's norm block
constexpr int kBHalf = kNT * kD * 2;             // 16 KB: one half of one codebook tile
constexpr int kBStage = 2 * kBHalf + kExBytes;   // hi, lo, norm block
constexpr int kConsumerWarps = 8;
constexpr int kMmaWarp0 = kConsumerWarps, kLoaderWarp = kConsumerWarps + 2;
constexpr int kThreads = (kConsumerWarps + 3) * 32;
constexpr int kChunk = 16;

struct FLayout {
    static constexpr int oX = 0;
    static constexpr int oEx = oX + kNG * kXBytes;
    static constexpr int oB = oEx + kNG * kExBytes;
    static constexpr int oBar = oB + kStages * kBStage;
    // bars: full[kStages], empty[kStages], xload[kNG], a_ready[kNG], ready[kNG], freeb[kNG], drain[2]
    static constexpr int kBars = 2 * kStages + 4 * kNG + 2;
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;
    static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

struct FullParams {
    int64_t M;
    RowMap map;
    int N, B;
    const uint16_t *norm;    // [N / kNT][kRows][16] bf16 parts of 2^12 (|c_n|^2 + 1), no-swizzle K-major
    float *nu;
    uint32_t *codes;
    uint32_t *flags;
};

// K-major operand without swizzle, 16 elements wide: 8-row x 16-byte core matrices, the second
// 8-element half 128 bytes on, the next 8-row group 256 bytes on.
__device__ __forceinline__ uint64_t sdesc_k16_noswz(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(256u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// Byte offset of row t's 16-byte chunk kc (0 or 1) in a 16-element no-swizzle K-major block.
__host__ __device__ constexpr uint32_t k16_off(int t, int kc) { return (uint32_t)((t / 8) * 256 + kc * 128 + (t % 8) * 16); }

// Three bf16 parts of v (v1 + v2 + v3 = v to about 24 bits), as raw bits.
__device__ __forceinline__ void split3_bf16(float v, uint16_t &a, uint16_t &b, uint16_t &c) {
    const __nv_bfloat16 h1 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(h1);
    const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
    const __nv_bfloat16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
    a = __bfloat16_as_ushort(h1);
    b = __bfloat16_as_ushort(h2);
    c = __bfloat16_as_ushort(h3);
}

__global__ void __launch_bounds__(kThreads, 1)
encode_full_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bhi_map,
               const __grid_constant__ CUtensorMap blo_map, const FullParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + FLayout::oBar);
    uint64_t *full = bars, *empty = bars + kStages, *xload = bars + 2 * kStages;
    uint64_t *a_ready = xload + kNG, *ready = a_ready + kNG, *freeb = ready + kNG, *drain = freeb + kNG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + FLayout::oTmem);

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid & 31;
    const int64_t ntiles = (p.M + kNG * kRows - 1) / (kNG * kRows);     // CTA tiles of 512 rows
    const int nbt = p.N / kNT;                                            // codebook tiles

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 2);                  // both MMA warps have read the stage
        }
        for (int g = 0; g < kNG; ++g) {
            mbar_init(xload + g, 1);
            mbar_init(a_ready + g, 4);                // the group's four consumer warps wrote its nu block
            mbar_init(ready + g, 1);
            mbar_init(freeb + g, 4);                  // the group's four consumer warps read its scores
        }
        mbar_init(drain, 1);
        mbar_init(drain + 1, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_launch_dependents();

    if (warp == kLoaderWarp) {
        // Loader: the first x tile of every group, then the codebook tiles, for every CTA tile in turn.
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            prefetch_tensormap(&bhi_map);
            prefetch_tensormap(&blo_map);
            griddep_wait();                           // x may be written by the previous kernel
            if ((int64_t)blockIdx.x < ntiles)
                for (int g = 0; g < kNG; ++g) {
                    mbar_arrive_expect_tx(xload + g, (uint32_t)kXBytes);
                    tma_load_2d(sm + FLayout::oX + g * kXBytes, &xmap, 0, (int)(blockIdx.x * (kNG * kRows) + g * kRows),
                                xload + g);
                }
            uint32_t k = 0;
            bool ok = true;
            for (int64_t ct = blockIdx.x; ct < ntiles && ok; ct += gridDim.x) {
                for (int bt = 0; bt < nbt; ++bt, ++k) {
                    const uint32_t s = k % kStages, round = k / kStages;
                    if (round > 0) ok = mbar_wait(empty + s, (round - 1) & 1);
                    if (!ok) break;
                    uint8_t *dst = sm + FLayout::oB + s * kBStage;
                    mbar_arrive_expect_tx(full + s, (uint32_t)kBStage);
                    tma_load_2d(dst, &bhi_map, 0, bt * kNT, full + s);
                    tma_load_2d(dst + kBHalf, &blo_map, 0, bt * kNT, full + s);
                    bulk_g2s(dst + 2 * kBHalf, p.norm + (size_t)bt * (kExBytes / 2), (uint32_t)kExBytes, full + s);
                }
            }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
            // Every copy issued into the ring has landed before the CTA can exit.
            for (uint32_t s = 0; s < (uint32_t)kStages && s < k; ++s) {
                const uint32_t n_s = (k - 1 - s) / kStages + 1;
                mbar_wait(full + s, (n_s - 1) & 1, ok ? 2000000000ull : 1000000ull);
            }
        }
    } else if (warp >= kMmaWarp0) {
        // MMA warp q issues the items of groups 2q and 2q + 1: per codebook tile, group 2q then 2q + 1.
        const int q = warp - kMmaWarp0;
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, kNT);
            const uint32_t idesc_n = idesc_f16_f32(128, kNT) | (1u << 7) | (1u << 10);   // A, B bf16
            const uint32_t xbase = smem_addr(sm + FLayout::oX), exbase = smem_addr(sm + FLayout::oEx);
            const uint32_t bbase = smem_addr(sm + FLayout::oB);
            uint32_t k = 0, nitem = 0;                // ring position; items of group 2q (= of 2q + 1)
            bool ok = true;
            int64_t it = 0;
            for (int64_t ct = blockIdx.x; ct < ntiles && ok; ct += gridDim.x, ++it) {
                for (int gg = 0; gg < 2 && ok; ++gg) ok = mbar_wait(a_ready + 2 * q + gg, (uint32_t)(it & 1));
                for (int bt = 0; bt < nbt && ok; ++bt, ++k, ++nitem) {
                    const uint32_t s = k % kStages;
                    ok = mbar_wait(full + s, (k / kStages) & 1);
                    const uint32_t bh = bbase + s * (uint32_t)kBStage, bl = bh + kBHalf, bn = bh + 2 * kBHalf;
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg) {
                        const int g = 2 * q + gg;
                        if (ok && nitem > 0) ok = mbar_wait(freeb + g, (nitem - 1) & 1);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t acc = tmem_base + (uint32_t)(g * kNT);
                        const uint32_t xa = xbase + (uint32_t)(g * kXBytes);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk)
                            mma_f16(acc, sdesc_sw128(xa + kk * 32), sdesc_sw128(bh + kk * 32), idesc, kk ? 1u : 0u);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk)
                            mma_f16(acc, sdesc_sw128(xa + kk * 32), sdesc_sw128(bl + kk * 32), idesc, 1u);
                        mma_f16(acc, sdesc_k16_noswz(exbase + (uint32_t)(g * kExBytes)), sdesc_k16_noswz(bn), idesc_n, 1u);
                        mma_commit(ready + g);
                    }
                    if (ok) mma_commit(empty + s);
                }
            }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
            mma_commit(drain + q);
            mbar_wait(drain + q, 0, ok ? 2000000000ull : 1000000ull);
        }
    } else {
        // Consumers: warp w reads TMEM lanes 32 (w % 4) .. +31 of groups 2 h and 2 h + 1, h = w / 4.
        const int lq = warp % 4, h = warp / 4;
        const int t = 32 * lq + lane;
        const uint32_t lane_off = (uint32_t)(32 * lq) << 16;
        griddep_wait();                               // the code store may be the previous kernel's
        uint32_t nitem = 0;
        bool ok = true;
        int64_t it = 0;
        for (int64_t ct = blockIdx.x; ct < ntiles && ok; ct += gridDim.x, ++it) {
            float nu[2];
            bool finite[2];
            // nu of this thread's row in both groups, and the groups' nu blocks (A of the bf16 MMA).
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int g = 2 * h + gg;
                ok = ok && __all_sync(0xffffffffu, mbar_wait(xload + g, (uint32_t)(it & 1)));
                const uint8_t *xt = sm + FLayout::oX + g * kXBytes;
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xt + t * 128 + ((c ^ (t & 7)) << 4));
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(h2[e]);
                        ss = fmaf(f.x, f.x, ss);
                        ss = fmaf(f.y, f.y, ss);
                    }
                }
                // fp16 inputs are bounded by 65504, so ss is finite unless an element is Inf or NaN.
                finite[gg] = isfinite(ss);
                nu[gg] = finite[gg] ? sqrtf(ss) : 0.f;
                uint16_t a1, a2, a3;
                split3_bf16(nu[gg], a1, a2, a3);
                // A block: [n1, n1, n2, n1, n2, n3, 0...] against B's [H1, H2, H1, H3, H2, H1, 0...]
                uint8_t *ex = sm + FLayout::oEx + g * kExBytes;
                *reinterpret_cast<uint4 *>(ex + k16_off(t, 0)) =
                    make_uint4((uint32_t)a1 | ((uint32_t)a1 << 16), (uint32_t)a2 | ((uint32_t)a1 << 16),
                               (uint32_t)a2 | ((uint32_t)a3 << 16), 0u);
                *reinterpret_cast<uint4 *>(ex + k16_off(t, 1)) = make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_ready + g);
            }
            if (!ok) break;
            // Score items: per codebook tile, group 2h then 2h + 1.
            int bkey[2] = {0x7FFFFFFF, 0x7FFFFFFF}, bchunk[2] = {0, 0};
#pragma unroll 1
            for (int bt = 0; bt < nbt && ok; ++bt, ++nitem) {
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {
                    const int g = 2 * h + gg;
                    const bool w = __all_sync(0xffffffffu, mbar_wait(ready + g, nitem & 1));
                    if (!w) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // Each 16-column chunk with its minimum (tcgen05.ld.red), one batch, one wait.
                    uint32_t sc[kNT / kChunk][16];
                    float mc[kNT / kChunk];
                    const uint32_t col = tmem_base + lane_off + (uint32_t)(g * kNT);
#pragma unroll
                    for (int c = 0; c < kNT / kChunk; ++c) mc[c] = tmem_ldred16_min(col + kChunk * c, sc[c]);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(freeb + g);            // the scores are in registers
#pragma unroll
                    for (int c = 0; c < kNT / kChunk; ++c) {
                        // A chunk can change a row's best only if its minimum's key is not above
                        // the best key (or the minimum is negative, where float and key order
                        // differ): chunks that no lane of the warp needs are skipped.
                        const bool may = (int)(__float_as_uint(mc[c]) & ~15u) <= (bkey[gg] & ~15) || mc[c] < 0.f;
                        if (!__any_sync(0xffffffffu, may)) continue;
                        int v[16];
#pragma unroll
                        for (int z = 0; z < 16; ++z) v[z] = (int)((sc[c][z] & ~15u) | (uint32_t)z);
#pragma unroll
                        for (int wd = 8; wd > 0; wd /= 2)
#pragma unroll
                            for (int z = 0; z < wd; ++z) v[z] = min(v[z], v[z + wd]);
                        const bool better = v[0] < bkey[gg];
                        bkey[gg] = better ? v[0] : bkey[gg];
                        bchunk[gg] = better ? bt * (kNT / kChunk) + c : bchunk[gg];
                    }
                }
            }
            if (!ok) break;
            // Both groups' items of this tile are done (their last MMAs completed): fetch the next
            // x tiles, then store nu and the indices.
            const int64_t next = ct + gridDim.x;
            if (lq == 0 && lane == 0 && next < ntiles)
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {
                    const int g = 2 * h + gg;
                    mbar_arrive_expect_tx(xload + g, (uint32_t)kXBytes);
                    tma_load_2d(sm + FLayout::oX + g * kXBytes, &xmap, 0, (int)(next * (kNG * kRows) + g * kRows),
                                xload + g);
                }
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int64_t r = ct * (kNG * kRows) + (2 * h + gg) * kRows + t;
                if (r < p.M) {
                    const int64_t orow = p.map(r);
                    p.nu[orow] = nu[gg];
                    if (!finite[gg]) atomicOr(p.flags, (uint32_t)FQ_FLAG_NONFINITE);
                    const uint32_t bi = (uint32_t)(bchunk[gg] * kChunk + (bkey[gg] & 15));
                    BitWriter wr(p.codes, orow * (int64_t)p.B);
                    wr.put(nu[gg] > 0.f ? bi : 0u, p.B);
                    wr.flush();
                }
            }
        }
        if (!ok && tid == 0) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
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
    std::vector<float> R((size_t)N * kD), C((size_t)N * kD);
    cudaError_t e = cudaMemcpy(R.data(), ctx->Crot, R.size() * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(C.data(), ctx->C, C.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    // Row-major fp16 halves of -2 * 2^12 * Crot (TMA applies the swizzle when loading), then the
    // norm blocks: per 128-codeword tile, [128][16] bf16 in the no-swizzle K-major layout, row n =
    // [H1, H2, H1, H3, H2, H1, 0...] with H1 + H2 + H3 = 2^12 (|c_n|^2 + 1).
    const size_t nhl = (size_t)2 * N * kD;
    std::vector<uint16_t> hl(nhl + (size_t)N * 16, 0);
    for (size_t i = 0; i < (size_t)N * kD; ++i) {
        const float v = -2.0f * kBScale * R[i];
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        memcpy(&hl[i], &hi, 2);
        memcpy(&hl[(size_t)N * kD + i], &lo, 2);
    }
    for (int n = 0; n < N; ++n) {
        double cc = 0;
        for (int j = 0; j < kD; ++j) cc += (double)C[(size_t)n * kD + j] * C[(size_t)n * kD + j];
        const double H = kBScale * (cc + 1.0);
        const __nv_bfloat16 h1 = __float2bfloat16_rn((float)H);
        const double r1 = H - (double)__bfloat162float(h1);
        const __nv_bfloat16 h2 = __float2bfloat16_rn((float)r1);
        const __nv_bfloat16 h3 = __float2bfloat16_rn((float)(r1 - (double)__bfloat162float(h2)));
        const uint16_t b1 = __bfloat16_as_ushort(h1), b2 = __bfloat16_as_ushort(h2), b3 = __bfloat16_as_ushort(h3);
        const uint16_t row[8] = {b1, b2, b1, b3, b2, b1, 0, 0};
        const int t = n % kNT;
        uint16_t *blk = &hl[nhl + (size_t)(n / kNT) * (kExBytes / 2)];
        memcpy(reinterpret_cast<uint8_t *>(blk) + k16_off(t, 0), row, 16);   // chunk 1 (elements 8..15) stays 0
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
    p.norm = ctx->crot_split + (size_t)2 * ctx->N * kD;
    p.nu = nu;
    p.codes = codes;
    p.flags = ctx->flags;
    const int64_t ntiles = (M + kNG * kRows - 1) / (kNG * kRows);
    const int64_t grid = ntiles < ctx->num_sms ? ntiles : ctx->num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = FLayout::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, encode_full_tc, xm, bh, bl, p);
}

}  // namespace fq
