// Tensor-core block encoder for k = 4 and k = 8 [FibQuant §2.3, encoder].
//
// Per CTA: 16 consumer warps over one 128-row tile (warp w owns TMEM lanes 32 (w % 4)..+31, i.e.
// its rows, and column quarter w / 4 of every score item) and a producer warp.
// For every 128-row tile of x:
//   1. Rotation as in the k = 2 encoder: TMA x tile (128-byte swizzle), tcgen05.mma of x against
//      fp16 hi/lo halves of 2^12 Pi into TMEM; nu from the shared-memory tile.
//   2. Each thread turns its row of u = Y / (2^12 nu) into one A-operand row per block b:
//          A_b = [uh, ul, uh, 2^10, 2^10, 0...],   uh + ul = fp16 hi/lo halves of 2^10 u_b,
//      while every codeword n is a B-operand row
//          B_n = [ch, ch, cl, hh, hl, 0...],        ch + cl = halves of 2^10 (-2 c_n),
//                                                  hh + hl = halves of 2^10 |c_n|^2,
//      so one MMA of K = 16 (k = 4) or K = 32 (k = 8) gives 2^20 (|c_n|^2 - 2 u_b.c_n) for 128 rows
//      and 128 codewords, with fp32 accumulation of exact fp16 products (the dropped ul*cl term
//      is below 2^-22 of the result). |u_b - c_n|^2 differs from it by |u_b|^2, common to all n.
//   3. The codebook streams through a shared-memory ring in 128-codeword tiles (producer warp,
//      bulk copies); two TMEM score buffers let the MMA of one (tile, block) item overlap the
//      argmin of the previous one. Each warp keeps a running minimum per (block, row) over its
//      column quarter: per 16-column chunk a min-tree, and only when the quarter improves on its
//      best so far, a search for its lowest index. The four quarters merge at the end of a pass
//      (lowest score, then lowest index: ties go to the lowest n).
//   4. Indices are packed at the record's fixed bit address; nu is stored.
// Blocks are handled in passes of NBH so that their A operands fit in shared memory.
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

constexpr int kRows = 128;
constexpr int kStages = 4;
constexpr int kCQ = 4;                    // consumer warps per lane quarter (column quarters of an item)
constexpr int kSB = 3;                    // TMEM score buffers (MMAs in flight ahead of the readers)
constexpr int kConsumerWarps = 4 * kCQ;
constexpr int kThreads = kConsumerWarps * 32 + 64;      // + the loader warp and the MMA warp
constexpr float kPiScale = 4096.f;        // 2^12 on Pi
constexpr float kOpScale = 1024.f;        // 2^10 on u, -2c and |c|^2

template <int D, int K, int NBH, int NT>
struct KQ {
    static constexpr int kNT = NT;                                // codewords per B tile (MMA N)
    static constexpr int NB = D / K;
    static constexpr int NPASS = NB / NBH;
    static constexpr int KP = (3 * K + 2 <= 16) ? 16 : 32;        // padded K of one block's operand
    static constexpr int kPiPart = D * D * 2;
    static constexpr int kXTile = kRows * D * 2;
    static constexpr int kABlock = kRows * KP * 2;                // one block's A operand
    static constexpr int kBTile = kNT * KP * 2;                   // one codebook tile
    static constexpr int oPi = 0;
    static constexpr int oX = oPi + 2 * kPiPart;
    static constexpr int oA = oX + kXTile;
    static constexpr int oB = oA + NBH * kABlock;
    static constexpr int oState = oB + kStages * kBTile;         // per (block, quarter, row): best, index
    static constexpr int oBar = oState + NBH * kCQ * kRows * 8;
    // bars: pi, x, rot, a_ready, rot_free, ready[kSB], free[kSB], full[kStages], empty[kStages]
    static constexpr int kBars = 5 + 2 * kSB + 2 * kStages;
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;
    // TMEM: kSB score buffers of kNT columns, then the rotation (so that the next tile's rotation
    // can run while the last scores are read).
    static constexpr int kRotCol = kSB * kNT;
    static constexpr int kCols = kRotCol + D;
    static constexpr uint32_t kTmemCols = kCols <= 256 ? 256 : 512;
    static_assert(kCols <= 512, "tensor memory");
};

struct KQParams {
    int64_t M;
    RowMap map;
    int N, B;
    const uint8_t *pi_split;   // fp16 halves of 2^12 Pi, swizzled (as the k = 2 encoder)
    const uint8_t *cb_ops;     // [N / kNT] tiles of B rows, no-swizzle K-major core-matrix layout
    float *nu;
    uint32_t *codes;
    uint32_t *flags;
};

// K-major operand without swizzle: 8-row x 16-byte core matrices, the next one along K 128 bytes
// on (leading byte offset), the next 8-row group kp * 16 bytes on (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_kmajor_noswz(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    return d;                                          // layout type 0: no swizzle
}

template <int D, int K, int NBH, int NT>
__global__ void __launch_bounds__(kThreads, 1)
encode_kq_tc(const __grid_constant__ CUtensorMap xmap, const KQParams p) {
    using L = KQ<D, K, NBH, NT>;
    constexpr int kNT = NT;
    constexpr int KP = L::KP;
    constexpr int kQC = kNT / kCQ;             // columns of an item read by one warp
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
    uint64_t *bar_pi = bars + 0, *bar_x = bars + 1, *bar_rot = bars + 2;
    uint64_t *a_ready = bars + 3, *rot_free = bars + 4;
    uint64_t *ready = bars + 5, *freeb = bars + 5 + kSB;              // [kSB] each
    uint64_t *full = bars + 5 + 2 * kSB, *empty = bars + 5 + 2 * kSB + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oTmem);
    uint8_t *xt = sm + L::oX;
    float *st_best = reinterpret_cast<float *>(sm + L::oState);
    uint32_t *st_bi = reinterpret_cast<uint32_t *>(sm + L::oState + NBH * kCQ * kRows * 4);

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid & 31;
    const int64_t ntiles = (p.M + kRows - 1) / kRows;
    const int nbt = p.N / kNT;
    constexpr uint32_t kCons = kConsumerWarps * 32;

    if (tid == 0) {
        mbar_init(bar_pi, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_rot, 1);
        mbar_init(a_ready, kConsumerWarps);
        mbar_init(rot_free, kConsumerWarps);
        for (int b = 0; b < kSB; ++b) {
            mbar_init(ready + b, 1);
            mbar_init(freeb + b, kConsumerWarps);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, L::kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t rot_acc = tmem_base + (uint32_t)L::kRotCol;

    if (warp == kConsumerWarps) {
        // Loader: Pi, the first x tile, then the codebook tiles in the order they are used.
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            mbar_arrive_expect_tx(bar_pi, 2u * L::kPiPart);
            bulk_g2s(sm + L::oPi, p.pi_split, 2u * L::kPiPart, bar_pi);
            if ((int64_t)blockIdx.x < ntiles) {
                mbar_arrive_expect_tx(bar_x, (uint32_t)L::kXTile);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb)
                    tma_load_2d(xt + kb * 16384, &xmap, kb * 64, (int)(blockIdx.x * kRows), bar_x);
            }
            uint32_t k = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x)
                for (int pass = 0; pass < L::NPASS && ok; ++pass)
                    for (int bt = 0; bt < nbt && ok; ++bt, ++k) {
                        const uint32_t s = k % kStages, round = k / kStages;
                        if (round > 0) ok = mbar_wait(empty + s, (round - 1) & 1);
                        if (!ok) break;
                        mbar_arrive_expect_tx(full + s, (uint32_t)L::kBTile);
                        bulk_g2s(sm + L::oB + s * L::kBTile, p.cb_ops + (size_t)bt * L::kBTile, L::kBTile, full + s);
                    }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
        }
    } else if (warp == kConsumerWarps + 1) {
        // MMA issuer: the rotation of each tile, then its score items in order.
        if (lane == 0) {
            const uint32_t idesc_rot = idesc_f16_f32(128, D);
            const uint32_t idesc_sc = idesc_f16_f32(128, kNT);
            const uint32_t pi_hi = smem_addr(sm + L::oPi), pi_lo = pi_hi + L::kPiPart;
            const uint32_t a_base = smem_addr(sm + L::oA), b_base = smem_addr(sm + L::oB);
            bool ok = mbar_wait(bar_pi, 0);
            uint32_t k = 0, item = 0, npass = 0;
            int64_t it = 0;
            for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
                ok = mbar_wait(bar_x, (uint32_t)(it & 1));
                // The consumers have read the previous tile's rotation.
                if (ok && it > 0) ok = mbar_wait(rot_free, (uint32_t)((it - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint32_t xa = smem_addr(xt);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint32_t pb = half ? pi_lo : pi_hi;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32);
                        const uint32_t boff = (uint32_t)((kk >> 2) * (D * 128) + (kk & 3) * 32);
                        mma_f16(rot_acc, sdesc_sw128(xa + koff), sdesc_sw128(pb + boff), idesc_rot, (half | kk) ? 1u : 0u);
                    }
                }
                mma_commit(bar_rot);
                for (int pass = 0; pass < L::NPASS && ok; ++pass, ++npass) {
                    ok = mbar_wait(a_ready, npass & 1);
                    for (int bt = 0; bt < nbt && ok; ++bt, ++k) {
                        const uint32_t s = k % kStages;
                        ok = mbar_wait(full + s, (k / kStages) & 1);
                        for (int bb = 0; bb < NBH && ok; ++bb, ++item) {
                            const uint32_t buf = item % kSB;
                            // Buffer `buf` was last filled by item - kSB; wait until it has been read.
                            if (item >= kSB) ok = mbar_wait(freeb + buf, ((item - kSB) / kSB) & 1);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t aa = a_base + (uint32_t)(bb * L::kABlock);
                            const uint32_t ba = b_base + s * (uint32_t)L::kBTile;
                            const uint32_t dst = tmem_base + buf * (uint32_t)kNT;
#pragma unroll
                            for (int kk = 0; kk < KP / 16; ++kk)
                                mma_f16(dst, sdesc_kmajor_noswz(aa + kk * 256, (KP / 8) * 128),
                                        sdesc_kmajor_noswz(ba + kk * 256, (KP / 8) * 128), idesc_sc, kk ? 1u : 0u);
                            mma_commit(ready + buf);
                        }
                        if (ok) mma_commit(empty + s);
                    }
                }
            }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
        }
    } else {
        // Consumers: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows) and column quarter w / 4
        // of every score item.
        const int lq = warp % 4, cq = warp / 4;
        const int t = 32 * lq + lane;             // row within the tile = TMEM lane
        const bool lead = tid == 0;
        const uint32_t lane_off = (uint32_t)(32 * lq) << 16;
        const int R = L::NB * p.B;
        uint32_t item = 0;
        bool ok = true;
        int64_t it = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
            ok = mbar_wait(bar_x, (uint32_t)(it & 1));
            float ss = 0.f;
            if (ok) {
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(xt + kb * 16384 + t * 128 + ((c ^ (t & 7)) << 4));
                        const __half2 *h2 = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __half22float2(h2[q]);
                            ss = fmaf(f.x, f.x, ss);
                            ss = fmaf(f.y, f.y, ss);
                        }
                    }
                }
            }
            ok = named_sync_and(1, kCons, ok && mbar_wait(bar_rot, (uint32_t)(it & 1)));
            if (!ok) break;
            tc_fence_after();
            // nu is read and the rotation has consumed the x tile: fetch the next one.
            const int64_t next = tile + gridDim.x;
            if (lead && next < ntiles) {
                mbar_arrive_expect_tx(bar_x, (uint32_t)L::kXTile);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb)
                    tma_load_2d(xt + kb * 16384, &xmap, kb * 64, (int)(next * kRows), bar_x);
            }
            const bool finite = isfinite(ss);
            const float nu = finite ? sqrtf(ss) : 0.f;
            const float us = nu > 0.f ? (kOpScale / kPiScale) / nu : 0.f;     // 2^10 u = Y * us
            const int64_t r = tile * kRows + t;
            const bool live = r < p.M;
            const int64_t orow = live ? p.map(r) : 0;
            BitWriter wr(p.codes, orow * (int64_t)R);

            for (int pass = 0; pass < L::NPASS && ok; ++pass) {
                // A operands of this pass's blocks (this warp: blocks cq, cq + 4, ...), row t of each.
#pragma unroll
                for (int j = 0; j < NBH / kCQ; ++j) {
                    const int bb = j * kCQ + cq;
                    const int b = pass * NBH + bb;
                    float v[K];
                    float w16[16];
                    tmem_ld16(rot_acc + lane_off + (uint32_t)((b * K / 16) * 16), w16);
                    tmem_wait_ld();
                    const int off = (b * K) % 16;                    // run-time: pick with static indices
#pragma unroll
                    for (int o = 0; o < 16; o += K)
                        if (off == o) {
#pragma unroll
                            for (int q = 0; q < K; ++q) v[q] = w16[o + q] * us;
                        }
                    uint32_t uh[K / 2], ul[K / 2];
#pragma unroll
                    for (int q = 0; q < K / 2; ++q) split_half2(v[2 * q], v[2 * q + 1], uh[q], ul[q]);
                    const uint32_t one2 = 0x64006400u;                // (1024, 1024) in fp16
                    uint8_t *arow = sm + L::oA + bb * L::kABlock + (t / 8) * (KP / 8) * 128 + (t % 8) * 16;
                    if constexpr (K == 4) {
                        *reinterpret_cast<uint4 *>(arow) = make_uint4(uh[0], uh[1], ul[0], ul[1]);
                        *reinterpret_cast<uint4 *>(arow + 128) = make_uint4(uh[0], uh[1], one2, 0u);
                    } else {
                        *reinterpret_cast<uint4 *>(arow) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
                        *reinterpret_cast<uint4 *>(arow + 128) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
                        *reinterpret_cast<uint4 *>(arow + 256) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
                        *reinterpret_cast<uint4 *>(arow + 384) = make_uint4(one2, 0u, 0u, 0u);
                    }
                }
                for (int bb = 0; bb < NBH; ++bb) {
                    st_best[(bb * kCQ + cq) * kRows + t] = INFINITY;
                    st_bi[(bb * kCQ + cq) * kRows + t] = 0u;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(a_ready);
                    if (pass == L::NPASS - 1) mbar_arrive(rot_free);
                }

                const int items = nbt * NBH;
#pragma unroll 1
                for (int i = 0; i < items; ++i, ++item) {
                    const uint32_t buf = item % kSB;
                    const int bt = i / NBH, bb = i % NBH;
                    bool w = mbar_wait(ready + buf, (item / kSB) & 1);
                    w = __all_sync(0xffffffffu, w);
                    if (!w) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float *pb = st_best + (bb * kCQ + cq) * kRows + t;
                    uint32_t *pi = st_bi + (bb * kCQ + cq) * kRows + t;
                    float best = *pb;
                    // This warp's kQC columns of the item, all loads in flight before one wait.
                    uint32_t rr[kQC / 32][32];
#pragma unroll
                    for (int h = 0; h < kQC / 32; ++h)
                        tmem_ld32_nowait(tmem_base + lane_off + (uint32_t)(buf * kNT + cq * kQC + 32 * h), rr[h]);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(freeb + buf);      // the buffer's scores are in registers
                    float cm[kQC / 16];
#pragma unroll
                    for (int c = 0; c < kQC / 16; ++c) {
                        float v16[16];
#pragma unroll
                        for (int z = 0; z < 16; ++z) v16[z] = __uint_as_float(rr[c / 2][16 * (c % 2) + z]);
                        cm[c] = min16(v16);
                    }
                    float qmin = cm[0];
#pragma unroll
                    for (int c = 1; c < kQC / 16; ++c) qmin = fminf(qmin, cm[c]);
                    if (qmin < best) {
                        // The lowest column of this quarter holding the minimum: first the
                        // 16-column chunk (from the chunk minima), then the column within it.
                        int c0 = kQC / 16 - 1;
#pragma unroll
                        for (int c = kQC / 16 - 1; c >= 0; --c)
                            if (cm[c] == qmin) c0 = c;
                        uint32_t j = 15;
#pragma unroll
                        for (int c = 0; c < kQC / 16; ++c)
                            if (c == c0) {
#pragma unroll
                                for (int z = 15; z >= 0; --z)
                                    if (__uint_as_float(rr[c / 2][16 * (c % 2) + z]) == qmin) j = (uint32_t)z;
                            }
                        *pb = qmin;
                        *pi = (uint32_t)(bt * kNT + cq * kQC + c0 * 16) + j;
                    }
                }
                ok = named_sync_and(1, kCons, ok);
                if (!ok) break;
                // Merge the four column quarters of each block (lowest score, then lowest index),
                // pack, and free the state for the next pass.
                if (cq == 0 && live) {
                    for (int bb = 0; bb < NBH; ++bb) {
                        float best = st_best[(bb * kCQ) * kRows + t];
                        uint32_t bi = st_bi[(bb * kCQ) * kRows + t];
#pragma unroll
                        for (int q = 1; q < kCQ; ++q) {
                            const float v = st_best[(bb * kCQ + q) * kRows + t];
                            const uint32_t n = st_bi[(bb * kCQ + q) * kRows + t];
                            if (v < best || (v == best && n < bi)) {
                                best = v;
                                bi = n;
                            }
                        }
                        wr.put(nu > 0.f ? bi : 0u, p.B);
                    }
                }
                ok = named_sync_and(1, kCons, true);
            }
            if (!ok) break;
            if (cq == 0 && live) {
                wr.flush();
                p.nu[orow] = nu;
                if (!finite) atomicOr(p.flags, (uint32_t)FQ_FLAG_NONFINITE);
            }
        }
        if (!ok && lead) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int D, int K, int NBH, int NT>
cudaError_t launch_kq(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu, uint32_t *codes,
                      cudaStream_t s) {
    using L = KQ<D, K, NBH, NT>;
    CUtensorMap tm;
    if (!encode_rows_tensor_map(&tm, x, M, D)) return cudaErrorInvalidValue;
    KQParams p;
    p.M = M;
    p.map = map;
    p.N = ctx->N;
    p.B = ctx->B;
    p.pi_split = ctx->pi_split;
    p.cb_ops = ctx->cb_ops;
    p.nu = nu;
    p.codes = codes;
    p.flags = ctx->flags;
    const int64_t ntiles = (M + kRows - 1) / kRows;
    int64_t grid = ntiles < ctx->kq_max_ctas ? ntiles : ctx->kq_max_ctas;
    encode_kq_tc<D, K, NBH, NT><<<(unsigned)grid, kThreads, L::kBytes, s>>>(tm, p);
    return cudaGetLastError();
}

template <int D, int K, int NBH, int NT>
cudaError_t prep_kq(fq_ctx *ctx) {
    using L = KQ<D, K, NBH, NT>;
    static_assert(L::kBytes <= 227 * 1024, "shared memory budget");
    static_assert(L::NB % NBH == 0, "passes");
    cudaError_t e = cudaFuncSetAttribute(encode_kq_tc<D, K, NBH, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kq_tc<D, K, NBH, NT>, kThreads, L::kBytes);
    if (e != cudaSuccess) return e;
    // TMEM: each resident CTA holds kTmemCols of the SM's 512 columns.
    const int by_tmem = 512 / (int)L::kTmemCols;
    if (per_sm > by_tmem) per_sm = by_tmem;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ctx->kq_max_ctas = per_sm * ctx->num_sms;
    return cudaSuccess;
}

}  // namespace

bool kq_tc_supported(const fq_ctx *ctx) {
    CUtensorMap probe;
    const bool shape = (ctx->d == 64 && ctx->k == 4) || (ctx->d == 128 && ctx->k == 8) ||
                       (ctx->d == 64 && ctx->k == 8) || (ctx->d == 128 && ctx->k == 4);
    return shape && ctx->N >= 128 && ctx->N % 128 == 0 && ctx->N <= 65536 &&
           encode_rows_tensor_map(&probe, ctx->Pi, 128, ctx->d);
}

// Codebook rows as B operands: [ch, ch, cl, hh, hl, 0...] per codeword (k-wide groups), in the
// K-major no-swizzle layout: codeword n, 16-byte chunk kc of its row at
// (n / 8) * (KP / 8) * 128 + kc * 128 + (n % 8) * 16, so any run of whole 8-codeword groups (a
// 128- or 256-codeword tile) is contiguous.
cudaError_t prepare_kq_tc(fq_ctx *ctx) {
    const int N = ctx->N, k = ctx->k, d = ctx->d;
    const int KP = (3 * k + 2 <= 16) ? 16 : 32;
    std::vector<float> C((size_t)N * k), P((size_t)d * d);
    cudaError_t e = cudaMemcpy(C.data(), ctx->C, C.size() * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(P.data(), ctx->Pi, P.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    std::vector<uint16_t> ops((size_t)N * KP, 0);
    auto split = [](double v, __half &hi, __half &lo) {
        hi = __float2half_rn((float)v);
        lo = __float2half_rn((float)(v - (double)__half2float(hi)));
    };
    for (int n = 0; n < N; ++n) {
        std::vector<__half> row(KP, __float2half_rn(0.f));
        double h = 0;
        for (int q = 0; q < k; ++q) {
            const double c = C[(size_t)n * k + q];
            h += c * c;
            __half hi, lo;
            split(kOpScale * -2.0 * c, hi, lo);
            row[q] = hi;
            row[k + q] = hi;
            row[2 * k + q] = lo;
        }
        __half hh, hl;
        split(kOpScale * h, hh, hl);
        row[3 * k] = hh;
        row[3 * k + 1] = hl;
        for (int kc = 0; kc < KP / 8; ++kc)
            for (int q = 0; q < 8; ++q) {
                const size_t off = (size_t)(n / 8) * (KP / 8) * 64 + (size_t)kc * 64 + (size_t)(n % 8) * 8 + q;
                memcpy(&ops[off], &row[kc * 8 + q], 2);
            }
    }
    e = cudaMalloc((void **)&ctx->cb_ops, ops.size() * 2);
    if (e == cudaSuccess) e = cudaMemcpy(ctx->cb_ops, ops.data(), ops.size() * 2, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return e;
    if (!ctx->pi_split) {
        std::vector<uint16_t> pis;
        split_operand_sw128(P.data(), d, kPiScale, pis);
        e = cudaMalloc((void **)&ctx->pi_split, pis.size() * 2);
        if (e == cudaSuccess) e = cudaMemcpy(ctx->pi_split, pis.data(), pis.size() * 2, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return e;
    }
    if (d == 64 && k == 4) return prep_kq<64, 4, 16, 128>(ctx);
    if (d == 64 && k == 8) return prep_kq<64, 8, 8, 128>(ctx);
    if (d == 128 && k == 4) return prep_kq<128, 4, 8, 128>(ctx);
    return prep_kq<128, 8, 8, 128>(ctx);
}

cudaError_t launch_encode_kq_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                uint32_t *codes, cudaStream_t s) {
    if (ctx->d == 64 && ctx->k == 4) return launch_kq<64, 4, 16, 128>(ctx, x, M, map, nu, codes, s);
    if (ctx->d == 64 && ctx->k == 8) return launch_kq<64, 8, 8, 128>(ctx, x, M, map, nu, codes, s);
    if (ctx->d == 128 && ctx->k == 4) return launch_kq<128, 4, 8, 128>(ctx, x, M, map, nu, codes, s);
    return launch_kq<128, 8, 8, 128>(ctx, x, M, map, nu, codes, s);
}

}  // namespace fq
