// Tensor-core block encoder for k = 4 and k = 8 [FibQuant §2.3, encoder].
//
// Persistent CTAs, one per SM: a loader warp (bulk and TMA copies), two MMA warps and 8 consumer
// warps (two per TMEM lane quarter). Issuing tcgen05.mma costs the issuing thread about as much
// time per instruction whatever the instruction's N, so the score MMAs take the widest N (256
// codewords), two threads issue them (items alternate) and the issue loop is kept short
// (descriptors built once, advanced by adds).
// For every 128-row tile of x, in passes of NBH blocks:
//   1. Rotation item: tcgen05.mma of the x tile (TMA, 128-byte swizzle) against fp16 hi/lo halves
//      of 2^12 Pi, for the pass's columns of Y, into a TMEM buffer. Products of fp16 values are
//      exact and the sums fp32, so Y carries fp32 accuracy. The consumers take nu from the
//      shared-memory tile (first pass), read Y and write one A-operand row per block b and row t:
//          A_b = [uh, ul, uh, 2^10, 2^10, sh, sl, 0...],   uh + ul = fp16 hi/lo halves of 2^10 u_b,
//                                                         sh + sl = halves of 2^10 |u_b|^2,
//      while every codeword n is a B-operand row
//          B_n = [ch, ch, cl, hh, hl, 2^10, 2^10, 0...],   ch + cl = halves of 2^10 (-2 c_n),
//                                                         hh + hl = halves of 2^10 |c_n|^2,
//      so one MMA of K = 16 (k = 4) or K = 32 (k = 8) gives 2^20 |u_b - c_n|^2 (as
//      |c_n|^2 - 2 u_b.c_n + |u_b|^2) for 128 rows and NT codewords; the dropped ul*cl term is
//      below 2^-22 of the terms. These scores are non-negative up to rounding.
//   2. Score items: for each NT-codeword tile of the codebook (resident in shared memory when it
//      fits, else streamed through a ring) and each block of the pass, one MMA into one of two
//      NT-column TMEM buffers. The two consumer warps of a lane quarter read every item, each
//      half of the columns (32 rows x 128 scores, sixteen 8-column loads in one batch), and release
//      the buffer once the loads have landed. Each load is a tcgen05.ld.red: with the columns it
//      returns their minimum per row, so an 8-column chunk folds to its minimum without CUDA-core
//      work; the chunk's number within the half goes into the four low mantissa bits (a
//      relative change below 2^-19 of the score), so one integer minimum per chunk keeps the
//      running (score, chunk) of the item and the lowest chunk wins a tie. Per (row, block) the
//      best item so far and its codeword tile are kept (a later tile wins only by a lower key).
//   3. Resolution: at the end of the pass the two halves' candidates of each (row, block) meet in
//      shared memory (lower score, then lower codeword index), which gives the 8-codeword chunk
//      that holds the smallest tensor-core score. Its 8 codewords are scored again on the CUDA
//      cores by squared difference |u_b - c_n|^2 in fp32 (u_b = (uh + ul) / 2^10, the values the
//      MMA used; packed two-lane arithmetic), lowest score first, ties to the lowest n. The
//      codeword found is within the tensor-core scores' rounding (about 2^-20 of the terms) of
//      the true nearest one. The fp32
//      codebook is read from shared memory: once u is in registers, the A operands' space takes
//      it by bulk copies (as many rounds as it needs), so that these random reads never go to L2.
//   4. Indices are staged in shared memory and packed at the record's fixed bit address; nu is
//      stored.
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

constexpr int kRows = 128;
constexpr int kChunk = 8;                 // codewords per tracked chunk
constexpr int kBufs = 2;                  // TMEM score buffers of NT columns
constexpr int kQ = 2;                     // consumer warps per TMEM lane quarter (column parts of an item)
constexpr int kConsumerWarps = 4 * kQ;
constexpr int kLoaderWarp = kConsumerWarps, kMmaWarp0 = kConsumerWarps + 1;
constexpr int kThreads = kConsumerWarps * 32 + 96;      // + the loader warp and two MMA warps
constexpr uint32_t kCons = kConsumerWarps * 32;
constexpr float kPiScale = 4096.f;        // 2^12 on Pi
constexpr float kOpScale = 1024.f;        // 2^10 on u, -2c and |c|^2
constexpr int kSmemBudget = 227 * 1024;

template <int D, int K, int NBH, int NT>
struct KQ {
    static constexpr int NB = D / K;
    static constexpr int NPASS = NB / NBH;
    static constexpr int kPassCols = NBH * K;                     // Y columns one pass reads
    static constexpr int KP = (3 * K + 4 <= 16) ? 16 : 32;        // padded K of one block's operand
    static constexpr int kPiPart = D * D * 2;
    static constexpr int kXTile = kRows * D * 2;
    static constexpr int kABlock = kRows * KP * 2;                // one block's A operand
    static constexpr int kBTile = NT * KP * 2;                    // one codebook tile
    static constexpr int oPi = 0;
    static constexpr int oX = oPi + 2 * kPiPart;
    static constexpr int oA = oX + kXTile;
    static constexpr int kLd = NT / kQ;                           // score columns one consumer warp reads
    static constexpr int oIdx = oA + NBH * kABlock;               // uint16 [kRows][NB]
    static constexpr int oXch = oIdx + ((kRows * NB * 2 + 1023) & ~1023);   // [kQ][NBH][kRows] key, then tile
    static constexpr int kXchBytes = (kQ * NBH * kRows * 6 + 1023) & ~1023;
    static constexpr int oRing = oXch + kXchBytes;
    static constexpr int kTail = 512 + 16 + 1024;                 // barriers, TMEM slot, alignment slack
    static constexpr int kStagesFit = (kSmemBudget - oRing - kTail) / kBTile;
    static constexpr int kStages = kStagesFit > 16 ? 16 : kStagesFit;
    static constexpr int oBar = oRing + kStages * kBTile;
    // bars: pi, x, a_ready, res, drain[2], ready[kBufs], freeb[kBufs], full[kStages], empty[kStages]
    static constexpr int kBars = 6 + 2 * kBufs + 2 * kStages;
    static constexpr int kResCw = NBH * kABlock / (K * 4);         // fp32 codewords the A space holds
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;
    static_assert(kStages >= 2, "codebook ring");
    static_assert(kBars * 8 <= 512, "barrier space");
    static_assert(kPassCols % 32 == 0 && kPassCols <= 64, "one pass reads 32 or 64 columns of Y");
    static_assert(kBufs * NT <= 512, "tensor memory");
    static_assert(kLd % 32 == 0 && kPassCols <= NT, "score buffers: whole 32-column groups per consumer warp and item");
    static_assert(kResCw % kChunk == 0, "resolution rounds hold whole chunks");
    static_assert(NBH % kQ == 0, "the consumer warps of a lane quarter split the blocks' A rows");
};

struct KQParams {
    int64_t M;
    RowMap map;
    int N, B;
    const uint8_t *pi_split;   // fp16 halves of 2^12 Pi, swizzled (as the k = 2 encoder)
    const uint8_t *cb_ops;     // [N / NT] tiles of B rows, no-swizzle K-major core-matrix layout
    const float *C;            // [N x K] fp32 codebook (chunk resolution)
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

__device__ __forceinline__ float h2f_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float h2f_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

template <int D, int K, int NBH, int NT>
__global__ void __launch_bounds__(kThreads, 1)
encode_kq_tc(const __grid_constant__ CUtensorMap xmap, const KQParams p) {
    using L = KQ<D, K, NBH, NT>;
    constexpr int KP = L::KP, NB = L::NB, NPASS = L::NPASS, S = L::kStages;
    constexpr int OWN = NBH / kQ;                      // blocks of a pass whose A rows one consumer warp writes
    constexpr uint32_t kSubMask = (uint32_t)(L::kLd / kChunk) - 1u;   // key bits that carry the chunk within a part
    constexpr int kLd = L::kLd;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
    uint64_t *bar_pi = bars + 0, *bar_x = bars + 1, *a_ready = bars + 2, *res_bar = bars + 3, *drain = bars + 4;
    uint64_t *ready = bars + 6, *freeb = bars + 6 + kBufs;
    uint64_t *full = bars + 6 + 2 * kBufs, *empty = bars + 6 + 2 * kBufs + S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oTmem);
    uint8_t *xt = sm + L::oX;
    uint8_t *ring = sm + L::oRing;
    uint16_t *idx_s = reinterpret_cast<uint16_t *>(sm + L::oIdx);

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid & 31;
    const int64_t ntiles = (p.M + kRows - 1) / kRows;
    const int nbt = p.N / NT;
    const bool resident = nbt <= S;                   // the whole codebook fits the ring

    if (tid == 0) {
        mbar_init(bar_pi, 1);
        mbar_init(bar_x, 1);
        mbar_init(a_ready, 1);
        mbar_init(res_bar, 1);
        mbar_init(drain, 1);
        mbar_init(drain + 1, 1);
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(ready + b, 1);
            mbar_init(freeb + b, kConsumerWarps);     // every consumer warp reads its part of an item
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 2);                  // both MMA warps' items on the stage are done
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The next kernel in the stream may start its prologue; it waits for this grid before it
    // touches memory this one writes.
    griddep_launch_dependents();

    if (warp == kLoaderWarp) {
        // Loader: Pi and (when resident) the whole codebook, then the first x tile, then the
        // codebook tiles in the order the MMA warp uses them.
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            mbar_arrive_expect_tx(bar_pi, 2u * L::kPiPart);
            bulk_g2s(sm + L::oPi, p.pi_split, 2u * L::kPiPart, bar_pi);
            if (resident)
                for (int bt = 0; bt < nbt; ++bt) {
                    mbar_arrive_expect_tx(full + bt, (uint32_t)L::kBTile);
                    bulk_g2s(ring + bt * L::kBTile, p.cb_ops + (size_t)bt * L::kBTile, L::kBTile, full + bt);
                }
            griddep_wait();                           // x may be written by the previous kernel
            if ((int64_t)blockIdx.x < ntiles) {
                mbar_arrive_expect_tx(bar_x, (uint32_t)L::kXTile);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb)
                    tma_load_2d(xt + kb * 16384, &xmap, kb * 64, (int)(blockIdx.x * kRows), bar_x);
            }
            uint32_t k = 0;
            bool ok = true;
            if (!resident)
                for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x)
                    for (int pass = 0; pass < NPASS && ok; ++pass)
                        for (int bt = 0; bt < nbt; ++bt, ++k) {
                            const uint32_t s = k % S, round = k / S;
                            if (round > 0) ok = mbar_wait(empty + s, (round - 1) & 1);
                            if (!ok) break;
                            mbar_arrive_expect_tx(full + s, (uint32_t)L::kBTile);
                            bulk_g2s(ring + s * L::kBTile, p.cb_ops + (size_t)bt * L::kBTile, L::kBTile, full + s);
                        }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
            // Every copy issued into the ring has landed before the CTA can exit (at once on the
            // normal path, where the MMA warp consumed them all).
            const uint32_t issued = resident ? (uint32_t)nbt : k;
            for (uint32_t s = 0; s < (uint32_t)S && s < issued; ++s) {
                const uint32_t n_s = (issued - 1 - s) / S + 1;              // copies into stage s
                mbar_wait(full + s, (n_s - 1) & 1, ok ? 2000000000ull : 1000000ull);
            }
        }
    } else if (warp >= kMmaWarp0) {
        // MMA issuers: per pass a rotation item, then the score items in (codeword tile, block)
        // order; item n goes to buffer n mod 2 and is issued by MMA warp n mod 2.
        const uint32_t q = (uint32_t)(warp - kMmaWarp0);
        if (lane == 0) {
            const uint32_t idesc_rot = idesc_f16_f32(128, L::kPassCols);
            const uint32_t idesc_sc = idesc_f16_f32(128, NT);
            const uint32_t pi_hi = smem_addr(sm + L::oPi), pi_lo = pi_hi + L::kPiPart;
            const uint64_t da0 = sdesc_kmajor_noswz(smem_addr(sm + L::oA), (KP / 8) * 128);
            const uint64_t db0 = sdesc_kmajor_noswz(smem_addr(ring), (KP / 8) * 128);
            constexpr uint32_t kStepK = 256u >> 4;    // the next 16 K elements: two 128-byte core columns
            constexpr uint32_t kAStep = (uint32_t)L::kABlock >> 4, kBStep = (uint32_t)L::kBTile >> 4;
            bool ok = mbar_wait(bar_pi, 0);
            uint32_t n = 0;                           // items issued
            uint32_t k = 0, npass = 0;
            int64_t it = 0;
            for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
                for (int pass = 0; pass < NPASS && ok; ++pass, ++npass) {
                    if ((n & 1u) == q) {
                        const uint32_t buf = n & 1u, use = n >> 1;
                        if (use > 0) ok = mbar_wait(freeb + buf, (use - 1) & 1);
                        if (ok && pass == 0) ok = mbar_wait(bar_x, (uint32_t)(it & 1));
                        if (!ok) break;
                        tc_fence_after();
                        // Y[:, pass*64 .. +64) = X Pi[pass*64 .. +64, :]^T: the B rows of this pass.
                        const uint32_t xa = smem_addr(xt);
                        const uint32_t rot = tmem_base + buf * (uint32_t)NT;
                        const uint32_t prow = (uint32_t)(pass * L::kPassCols * 128);
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t pb = (half ? pi_lo : pi_hi) + prow;
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t koff = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32);
                                const uint32_t boff = (uint32_t)((kk >> 2) * (D * 128) + (kk & 3) * 32);
                                mma_f16(rot, sdesc_sw128(xa + koff), sdesc_sw128(pb + boff), idesc_rot,
                                        (half | kk) ? 1u : 0u);
                            }
                        }
                        mma_commit(ready + buf);
                    }
                    ++n;
                    // The consumers have written this pass's A operands (and read the rotation).
                    ok = mbar_wait(a_ready, npass & 1);
                    if (!ok) break;
                    tc_fence_after();
                    for (int bt = 0; bt < nbt && ok; ++bt) {
                        const uint32_t s = resident ? (uint32_t)bt : k % S;
                        ok = mbar_wait(full + s, resident ? 0u : (k / S) & 1);
                        const uint64_t db = db0 + (uint64_t)(s * kBStep);
                        uint64_t da = da0;
                        // This warp's items of the tile: blocks bb with (n + bb) mod 2 = q.
                        const uint32_t b0 = (n & 1u) ^ q;
                        n += (uint32_t)NBH;
                        da += b0 * kAStep;
#pragma unroll 1
                        for (uint32_t bb = b0; bb < (uint32_t)NBH && ok; bb += 2, da += 2 * kAStep) {
                            const uint32_t g = n - (uint32_t)NBH + bb;
                            const uint32_t buf = g & 1u, use = g >> 1;
                            if (use > 0) ok = mbar_wait(freeb + buf, (use - 1) & 1);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t dst = tmem_base + buf * (uint32_t)NT;
                            mma_f16(dst, da, db, idesc_sc, 0u);
#pragma unroll
                            for (int kk = 1; kk < KP / 16; ++kk) mma_f16(dst, da + kk * kStepK, db + kk * kStepK, idesc_sc, 1u);
                            mma_commit(ready + buf);
                        }
                        if (!resident) {
                            if (ok) mma_commit(empty + s);
                            ++k;
                        }
                    }
                }
            }
            if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
            // Every MMA issued has completed before the CTA can exit.
            mma_commit(drain + q);
            mbar_wait(drain + q, 0, ok ? 2000000000ull : 1000000ull);
        }
    } else {
        // Consumers: warp w reads TMEM lanes 32 (w % 4) .. +31, i.e. rows t of the tile; it reads
        // column part w / 4 of every item and writes (and resolves) the blocks b = w / 4 (mod kQ).
        const int lq = warp % 4, cq = warp / 4;
        const int t = 32 * lq + lane;
        const uint32_t lane_off = (uint32_t)(32 * lq) << 16;
        const int R = NB * p.B;
        griddep_wait();                               // the code store may be the previous kernel's
        uint32_t n = 0;                               // items of the MMA warps' sequence passed
        uint32_t res_n = 0;                           // codebook rounds copied for the resolution
        bool ok = true;
        int64_t it = 0;
        uint32_t x_issued = (int64_t)blockIdx.x < ntiles ? 1u : 0u, x_done = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
            const int64_t r = tile * kRows + t;
            const bool live = r < p.M;
            float nu = 0.f, us = 0.f;
            bool finite = true;
            for (int pass = 0; pass < NPASS && ok; ++pass) {
                // --- rotation item: nu (first pass), then this pass's A operands ---------------
                {
                    const uint32_t buf = n & 1u;
                    bool w = mbar_wait(ready + buf, (n >> 1) & 1);
                    if (pass == 0) w = w && mbar_wait(bar_x, (uint32_t)(it & 1));
                    ok = named_sync_and(1, kCons, w);
                    if (!ok) break;
                    if (pass == 0) ++x_done;
                    tc_fence_after();
                    if (pass == 0) {
                        float ss = 0.f;
#pragma unroll
                        for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const uint4 v =
                                    *reinterpret_cast<const uint4 *>(xt + kb * 16384 + t * 128 + ((c ^ (t & 7)) << 4));
                                const __half2 *h2 = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = __half22float2(h2[e]);
                                    ss = fmaf(f.x, f.x, ss);
                                    ss = fmaf(f.y, f.y, ss);
                                }
                            }
                        }
                        // fp16 inputs are bounded by 65504, so ss is finite unless an element is
                        // Inf or NaN.
                        finite = isfinite(ss);
                        nu = finite ? sqrtf(ss) : 0.f;
                        us = nu > 0.f ? (kOpScale / kPiScale) / nu : 0.f;     // 2^10 u = Y * us
                    }
                    // This warp's blocks' columns of Y (the column address is per warp, so each
                    // block's K columns are one load).
                    uint32_t y[OWN][K];
                    const uint32_t ycol = tmem_base + lane_off + buf * (uint32_t)NT;
#pragma unroll
                    for (int j = 0; j < OWN; ++j) {
                        const uint32_t ca = ycol + (uint32_t)((kQ * j + cq) * K);
                        if constexpr (K == 4) tmem_ld4_nowait(ca, y[j]);
                        else tmem_ld8_nowait(ca, y[j]);
                    }
                    tmem_wait_ld();
                    const bool zero = !(nu > 0.f);
#pragma unroll
                    for (int j = 0; j < OWN; ++j) {
                        const int bb = kQ * j + cq;
                        float v[K];
                        float uu = 0.f;
#pragma unroll
                        for (int e = 0; e < K; ++e) {
                            v[e] = zero ? 0.f : __uint_as_float(y[j][e]) * us;
                            uu = fmaf(v[e], v[e], uu);
                        }
                        uint32_t uh[K / 2], ul[K / 2], ss2, sdummy;
#pragma unroll
                        for (int e = 0; e < K / 2; ++e) split_half2(v[2 * e], v[2 * e + 1], uh[e], ul[e]);
                        // 2^10 |u_b|^2 = sum (2^10 u)^2 / 2^10 as fp16 hi/lo, packed (hi, lo)
                        {
                            const float su = uu * (1.f / kOpScale);
                            const __half sh = __float2half_rn(su);
                            const __half sl = __float2half_rn(su - __half2float(sh));
                            ss2 = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(sl) << 16);
                            sdummy = 0u;
                        }
                        const uint32_t one2 = 0x64006400u;            // (1024, 1024) in fp16
                        uint8_t *arow = sm + L::oA + bb * L::kABlock + (t / 8) * (KP / 8) * 128 + (t % 8) * 16;
                        if constexpr (K == 4) {
                            *reinterpret_cast<uint4 *>(arow) = make_uint4(uh[0], uh[1], ul[0], ul[1]);
                            *reinterpret_cast<uint4 *>(arow + 128) = make_uint4(uh[0], uh[1], one2, ss2);
                        } else {
                            *reinterpret_cast<uint4 *>(arow) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
                            *reinterpret_cast<uint4 *>(arow + 128) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
                            *reinterpret_cast<uint4 *>(arow + 256) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
                            *reinterpret_cast<uint4 *>(arow + 384) = make_uint4(one2, ss2, sdummy, 0u);
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    named_sync(1, kCons);
                    if (tid == 0) {
                        mbar_arrive(a_ready);
#pragma unroll
                        for (int e = 0; e < kConsumerWarps; ++e) mbar_arrive(freeb + buf);
                        // The last pass's rotation was the x tile's last reader: fetch the next.
                        const int64_t next = tile + gridDim.x;
                        if (pass == NPASS - 1 && next < ntiles) {
                            mbar_arrive_expect_tx(bar_x, (uint32_t)L::kXTile);
#pragma unroll
                            for (int kb = 0; kb < D / 64; ++kb)
                                tma_load_2d(xt + kb * 16384, &xmap, kb * 64, (int)(next * kRows), bar_x);
                        }
                    }
                    if (pass == NPASS - 1 && tile + gridDim.x < ntiles) ++x_issued;
                    ++n;
                }
                // --- score items: this warp's part of the columns of every item --------------------
                // All kLd columns of an item in one batch of loads and one wait, then the buffer is
                // released and the columns are folded.
                int bkey[NBH], btile[NBH];
#pragma unroll
                for (int bb = 0; bb < NBH; ++bb) {
                    bkey[bb] = 0x7FFFFFFF;
                    btile[bb] = 0;
                }
                const uint32_t colq = tmem_base + lane_off + (uint32_t)(cq * kLd);
#pragma unroll 1
                for (int bt = 0; bt < nbt && ok; ++bt) {
#pragma unroll
                    for (int bb = 0; bb < NBH; ++bb) {
                        const uint32_t g = n + (uint32_t)(bt * NBH + bb);
                        const uint32_t buf = g & 1u;
                        ok = __all_sync(0xffffffffu, mbar_wait(ready + buf, (g >> 1) & 1));
                        if (!ok) break;
                        tc_fence_after();
                        // Each 8-column chunk's minimum comes with its load (tcgen05.ld.red);
                        // all kLd columns in one batch and one wait, then the buffer is released.
                        uint32_t rr[kLd / kChunk][8];
                        float mc[kLd / kChunk];
#pragma unroll
                        for (int c = 0; c < kLd / kChunk; ++c)
                            mc[c] = tmem_ldred8_min(colq + buf * (uint32_t)NT + (uint32_t)(kChunk * c), rr[c]);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < kLd / kChunk; ++c) keep8(rr[c]);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(freeb + buf);      // the minima are in registers
                        int ikey = 0x7FFFFFFF;
#pragma unroll
                        for (int c = 0; c < kLd / kChunk; ++c)
                            ikey = min(ikey, (int)((__float_as_uint(mc[c]) & ~kSubMask) | (uint32_t)c));
                        const bool better = ikey < bkey[bb];
                        bkey[bb] = better ? ikey : bkey[bb];
                        btile[bb] = better ? bt : btile[bb];
                    }
                }
                n += (uint32_t)(nbt * NBH);
                // Candidates of the column parts to shared memory: the resolver of a block takes all.
                int *xk = reinterpret_cast<int *>(sm + L::oXch);
                uint16_t *xt16 = reinterpret_cast<uint16_t *>(sm + L::oXch + kQ * NBH * kRows * 4);
#pragma unroll
                for (int bb = 0; bb < NBH; ++bb) {
                    xk[(cq * NBH + bb) * kRows + t] = bkey[bb];
                    xt16[(cq * NBH + bb) * kRows + t] = (uint16_t)btile[bb];
                }
                ok = named_sync_and(1, kCons, ok);
                if (!ok) break;
                // --- resolution of the owned blocks' chunks, by squared difference ------------
                // u of the owned blocks into registers (from the A rows: the values the MMA used),
                // and the winning chunk of each: the lowest score part of the parts' keys, then the
                // lowest codeword index (tile, part, chunk within the part).
                float u[OWN][K];
                int cjs[OWN];
#pragma unroll
                for (int j = 0; j < OWN; ++j) {
                    const int bb = kQ * j + cq;
                    const uint8_t *arow = sm + L::oA + bb * L::kABlock + (t / 8) * (KP / 8) * 128 + (t % 8) * 16;
                    if constexpr (K == 4) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(arow);      // uh[4], ul[4]
                        u[j][0] = (h2f_lo(a.x) + h2f_lo(a.z)) * (1.f / kOpScale);
                        u[j][1] = (h2f_hi(a.x) + h2f_hi(a.z)) * (1.f / kOpScale);
                        u[j][2] = (h2f_lo(a.y) + h2f_lo(a.w)) * (1.f / kOpScale);
                        u[j][3] = (h2f_hi(a.y) + h2f_hi(a.w)) * (1.f / kOpScale);
                    } else {
                        const uint4 a = *reinterpret_cast<const uint4 *>(arow);         // uh[8]
                        const uint4 b = *reinterpret_cast<const uint4 *>(arow + 128);   // ul[8]
                        const uint32_t ah[4] = {a.x, a.y, a.z, a.w}, al[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            u[j][2 * e] = (h2f_lo(ah[e]) + h2f_lo(al[e])) * (1.f / kOpScale);
                            u[j][2 * e + 1] = (h2f_hi(ah[e]) + h2f_hi(al[e])) * (1.f / kOpScale);
                        }
                    }
                    int bs = 0x7FFFFFFF, bc = 0;
#pragma unroll
                    for (int q = 0; q < kQ; ++q) {
                        const int key = xk[(q * NBH + bb) * kRows + t];
                        const int sc = key & ~(int)kSubMask;
                        const int cidx = (int)xt16[(q * NBH + bb) * kRows + t] * (NT / kChunk) + q * (kLd / kChunk) +
                                         (key & (int)kSubMask);
                        if (sc < bs || (sc == bs && cidx < bc)) {
                            bs = sc;
                            bc = cidx;
                        }
                    }
                    cjs[j] = bc;
                }
                // The A space is free once every consumer holds its u: it takes the fp32 codebook,
                // L::kResCw codewords per round.
                fence_proxy_async_smem();
                named_sync(1, kCons);
                float bd[OWN];
                int bi[OWN];
                float2 nu2[OWN][K / 2];            // -u in pairs, for the packed differences
#pragma unroll
                for (int j = 0; j < OWN; ++j) {
                    bd[j] = INFINITY;
                    bi[j] = cjs[j] * kChunk;
#pragma unroll
                    for (int e = 0; e < K / 2; ++e) nu2[j][e] = make_float2(-u[j][2 * e], -u[j][2 * e + 1]);
                }
                const float *cs = reinterpret_cast<const float *>(sm + L::oA);
#pragma unroll 1
                for (int base = 0; base < p.N && ok; base += L::kResCw) {
                    const int ncw = p.N - base < L::kResCw ? p.N - base : L::kResCw;
                    if (tid == 0) {
                        mbar_arrive_expect_tx(res_bar, (uint32_t)(ncw * K * 4));
                        bulk_g2s(sm + L::oA, p.C + (size_t)base * K, (uint32_t)(ncw * K * 4), res_bar);
                    }
                    ok = named_sync_and(1, kCons, mbar_wait(res_bar, res_n & 1));
                    ++res_n;
                    if (!ok) break;
#pragma unroll
                    for (int j = 0; j < OWN; ++j) {
                        const int c0 = cjs[j] * kChunk - base;
                        if (c0 >= 0 && c0 < ncw) {
                            // Every chunk starts on a kChunk-codeword boundary, so the lanes read
                            // their chunks in lane-rotated order (codeword (q + lane) mod kChunk at
                            // step q) to spread the reads over the banks; ties still go to the
                            // lowest index.
#pragma unroll 4
                            for (int q0 = 0; q0 < kChunk; ++q0) {
                                const int q = (q0 + lane) & (kChunk - 1);
                                const float4 *cp = reinterpret_cast<const float4 *>(cs + (size_t)(c0 + q) * K);
                                // |c - u|^2 in packed fp32 pairs: e = c + (-u), then the squares
                                // summed pairwise and the two lanes added.
                                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                                for (int e = 0; e < K / 4; ++e) {
                                    const float4 c = cp[e];
                                    const float2 e01 = __fadd2_rn(make_float2(c.x, c.y), nu2[j][2 * e]);
                                    const float2 e23 = __fadd2_rn(make_float2(c.z, c.w), nu2[j][2 * e + 1]);
                                    acc = __ffma2_rn(e01, e01, acc);
                                    acc = __ffma2_rn(e23, e23, acc);
                                }
                                const float dsum = acc.x + acc.y;
                                const int nq = base + c0 + q;
                                if (dsum < bd[j] || (dsum == bd[j] && nq < bi[j])) {
                                    bd[j] = dsum;
                                    bi[j] = nq;
                                }
                            }
                        }
                    }
                    named_sync(1, kCons);             // every read of this round is done
                }
#pragma unroll
                for (int j = 0; j < OWN; ++j) idx_s[t * NB + pass * NBH + kQ * j + cq] = (uint16_t)bi[j];
            }
            if (!ok) break;
            named_sync(1, kCons);                     // every block's index is staged
            if (cq == 0 && live) {
                const int64_t orow = p.map(r);
                BitWriter wr(p.codes, orow * (int64_t)R);
                const uint4 *row = reinterpret_cast<const uint4 *>(idx_s + t * NB);
#pragma unroll
                for (int w4 = 0; w4 < NB / 8; ++w4) {
                    const uint4 v = row[w4];
                    const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        wr.put(nu > 0.f ? (ws[q] & 0xFFFFu) : 0u, p.B);
                        wr.put(nu > 0.f ? (ws[q] >> 16) : 0u, p.B);
                    }
                }
                wr.flush();
                p.nu[orow] = nu;
                if (!finite) atomicOr(p.flags, (uint32_t)FQ_FLAG_NONFINITE);
            }
        }
        if (!ok && tid == 0) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
        // An x tile still in flight after a timeout lands before the CTA exits.
        if (!ok && tid == 0 && x_issued > x_done) mbar_wait(bar_x, (x_issued - 1) & 1, 1000000ull);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base, 512);
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
    p.C = ctx->C;
    p.nu = nu;
    p.codes = codes;
    p.flags = ctx->flags;
    const int64_t ntiles = (M + kRows - 1) / kRows;
    const int64_t grid = ntiles < ctx->kq_max_ctas ? ntiles : ctx->kq_max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, encode_kq_tc<D, K, NBH, NT>, tm, p);
}

template <int D, int K, int NBH, int NT>
cudaError_t prep_kq(fq_ctx *ctx) {
    using L = KQ<D, K, NBH, NT>;
    static_assert(L::kBytes <= kSmemBudget, "shared memory budget");
    static_assert(L::NB % NBH == 0, "passes");
    cudaError_t e = cudaFuncSetAttribute(encode_kq_tc<D, K, NBH, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kq_tc<D, K, NBH, NT>, kThreads, L::kBytes);
    if (e != cudaSuccess) return e;
    // TMEM: each resident CTA holds all 512 columns of its SM.
    if (per_sm > 1) per_sm = 1;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ctx->kq_max_ctas = per_sm * ctx->num_sms;
    return cudaSuccess;
}

}  // namespace

bool kq_tc_supported(const fq_ctx *ctx) {
    CUtensorMap probe;
    const bool shape = (ctx->d == 64 && ctx->k == 4) || (ctx->d == 128 && ctx->k == 8) ||
                       (ctx->d == 64 && ctx->k == 8) || (ctx->d == 128 && ctx->k == 4);
    return shape && ctx->N >= 256 && ctx->N % 256 == 0 && ctx->N <= 65536 &&
           encode_rows_tensor_map(&probe, ctx->Pi, 128, ctx->d);
}

// Codebook rows as B operands: [ch, ch, cl, hh, hl, 2^10, 2^10, 0...] per codeword (k-wide groups), in the
// K-major no-swizzle layout: codeword n, 16-byte chunk kc of its row at
// (n / 8) * (KP / 8) * 128 + kc * 128 + (n % 8) * 16, so any run of whole 8-codeword groups (a
// 256-codeword tile) is contiguous.
cudaError_t prepare_kq_tc(fq_ctx *ctx) {
    const int N = ctx->N, k = ctx->k, d = ctx->d;
    const int KP = (3 * k + 4 <= 16) ? 16 : 32;
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
        row[3 * k + 2] = __float2half_rn(kOpScale);   // times the A row's 2^10 |u_b|^2 halves
        row[3 * k + 3] = __float2half_rn(kOpScale);
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
    // Codeword tiles of 256: the widest MMA.
    if (d == 64 && k == 4) return prep_kq<64, 4, 8, 256>(ctx);
    if (d == 64 && k == 8) return prep_kq<64, 8, 8, 256>(ctx);
    if (d == 128 && k == 4) return prep_kq<128, 4, 8, 256>(ctx);
    return prep_kq<128, 8, 8, 256>(ctx);
}

cudaError_t launch_encode_kq_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                uint32_t *codes, cudaStream_t s) {
    if (ctx->d == 64 && ctx->k == 4) return launch_kq<64, 4, 8, 256>(ctx, x, M, map, nu, codes, s);
    if (ctx->d == 64 && ctx->k == 8) return launch_kq<64, 8, 8, 256>(ctx, x, M, map, nu, codes, s);
    if (ctx->d == 128 && ctx->k == 4) return launch_kq<128, 4, 8, 256>(ctx, x, M, map, nu, codes, s);
    return launch_kq<128, 8, 8, 256>(ctx, x, M, map, nu, codes, s);
}

}  // namespace fq
