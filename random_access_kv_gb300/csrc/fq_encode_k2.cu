// Tensor-core block encoder for k = 2 [FibQuant §2.3, encoder; §2.2, the k = 2 planar codebook].
//
// Per CTA: NG row groups of 128 threads, one thread per vector (= TMEM lane), looping over
// 128-row tiles of x:
//   1. TMA loads the x tile (fp16, 128-byte swizzle) into shared memory.
//   2. One thread issues tcgen05.mma: Y = X [Pi_hi + Pi_lo]^T into a TMEM fp32 accumulator.
//      Pi is carried as two fp16 halves of 2^12 Pi (hi = fp16(2^12 Pi), lo = fp16(2^12 Pi - hi)):
//      fp16 x times fp16 halves are exact products, summed in fp32, so the rotation keeps about
//      fp32 accuracy while running on the tensor pipe.
//   3. Meanwhile every thread computes nu = |x| of its row from the shared-memory tile.
//   4. Every thread reads its row of Y from TMEM, forms u = Y / (2^12 nu) block by block and
//      finds each block's nearest codeword exactly. A 128 x 128 grid over the block plane lists,
//      per cell, every codeword that can be nearest to some point of the cell (built on the host
//      from exact box-distance bounds), at most four per cell word. The common path is
//      branch-free: cell lookup, then the listed candidates compared by squared difference
//      |u_b - c|^2, ties to the lowest index. Cells with more candidates, and a ring of cells
//      around the grid that catches points outside it, are marked; marked blocks are redone
//      afterwards by squared difference over an overflow list or the whole codebook.
//   5. Indices are packed LSB-first at the record's fixed bit address; nu is stored.
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

constexpr int kGrid = 128;                 // grid cells per axis inside the ring
constexpr int kGridR = kGrid + 2;          // with the ring of marker cells
constexpr int kTileRows = 128;
constexpr float kPiScale = 4096.f;         // 2^12: keeps the fp16 low half of Pi out of subnormals
constexpr int kOvfSlots = 64;              // cells with 5..12 candidates
constexpr int kOvfMax = 12;
constexpr int kCellBytes = (kGridR * kGridR * 4 + 15) & ~15;
constexpr float kMagic = 12582912.f;       // 1.5 * 2^23: adding it rounds to an integer held in the low bits
constexpr int kMagicBits = 0x4B400000;

template <int D, int NG, int NBUF>
struct Layout {
    static constexpr int kPiPart = D * D * 2;                    // bytes of one fp16 half of Pi
    static constexpr int kXTile = kTileRows * D * 2;             // bytes of one x tile
    static constexpr int oPi = 0;
    static constexpr int oX = oPi + 2 * kPiPart;
    static constexpr int oGrid = oX + NG * NBUF * kXTile;
    static constexpr int oOvf = oGrid + kCellBytes;
    static constexpr int oCw = oOvf + kOvfSlots * 16;
    static constexpr int oBar = oCw + 256 * 8;
    static constexpr int kBars = 2 + NG * NBUF + NG;
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;             // + alignment slack
    static constexpr uint32_t kTmemCols = (NG * D <= 32) ? 32 : (NG * D <= 64) ? 64 : (NG * D <= 128) ? 128
                                          : (NG * D <= 256) ? 256 : 512;
};

struct K2Params {
    int64_t M;
    RowMap map;
    int N, B;
    const uint8_t *pi_split;   // [2][D*D] fp16, pre-swizzled
    const uint32_t *tables;    // kCellBytes of cell words, then [kOvfSlots][4] overflow slots
    const float2 *cw;          // [N] codewords
    float gscale, goffs;
    float *nu;
    uint32_t *codes;
    uint32_t *flags;
};

__device__ __forceinline__ void diff_score(float u0, float u1, float2 c, uint32_t n, float &best, uint32_t &bi) {
    const float e0 = u0 - c.x, e1 = u1 - c.y;
    const float s = fmaf(e1, e1, e0 * e0);
    if (s < best) {
        best = s;
        bi = n;
    }
}

// Slow path for a marked cell: its overflow slot, or (slot 0xFF: ring cell or no slot left)
// the whole codebook, compared by squared difference.
__device__ __noinline__ uint32_t marked_cell(float u0, float u1, uint32_t e, const uint4 *ovf, const float2 *cw,
                                             int N) {
    const uint32_t slot = (e >> 8) & 0xFFu;
    float best = INFINITY;
    uint32_t bi = 0;
    if (slot >= (uint32_t)kOvfSlots) {
        for (int n = 0; n < N; ++n) diff_score(u0, u1, cw[n], (uint32_t)n, best, bi);
        return bi;
    }
    const uint4 o = ovf[slot];
    for (uint32_t q = 0; q < o.x; ++q) {
        const uint32_t w = q < 4 ? o.y : (q < 8 ? o.z : o.w);
        const uint32_t n = (w >> (8 * (q & 3))) & 0xFFu;
        diff_score(u0, u1, cw[n], n, best, bi);
    }
    return bi;
}

// Loads the float2 at shared address `addr` into v when p holds; otherwise v keeps its value.
// Predicated rather than branched, so that the blocks of a chunk stay independent instruction
// streams, and lanes that skip the load issue no shared-memory wavefront.
__device__ __forceinline__ void ld_shared_f2_if(bool p, uint32_t addr, float2 &v) {
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q ld.shared.v2.f32 {%0, %1}, [%2];\n\t}"
        : "+f"(v.x), "+f"(v.y)
        : "r"(addr), "r"((uint32_t)p));
}

__device__ __forceinline__ float sqdiff(float u0, float u1, float2 c) {
    const float e0 = u0 - c.x, e1 = u1 - c.y;
    return fmaf(e1, e1, e0 * e0);
}

// Candidate scoring of one block by squared difference, branch-free. Returns the index; sets
// `marked` for marker cells (first byte above last byte: impossible for a real entry, whose bytes
// ascend and are padded with the first). A padded slot repeats the first candidate, so its load is
// skipped and its score equals the first one, which a strict comparison never prefers; a
// single-candidate cell reads no codeword at all.
__device__ __forceinline__ uint32_t fast_block(float a0, float a1, float s, float sg, float gom,
                                               const uint32_t *grid, uint32_t cw_base, uint32_t &e_out,
                                               bool &marked) {
    const float lo = kMagic, hi = kMagic + (float)(kGridR - 1);
    const float gx = fminf(fmaxf(fmaf(a0, sg, gom), lo), hi);
    const float gy = fminf(fmaxf(fmaf(a1, sg, gom), lo), hi);
    const int cell = (__float_as_int(gy) - kMagicBits) * kGridR + (__float_as_int(gx) - kMagicBits);
    const uint32_t e = grid[cell];
    e_out = e;
    const float u0 = a0 * s, u1 = a1 * s;
    const uint32_t b0 = e & 0xFFu, b1 = (e >> 8) & 0xFFu, b2 = (e >> 16) & 0xFFu, b3 = e >> 24;
    marked = b0 > b3;
    float2 c0 = make_float2(0.f, 0.f);
    ld_shared_f2_if(b1 != b0, cw_base + 8u * b0, c0);
    float2 c1 = c0, c2 = c0, c3 = c0;
    ld_shared_f2_if(b1 != b0, cw_base + 8u * b1, c1);
    ld_shared_f2_if(b2 != b0, cw_base + 8u * b2, c2);
    ld_shared_f2_if(b3 != b0, cw_base + 8u * b3, c3);
    float best = sqdiff(u0, u1, c0);
    uint32_t bi = b0;
    const float s1 = sqdiff(u0, u1, c1), s2 = sqdiff(u0, u1, c2), s3 = sqdiff(u0, u1, c3);
    bi = s1 < best ? b1 : bi;
    best = fminf(best, s1);
    bi = s2 < best ? b2 : bi;
    best = fminf(best, s2);
    bi = s3 < best ? b3 : bi;
    return bi;
}

// BS = log2 N when it divides 32 (records then hold whole 32/BS-index words: packed in
// registers and stored as words); BS = 0 packs a run-time B through the bit writer.
template <int D, int NG, int NBUF, int BS>
__global__ void __launch_bounds__(NG * 128, 1)
encode_k2_tc(const __grid_constant__ CUtensorMap xmap, const K2Params p) {
    using L = Layout<D, NG, NBUF>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *pi = sm + L::oPi;
    uint32_t *grid = reinterpret_cast<uint32_t *>(sm + L::oGrid);
    uint4 *ovf = reinterpret_cast<uint4 *>(sm + L::oOvf);
    float2 *cw = reinterpret_cast<float2 *>(sm + L::oCw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
    uint64_t *bar_pi = bars, *bar_grid = bars + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oTmem);

    const int tid = threadIdx.x;
    const int g = tid / 128;              // row group
    const int t = tid % 128;              // row within the tile = TMEM lane
    const int wq = t / 32;                // lane quarter of this warp
    uint64_t *bar_load = bars + 2 + g * NBUF;
    uint64_t *bar_mma = bars + 2 + NG * NBUF + g;
    uint8_t *xbuf0 = sm + L::oX + (g * NBUF) * L::kXTile;

    const int64_t ntiles = (p.M + kTileRows - 1) / kTileRows;
    const int64_t gstride = (int64_t)gridDim.x * NG;
    const int64_t first = (int64_t)blockIdx.x * NG + g;

    if (tid == 0) {
        for (int i = 0; i < L::kBars; ++i) mbar_init(bars + i, 1);
        fence_barrier_init();
    }
    if (tid < 32) tmem_alloc(tmem_slot, L::kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Shared tables, each CTA its own copy by plain bulk copies. Pi has its own barrier so that
    // the first rotation can start while the candidate grid is still arriving.
    if (tid == 0) {
        prefetch_tensormap(&xmap);
        const uint32_t cw_bytes = (uint32_t)p.N * 8u;
        const uint32_t tab_bytes = kCellBytes + kOvfSlots * 16u;
        mbar_arrive_expect_tx(bar_pi, 2u * L::kPiPart);
        bulk_g2s(pi, p.pi_split, 2u * L::kPiPart, bar_pi);
        mbar_arrive_expect_tx(bar_grid, tab_bytes + cw_bytes);
        bulk_g2s(grid, p.tables, tab_bytes, bar_grid);
        bulk_g2s(cw, p.cw, cw_bytes, bar_grid);
    }
    // Tables are in flight; x and the outputs may belong to the previous kernel in the stream.
    griddep_launch_dependents();
    griddep_wait();
    // Loads and MMA commits issued and waited for, per barrier (every thread of a group keeps the
    // same counts, the conditions being uniform over the group): after a timeout the cleanup
    // waits on the parity of the phase still in flight.
    uint32_t ld_issued[NBUF], ld_done[NBUF], mma_issued = 0, mma_done = 0;
#pragma unroll
    for (int i = 0; i < NBUF; ++i) ld_issued[i] = ld_done[i] = 0;
    if (first < ntiles) ld_issued[0] = 1;
    // Each row group's first x tile.
    if (t == 0 && first < ntiles) {
        mbar_arrive_expect_tx(bar_load, (uint32_t)L::kXTile);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(xbuf0 + kb * 16384, &xmap, kb * 64, (int)(first * kTileRows), bar_load);
    }
    bool ok = named_sync_and(1 + g, 128, mbar_wait(bar_pi, 0));

    const uint32_t idesc = idesc_f16_f32(128, D);
    const uint32_t tmem_acc = tmem_base + (uint32_t)(g * D);
    const uint32_t pi_hi = smem_addr(pi), pi_lo = pi_hi + L::kPiPart;
    const int R = (D / 2) * p.B;
    // +1: cell (i, j) sits at (i+1, j+1) inside the ring. goffs is an integer, so this is exact.
    const float gom = p.goffs + 1.0f + kMagic;
    const uint32_t cw_base = smem_addr(cw);

    int64_t it = 0;
    for (int64_t tile = first; tile < ntiles && ok; tile += gstride, ++it) {
        const int buf = (int)(it % NBUF);
        uint8_t *xt = xbuf0 + buf * L::kXTile;
        ok = named_sync_and(1 + g, 128, mbar_wait(bar_load + buf, (uint32_t)((it / NBUF) & 1)));
        if (!ok) break;
        ++ld_done[buf];
        const int64_t next = tile + gstride;
        if (NBUF == 2 && next < ntiles) ++ld_issued[buf ^ 1];
        if (NBUF == 2 && t == 0 && next < ntiles) {
            // The other buffer's last readers (tile it-1: its MMA and the nu loads) finished
            // before the group barrier that closed iteration it-1.
            uint8_t *xn = xbuf0 + (buf ^ 1) * L::kXTile;
            mbar_arrive_expect_tx(bar_load + (buf ^ 1), (uint32_t)L::kXTile);
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb)
                tma_load_2d(xn + kb * 16384, &xmap, kb * 64, (int)(next * kTileRows), bar_load + (buf ^ 1));
        }
        if (t == 0) {
            tc_fence_after();
            const uint32_t xa = smem_addr(xt);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t pb = half ? pi_lo : pi_hi;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32);
                    const uint32_t boff = (uint32_t)((kk >> 2) * (D * 128) + (kk & 3) * 32);
                    mma_f16(tmem_acc, sdesc_sw128(xa + koff), sdesc_sw128(pb + boff), idesc,
                            (half | kk) ? 1u : 0u);
                }
            }
            mma_commit(bar_mma);
        }
        ++mma_issued;
        // nu of this thread's row, from the swizzled tile (chunk c of row t sits at chunk c ^ (t % 8)).
        float ss = 0.f;
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = *reinterpret_cast<const uint4 *>(xt + kb * 16384 + t * 128 + ((c ^ (t & 7)) << 4));
                const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __half22float2(h[q]);
                    ss = fmaf(f.x, f.x, ss);
                    ss = fmaf(f.y, f.y, ss);
                }
            }
        }
        ok = named_sync_and(1 + g, 128, mbar_wait(bar_mma, (uint32_t)(it & 1)) && (it > 0 || mbar_wait(bar_grid, 0)));
        if (!ok) break;
        ++mma_done;
        tc_fence_after();

        const int64_t r = tile * kTileRows + t;
        const bool live = r < p.M;
        // fp16 inputs are bounded by 65504, so ss is finite unless an element is Inf or NaN.
        const bool finite = isfinite(ss);
        const float nu = finite ? sqrtf(ss) : 0.f;
        const float s = nu > 0.f ? (1.0f / kPiScale) / nu : 0.f;
        const float sg = s * p.gscale;
        const bool zero = !(nu > 0.f);
        const int64_t orow = live ? p.map(r) : 0;
        constexpr int W = BS ? (D / 2) * BS / 32 : 1;   // record words (static packing)
        uint32_t words[W];
#pragma unroll
        for (int w = 0; w < W; ++w) words[w] = 0u;
        BitWriter wr(p.codes, orow * (int64_t)R);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            float a[16];
            tmem_ld16(tmem_acc + ((uint32_t)(32 * wq) << 16) + (uint32_t)(16 * c), a);
            tmem_wait_ld();
            uint32_t idx[8], ent[8];
            uint32_t marks = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                bool m;
                idx[j] = fast_block(a[2 * j], a[2 * j + 1], s, sg, gom, grid, cw_base, ent[j], m);
                marks |= (uint32_t)m << j;
            }
            if (marks && live && !zero) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if ((marks >> j) & 1u) idx[j] = marked_cell(a[2 * j] * s, a[2 * j + 1] * s, ent[j], ovf, cw, p.N);
            }
            if constexpr (BS != 0) {
                // 8 indices of BS bits: bits [c * 8 BS, (c+1) * 8 BS) of the record.
                uint64_t acc = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) acc |= (uint64_t)(zero ? 0u : idx[j]) << (j * BS);
                constexpr int kBits = 8 * BS;
                const int bit0 = c * kBits;
                if constexpr (kBits >= 32) {
#pragma unroll
                    for (int q = 0; q < kBits / 32; ++q) words[bit0 / 32 + q] = (uint32_t)(acc >> (32 * q));
                } else {
                    words[bit0 / 32] |= (uint32_t)acc << (bit0 % 32);
                }
            } else {
                if (live) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) wr.put(zero ? 0u : idx[j], p.B);
                }
            }
        }
        if (live) {
            if constexpr (BS != 0) {
                uint32_t *dst = p.codes + orow * (int64_t)W;
                if ((W % 4) == 0 && ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0)) {
#pragma unroll
                    for (int w = 0; w < W; w += 4)
                        *reinterpret_cast<uint4 *>(dst + w) = make_uint4(words[w], words[w + 1], words[w + 2], words[w + 3]);
                } else {
#pragma unroll
                    for (int w = 0; w < W; ++w) dst[w] = words[w];
                }
            } else {
                wr.flush();
            }
            p.nu[orow] = nu;
            if (!finite) atomicOr(p.flags, (uint32_t)FQ_FLAG_NONFINITE);
        }
        tc_fence_before();
        named_sync(1 + g, 128);
        if (NBUF == 1 && next < ntiles) ++ld_issued[0];
        if (NBUF == 1 && t == 0 && next < ntiles) {
            mbar_arrive_expect_tx(bar_load, (uint32_t)L::kXTile);
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb)
                tma_load_2d(xbuf0 + kb * 16384, &xmap, kb * 64, (int)(next * kTileRows), bar_load);
        }
    }
    if (!ok && t == 0) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
    // A CTA without tiles still waits for the tables, so that nothing is in flight into it.
    if (it == 0) mbar_wait(bar_grid, 0);
    __syncthreads();
    if (!ok) {
        // Give in-flight copies and MMAs a bounded chance to land before the CTA's memory goes
        // away: wait (briefly) on the phase each barrier still has outstanding.
        mbar_wait(bar_pi, 0, 1000000ull);
        mbar_wait(bar_grid, 0, 1000000ull);
        for (int i = 0; i < NBUF; ++i)
            if (ld_issued[i] > ld_done[i]) mbar_wait(bar_load + i, (ld_issued[i] - 1u) & 1u, 1000000ull);
        if (mma_issued > mma_done) mbar_wait(bar_mma, (mma_issued - 1u) & 1u, 1000000ull);
    }
    tc_fence_after();
    if (tid < 32) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int D, int NG, int NBUF, int BS>
cudaError_t launch_k2(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu, uint32_t *codes,
                      cudaStream_t s) {
    using L = Layout<D, NG, NBUF>;
    CUtensorMap tm;
    if (!encode_rows_tensor_map(&tm, x, M, D)) return cudaErrorInvalidValue;
    K2Params p;
    p.M = M;
    p.map = map;
    p.N = ctx->N;
    p.B = ctx->B;
    p.pi_split = ctx->pi_split;
    p.tables = ctx->grid2;
    p.cw = reinterpret_cast<const float2 *>(ctx->C);
    p.gscale = ctx->g_scale;
    p.goffs = ctx->g_offs;
    p.nu = nu;
    p.codes = codes;
    p.flags = ctx->flags;
    const int64_t ntiles = (M + kTileRows - 1) / kTileRows;
    int64_t grid = (ntiles + NG - 1) / NG;
    if (grid > ctx->k2_max_ctas) grid = ctx->k2_max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NG * 128);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, encode_k2_tc<D, NG, NBUF, BS>, tm, p);
}

template <int D, int NG, int NBUF, int BS>
cudaError_t prep_k2(fq_ctx *ctx) {
    using L = Layout<D, NG, NBUF>;
    static_assert(L::kBytes <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(encode_k2_tc<D, NG, NBUF, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kBytes);
    if (e != cudaSuccess) return e;
    // The persistent grid: as many CTAs as can be resident at once (one per SM).
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_k2_tc<D, NG, NBUF, BS>, NG * 128, L::kBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ctx->k2_max_ctas = per_sm * ctx->num_sms;
    return cudaSuccess;
}

// Static packing when B divides 32 (B = 1, 2, 4, 8); the generic bit writer otherwise.
template <int D, int NG, int NBUF>
cudaError_t dispatch_prep(fq_ctx *ctx) {
    switch (ctx->B) {
        case 1: return prep_k2<D, NG, NBUF, 1>(ctx);
        case 2: return prep_k2<D, NG, NBUF, 2>(ctx);
        case 4: return prep_k2<D, NG, NBUF, 4>(ctx);
        case 8: return prep_k2<D, NG, NBUF, 8>(ctx);
        default: return prep_k2<D, NG, NBUF, 0>(ctx);
    }
}

template <int D, int NG, int NBUF>
cudaError_t dispatch_launch(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu, uint32_t *codes,
                            cudaStream_t s) {
    switch (ctx->B) {
        case 1: return launch_k2<D, NG, NBUF, 1>(ctx, x, M, map, nu, codes, s);
        case 2: return launch_k2<D, NG, NBUF, 2>(ctx, x, M, map, nu, codes, s);
        case 4: return launch_k2<D, NG, NBUF, 4>(ctx, x, M, map, nu, codes, s);
        case 8: return launch_k2<D, NG, NBUF, 8>(ctx, x, M, map, nu, codes, s);
        default: return launch_k2<D, NG, NBUF, 0>(ctx, x, M, map, nu, codes, s);
    }
}

}  // namespace

// Candidate grid for the k = 2 search. Cell (i, j) holds every codeword that is nearest to some
// point of the cell's box (widened by a small margin against rounding of the cell index):
// c_n qualifies iff its distance to the box is at most min_m (distance from c_m to the box's
// farthest corner), a bound that holds for every point of the box. Layout: a (kGrid + 2)^2 array
// of cell words whose outer ring marks points outside the grid, then kOvfSlots overflow slots of
// four words (count, then up to twelve index bytes).
static void build_k2_grid(const float *C, int N, int d, std::vector<uint32_t> &tab, float &gscale,
                          float &goffs) {
    // Grid half-width: the larger of the codebook's extent and the radius that a block of a
    // Haar-uniform unit vector exceeds with probability below 1e-7 (|u_b|^2 ~ Beta(1, d/2 - 1)).
    double cmax = 0;
    for (int i = 0; i < 2 * N; ++i) cmax = fmax(cmax, fabs((double)C[i]));
    const double rq = sqrt(1.0 - pow(1e-7, 1.0 / (0.5 * d - 1.0)));
    const double Rg = fmax(1.05 * cmax, rq);
    const double eps = 1e-3 * (2.0 * Rg / kGrid);
    // The device rounds u * gscale + goffs to the nearest integer. goffs is an integer so that
    // goffs + 1 + 1.5 * 2^23 (the device folds the ring offset and the rounding constant into one
    // addend) stays exact in fp32; cell i then covers u * gscale + goffs in [i - 1/2, i + 1/2],
    // and the 128 cells cover [-Rg, Rg]. Cell bounds follow from the fp32 constants.
    goffs = (float)(kGrid / 2);
    gscale = (float)((0.5 * kGrid - 0.5) / Rg);
    const double gs = gscale, go = goffs;
    const size_t cell_words = kCellBytes / 4;
    const uint32_t ring = 0xFFu | (0xFFu << 8);          // marker, no slot: scan everything
    tab.assign(cell_words + 4 * kOvfSlots, 0u);
    for (int iy = 0; iy < kGridR; ++iy)
        for (int ix = 0; ix < kGridR; ++ix) tab[(size_t)iy * kGridR + ix] = ring;
    std::vector<int> cand;
    int slots = 0;
    for (int iy = 0; iy < kGrid; ++iy) {
        const double y0 = (iy - 0.5 - go) / gs - eps, y1 = (iy + 0.5 - go) / gs + eps;
        for (int ix = 0; ix < kGrid; ++ix) {
            const double x0 = (ix - 0.5 - go) / gs - eps, x1 = (ix + 0.5 - go) / gs + eps;
            double U2 = INFINITY;
            for (int m = 0; m < N; ++m) {
                const double cx = C[2 * m], cy = C[2 * m + 1];
                const double fx = fmax(fabs(cx - x0), fabs(cx - x1)), fy = fmax(fabs(cy - y0), fabs(cy - y1));
                U2 = fmin(U2, fx * fx + fy * fy);
            }
            cand.clear();
            for (int n = 0; n < N; ++n) {
                const double cx = C[2 * n], cy = C[2 * n + 1];
                const double dx = fmax(0.0, fmax(x0 - cx, cx - x1)), dy = fmax(0.0, fmax(y0 - cy, cy - y1));
                if (dx * dx + dy * dy <= U2 * (1.0 + 1e-12)) cand.push_back(n);
            }
            uint32_t &cell = tab[(size_t)(iy + 1) * kGridR + (ix + 1)];
            if (cand.size() > 4) {
                uint32_t slot = 0xFFu;
                if (cand.size() <= (size_t)kOvfMax && slots < kOvfSlots) {
                    slot = (uint32_t)slots++;
                    uint32_t *o = &tab[cell_words + 4 * slot];
                    o[0] = (uint32_t)cand.size();
                    for (size_t q = 0; q < cand.size(); ++q) o[1 + q / 4] |= (uint32_t)cand[q] << (8 * (q % 4));
                }
                cell = 0xFFu | (slot << 8);            // first byte 0xFF above last byte 0x00: marker
                continue;
            }
            uint32_t e = 0;
            for (int q = 0; q < 4; ++q) e |= (uint32_t)cand[q < (int)cand.size() ? q : 0] << (8 * q);
            cell = e;
        }
    }
}

// Pi (or Pi^T) as two fp16 halves of scale * src, each in the K-major 128-byte-swizzle layout the
// MMA reads as its B operand: B[n][k] = src[n][k]; element (n, k) lives in K-block k / 64,
// row n (128 bytes), 16-byte chunk (k % 64) / 8 XOR (n % 8).
void split_operand_sw128(const float *src, int d, float scale, std::vector<uint16_t> &out) {
    const size_t part = (size_t)d * d;
    out.assign(2 * part, 0);
    for (int n = 0; n < d; ++n) {
        for (int k = 0; k < d; ++k) {
            const float v = src[(size_t)n * d + k] * scale;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            const int kb = k / 64, kin = k % 64;
            const size_t byte = (size_t)kb * d * 128 + (size_t)n * 128 + (size_t)(((kin / 8) ^ (n % 8)) * 16) +
                                (size_t)(kin % 8) * 2;
            memcpy(&out[byte / 2], &hi, 2);
            memcpy(&out[part + byte / 2], &lo, 2);
        }
    }
}

bool encode_rows_tensor_map(CUtensorMap *tm, const void *x, int64_t M, int D) {
    // The driver entry point, looked up once; a function-local static is initialised once even
    // when contexts on several host threads encode at the same time.
    static const PFN_cuTensorMapEncodeTiled_v12000 enc = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000)ptr;
        return nullptr;
    }();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)M};
    cuuint64_t gstride[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kTileRows};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(x), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool k2_tc_supported(const fq_ctx *ctx) {
    CUtensorMap probe;
    return ctx->k == 2 && (ctx->d == 64 || ctx->d == 128) && ctx->N <= 256 &&
           encode_rows_tensor_map(&probe, ctx->Pi, 128, ctx->d);
}

cudaError_t prepare_k2_tc(fq_ctx *ctx) {
    std::vector<uint32_t> tab;
    std::vector<uint16_t> pis;
    std::vector<float> C((size_t)ctx->N * 2);
    cudaError_t e = cudaMemcpy(C.data(), ctx->C, C.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    std::vector<float> P((size_t)ctx->d * ctx->d);
    e = cudaMemcpy(P.data(), ctx->Pi, P.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    build_k2_grid(C.data(), ctx->N, ctx->d, tab, ctx->g_scale, ctx->g_offs);
    split_operand_sw128(P.data(), ctx->d, kPiScale, pis);
    e = cudaMalloc((void **)&ctx->grid2, tab.size() * 4);
    if (e == cudaSuccess) e = cudaMemcpy(ctx->grid2, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc((void **)&ctx->pi_split, pis.size() * 2);
    if (e == cudaSuccess) e = cudaMemcpy(ctx->pi_split, pis.data(), pis.size() * 2, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return e;
    if (ctx->d == 64) return dispatch_prep<64, 4, 2>(ctx);
    return dispatch_prep<128, 2, 1>(ctx);
}

cudaError_t launch_encode_k2_tc(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                uint32_t *codes, cudaStream_t s) {
    if (ctx->d == 64) return dispatch_launch<64, 4, 2>(ctx, x, M, map, nu, codes, s);
    return dispatch_launch<128, 2, 1>(ctx, x, M, map, nu, codes, s);
}

}  // namespace fq
