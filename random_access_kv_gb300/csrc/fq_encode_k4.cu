// Candidate-grid block encoder for k = 4 [FibQuant §2.3, encoder: normalise, rotate, nearest
// codeword of each 4-dimensional block, fixed-address packing].
//
// Per CTA: NG row groups of 128 threads, one thread per vector (= TMEM lane), looping over
// 128-row tiles of x, as the k = 2 encoder does:
//   1. TMA loads the x tile (fp16, 128-byte swizzle) into shared memory.
//   2. One thread issues tcgen05.mma: Y = X [Pi_hi + Pi_lo]^T into a TMEM fp32 accumulator
//      (fp16 halves of 2^12 Pi: exact products summed in fp32).
//   3. Meanwhile every thread computes nu = |x| of its row from the shared-memory tile.
//   4. Every thread reads its row of Y from TMEM, 16 columns (4 blocks) at a time, and forms
//      u = Y / (2^12 nu). Each block's four coordinates pick a cell of a G^4 candidate grid
//      (a lattice index per coordinate, one fused multiply-add rounded to an integer, mapped to
//      a coarse index by a table that every lane reads from its own copy, without bank conflicts).
//      The cell's 32-byte record, read through the read-only cache from a table that stays in
//      L2, lists every codeword that can be nearest to some point of the cell (built on the host
//      from exact box bounds, see fq_grid4.h). The listed codewords are compared by squared
//      difference |u_b - c|^2 in fp32 (packed two-lane arithmetic), in ascending index order,
//      ties to the lowest index. Blocks outside the grid, or in a cell that lists more than
//      fifteen codewords, are redone afterwards: over the cell's overflow list or the whole
//      codebook.
// At d = 64 a CTA runs five row groups with one x tile each: more warps hide more of the record
// loads' latency, and a second tile per group would leave the record loads, which pass through
// L1, too little of it (measured slower).
//   5. Indices are packed LSB-first at the record's fixed bit address; nu is stored.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <vector>

#include "fq_bits.cuh"
#include "fq_grid4.h"
#include "fq_internal.h"
#include "fq_sm100.cuh"

namespace fq {

namespace {

using namespace sm100;

constexpr int kTileRows = 128;
constexpr float kPiScale = 4096.f;         // 2^12: keeps the fp16 low half of Pi out of subnormals
constexpr int kAxisF = 512;                // lattice entries per axis (Grid4::F)
constexpr int kAxisBytes = kAxisF * 64;    // the coarse-index table as uint16, one copy per lane
constexpr int kSlots = 15;                 // codeword slots of a cell record (32 bytes)
constexpr float kMagic = 12582912.f;       // 1.5 * 2^23: adding it rounds to an integer held in the low bits
constexpr int kMagicBits = 0x4B400000;
constexpr int kMaxN = 4096;                // the codebook lives in shared memory

template <int D, int NG, int NBUF>
struct Layout {
    static constexpr int kPiPart = D * D * 2;                    // bytes of one fp16 half of Pi
    static constexpr int kXTile = kTileRows * D * 2;             // bytes of one x tile
    static constexpr int oPi = 0;
    static constexpr int oX = oPi + 2 * kPiPart;
    static constexpr int oAxis = oX + NG * NBUF * kXTile;
    static constexpr int oBar = oAxis + kAxisBytes;
    static constexpr int kBars = 2 + NG * NBUF + NG;
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int oCb = (oTmem + 16 + 15) & ~15;          // then N x 16 bytes of codewords
    static constexpr uint32_t kTmemCols = (NG * D <= 32) ? 32 : (NG * D <= 64) ? 64 : (NG * D <= 128) ? 128
                                          : (NG * D <= 256) ? 256 : 512;
    static constexpr int bytes(int N) { return oCb + N * 16 + 1024; }   // + alignment slack
};

struct K4Params {
    int64_t M;
    RowMap map;
    int N, B, G;
    float fs;                  // lattice index = round(u * fs + fo)
    int fo;
    const uint8_t *pi_split;   // [2][D*D] fp16, pre-swizzled
    const uint4 *cells;        // [G^4][2] records: count, then up to 15 ascending indices (uint16)
    const uint16_t *pool;      // overflow lists
    const uint8_t *axis;       // [kAxisF] lattice-to-coarse table
    const float4 *ncb;         // [N] negated codewords
    float *nu;
    uint32_t *codes;
    uint32_t *flags;
};

// |u - c|^2 with c given negated: two packed adds, a packed multiply and a packed fused
// multiply-add, then one add: (e0^2 + e2^2) + (e1^2 + e3^2).
__device__ __forceinline__ float dist4(float2 u01, float2 u23, float4 nc) {
    const float2 e01 = __fadd2_rn(u01, make_float2(nc.x, nc.y));
    const float2 e23 = __fadd2_rn(u23, make_float2(nc.z, nc.w));
    float2 q = __fmul2_rn(e01, e01);
    q = __ffma2_rn(e23, e23, q);
    return q.x + q.y;
}

// Loads the float4 at shared address `addr` into v when p holds; otherwise v keeps its value.
__device__ __forceinline__ void ld_shared_f4_if(bool p, uint32_t addr, float4 &v) {
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t@q ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w)
        : "r"(addr), "r"((uint32_t)p));
}

// Slot q (0..14) of a record: index e[1 + q] of its sixteen uint16 (ra: e[0..7], rb: e[8..15]).
template <int Q>
__device__ __forceinline__ uint32_t slot(const uint4 &ra, const uint4 &rb) {
    static_assert(Q >= 0 && Q < kSlots, "slot");
    constexpr int e = Q + 1;
    const uint4 &r = e < 8 ? ra : rb;
    const int w = (e % 8) / 2;
    const uint32_t word = w == 0 ? r.x : w == 1 ? r.y : w == 2 ? r.z : r.w;
    return (e & 1) ? word >> 16 : word & 0xFFFFu;
}

// Slow path of a marked block: the cell's overflow list (its offset is the record's second
// word), or, outside the grid, the whole codebook; squared difference, ascending, ties to the
// lowest index.
__device__ __noinline__ uint32_t marked_block(float2 u01, float2 u23, uint4 rec, bool outside, const float4 *ncb,
                                              const uint16_t *pool, int N) {
    float best = INFINITY;
    uint32_t bi = 0;
    if (outside) {
        for (int n = 0; n < N; ++n) {
            const float s = dist4(u01, u23, ncb[n]);
            if (s < best) {
                best = s;
                bi = (uint32_t)n;
            }
        }
        return bi;
    }
    const uint32_t cnt = rec.x & 0xFFFFu;
    const uint16_t *lst = pool + rec.y;
    for (uint32_t q = 0; q < cnt; ++q) {
        const uint32_t n = __ldg(lst + q);
        const float s = dist4(u01, u23, ncb[n]);
        if (s < best) {
            best = s;
            bi = n;
        }
    }
    return bi;
}

// Records are written through the bit writer (whole words plainly, shared boundary words by
// masked atomics), B bits per index.
template <int D, int NG, int NBUF>
__global__ void __launch_bounds__(NG * 128, 1)
encode_k4_grid(const __grid_constant__ CUtensorMap xmap, const K4Params p) {
    using L = Layout<D, NG, NBUF>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *pi = sm + L::oPi;
    uint32_t *axr = reinterpret_cast<uint32_t *>(sm + L::oAxis);
    float4 *ncb = reinterpret_cast<float4 *>(sm + L::oCb);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
    uint64_t *bar_pi = bars, *bar_tab = bars + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oTmem);

    const int tid = threadIdx.x;
    const int g = tid / 128;              // row group
    const int t = tid % 128;              // row within the tile = TMEM lane
    const int wq = t / 32;                // lane quarter of this warp
    const int lane = t % 32;
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
    // The lattice-to-coarse table as uint16, one copy per lane: entry j of lane l at byte
    // 64 j + 2 l, so the 32 lanes of a warp read 32 distinct halves of 16 words (no conflict).
    for (int i = tid; i < kAxisF * 16; i += NG * 128) axr[i] = 0x10001u * (uint32_t)__ldg(p.axis + i / 16);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Shared tables, each CTA its own copy by plain bulk copies; Pi has its own barrier so that
    // the first rotation can start while the codebook is still arriving.
    if (tid == 0) {
        prefetch_tensormap(&xmap);
        mbar_arrive_expect_tx(bar_pi, 2u * L::kPiPart);
        bulk_g2s(pi, p.pi_split, 2u * L::kPiPart, bar_pi);
        mbar_arrive_expect_tx(bar_tab, (uint32_t)p.N * 16u);
        bulk_g2s(ncb, p.ncb, (uint32_t)p.N * 16u, bar_tab);
    }
    // Tables are in flight; x and the outputs may belong to the previous kernel in the stream.
    griddep_launch_dependents();
    griddep_wait();
    // Loads and MMA commits issued and waited for, per barrier (uniform over the group): after a
    // timeout the cleanup waits on the parity of the phase still in flight.
    uint32_t ld_issued[NBUF], ld_done[NBUF], mma_issued = 0, mma_done = 0;
#pragma unroll
    for (int i = 0; i < NBUF; ++i) ld_issued[i] = ld_done[i] = 0;
    if (first < ntiles) ld_issued[0] = 1;
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
    const int R = (D / 4) * p.B;
    const float fom = (float)p.fo + kMagic;          // fo is a small integer: exact
    const uint32_t ax_lane = smem_addr(axr) + 2u * (uint32_t)lane;
    const uint32_t cb_base = smem_addr(ncb);
    const int G = p.G;

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
        ok = named_sync_and(1 + g, 128, mbar_wait(bar_mma, (uint32_t)(it & 1)) && (it > 0 || mbar_wait(bar_tab, 0)));
        if (!ok) break;
        ++mma_done;
        tc_fence_after();

        const int64_t r = tile * kTileRows + t;
        const bool live = r < p.M;
        // fp16 inputs are bounded by 65504, so ss is finite unless an element is Inf or NaN.
        const bool finite = isfinite(ss);
        const float nu = finite ? sqrtf(ss) : 0.f;
        const float s = nu > 0.f ? (1.0f / kPiScale) / nu : 0.f;
        const bool zero = !(nu > 0.f);
        const int64_t orow = live ? p.map(r) : 0;
        BitWriter wr(p.codes, orow * (int64_t)R);
        // Four blocks (16 columns) per step.
#pragma unroll 1
        for (int h = 0; h < D / 16; ++h) {
            uint32_t a[16];
            tmem_ld16_nowait(tmem_acc + ((uint32_t)(32 * wq) << 16) + (uint32_t)(16 * h), a);
            tmem_wait_ld();
            float2 u01[4], u23[4];
            uint4 ra[4], rb[4];
            uint32_t cellv[4], vc[4];
            uint32_t outside = 0, marks = 0, lane_max = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float c0 = __uint_as_float(a[4 * j]) * s, c1 = __uint_as_float(a[4 * j + 1]) * s;
                const float c2 = __uint_as_float(a[4 * j + 2]) * s, c3 = __uint_as_float(a[4 * j + 3]) * s;
                u01[j] = make_float2(c0, c1);
                u23[j] = make_float2(c2, c3);
                const float cf[4] = {c0, c1, c2, c3};
                uint32_t cell = 0, orv = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // Lattice index, clamped to [0, F-1] (negative and NaN fall on an outer entry).
                    const float tq = fmaf(cf[e], p.fs, fom);
                    const uint32_t jl = min((uint32_t)(__float_as_int(tq) - kMagicBits), (uint32_t)(kAxisF - 1));
                    uint32_t cv;
                    asm("ld.shared.u16 %0, [%1];" : "=r"(cv) : "r"(ax_lane + (jl << 6)));
                    cell = cell * (uint32_t)G + cv;
                    orv |= cv;
                }
                const bool out = orv >= 0x80u;                  // an axis fell outside the grid
                cellv[j] = out ? 0u : cell;
                ra[j] = __ldg(p.cells + 2u * cellv[j]);
                rb[j] = make_uint4(0u, 0u, 0u, 0u);
                const uint32_t cnt = ra[j].x & 0xFFFFu;
                const bool mk = out || cnt > (uint32_t)kSlots;
                outside |= (uint32_t)out << j;
                marks |= (uint32_t)mk << j;
                vc[j] = mk ? 0u : cnt;                          // slots this lane compares
                lane_max = max(lane_max, vc[j]);
            }
            const uint32_t wmax = __reduce_max_sync(0xffffffffu, lane_max);
            float best[4];
            uint32_t bi[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                best[j] = INFINITY;
                bi[j] = 0;
            }
            // Slot q of every block, while some lane still has a listed codeword there. A slot
            // past a record's count is neither loaded nor compared. The record's second half
            // (slots 7..14) is read only when some lane needs it.
#define FQ_K4_SLOT(Q)                                                                                  \
    if ((Q) < wmax) {                                                                                  \
        _Pragma("unroll") for (int j = 0; j < 4; ++j) {                                                \
            const uint32_t n = slot<Q>(ra[j], rb[j]);                                                  \
            const bool pj = (uint32_t)(Q) < vc[j];                                                     \
            float4 c = make_float4(0.f, 0.f, 0.f, 0.f);                                                \
            ld_shared_f4_if(pj, cb_base + 16u * n, c);                                                 \
            const float dj = dist4(u01[j], u23[j], c);                                                 \
            const bool better = pj && dj < best[j];                                                    \
            best[j] = better ? dj : best[j];                                                           \
            bi[j] = better ? n : bi[j];                                                                \
        }                                                                                              \
    }
            FQ_K4_SLOT(0)
            FQ_K4_SLOT(1)
            FQ_K4_SLOT(2)
            FQ_K4_SLOT(3)
            FQ_K4_SLOT(4)
            FQ_K4_SLOT(5)
            FQ_K4_SLOT(6)
            if (wmax > 7u) {
#pragma unroll
                for (int j = 0; j < 4; ++j) rb[j] = __ldg(p.cells + 2u * cellv[j] + 1u);
                FQ_K4_SLOT(7)
                FQ_K4_SLOT(8)
                FQ_K4_SLOT(9)
                FQ_K4_SLOT(10)
                FQ_K4_SLOT(11)
                FQ_K4_SLOT(12)
                FQ_K4_SLOT(13)
                FQ_K4_SLOT(14)
            }
#undef FQ_K4_SLOT
            if (marks && live && !zero) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((marks >> j) & 1u)
                        bi[j] = marked_block(u01[j], u23[j], ra[j], (outside >> j) & 1u, ncb, p.pool, p.N);
            }
            if (live) {
#pragma unroll
                for (int j = 0; j < 4; ++j) wr.put(zero ? 0u : bi[j], p.B);
            }
        }
        if (live) {
            wr.flush();
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
    // A CTA without tiles still waits for the codebook, so that nothing is in flight into it.
    if (it == 0) mbar_wait(bar_tab, 0);
    __syncthreads();
    if (!ok) {
        // Give in-flight copies and MMAs a bounded chance to land before the CTA's memory goes
        // away: wait (briefly) on the phase each barrier still has outstanding.
        mbar_wait(bar_pi, 0, 1000000ull);
        mbar_wait(bar_tab, 0, 1000000ull);
        for (int i = 0; i < NBUF; ++i)
            if (ld_issued[i] > ld_done[i]) mbar_wait(bar_load + i, (ld_issued[i] - 1u) & 1u, 1000000ull);
        if (mma_issued > mma_done) mbar_wait(bar_mma, (mma_issued - 1u) & 1u, 1000000ull);
    }
    tc_fence_after();
    if (tid < 32) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int D, int NG, int NBUF>
cudaError_t launch_k4(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu, uint32_t *codes,
                      cudaStream_t s) {
    using L = Layout<D, NG, NBUF>;
    CUtensorMap tm;
    if (!encode_rows_tensor_map(&tm, x, M, D)) return cudaErrorInvalidValue;
    K4Params p;
    p.M = M;
    p.map = map;
    p.N = ctx->N;
    p.B = ctx->B;
    p.G = ctx->k4_G;
    p.fs = ctx->k4_fs;
    p.fo = kAxisF / 2;
    p.pi_split = ctx->pi_split;
    p.cells = reinterpret_cast<const uint4 *>(ctx->k4_cells);
    p.pool = ctx->k4_pool;
    p.axis = ctx->k4_axis;
    p.ncb = reinterpret_cast<const float4 *>(ctx->k4_ncb);
    p.nu = nu;
    p.codes = codes;
    p.flags = ctx->flags;
    const int64_t ntiles = (M + kTileRows - 1) / kTileRows;
    int64_t grid = (ntiles + NG - 1) / NG;
    if (grid > ctx->k4_max_ctas) grid = ctx->k4_max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NG * 128);
    cfg.dynamicSmemBytes = (size_t)L::bytes(ctx->N);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, encode_k4_grid<D, NG, NBUF>, tm, p);
}

template <int D, int NG, int NBUF>
cudaError_t prep_k4(fq_ctx *ctx) {
    using L = Layout<D, NG, NBUF>;
    const int bytes = L::bytes(ctx->N);
    if (bytes > 227 * 1024) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(encode_k4_grid<D, NG, NBUF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         bytes);
    if (e != cudaSuccess) return e;
    // The persistent grid: as many CTAs as can be resident at once (one per SM).
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_k4_grid<D, NG, NBUF>, NG * 128, bytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ctx->k4_max_ctas = per_sm * ctx->num_sms;
    return cudaSuccess;
}

template <typename T>
cudaError_t upload_vec(T **dst, const std::vector<T> &src) {
    cudaError_t e = cudaMalloc((void **)dst, src.size() * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
}

}  // namespace

bool k4_grid_supported(const fq_ctx *ctx) {
    CUtensorMap probe;
    return ctx->k == 4 && (ctx->d == 64 || ctx->d == 128) && ctx->N >= 2 && ctx->N <= kMaxN &&
           encode_rows_tensor_map(&probe, ctx->Pi, 128, ctx->d);
}

cudaError_t prepare_k4_grid(fq_ctx *ctx) {
    const int N = ctx->N, d = ctx->d;
    std::vector<float> C((size_t)N * 4);
    cudaError_t e = cudaMemcpy(C.data(), ctx->C, C.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    Grid4 grid;
    build_grid4(C.data(), N, d, grid);
    if (grid.F != kAxisF || grid.fo != kAxisF / 2 || grid.G > 40) return cudaErrorInvalidValue;
    ctx->k4_G = grid.G;
    ctx->k4_fs = grid.fs;
    std::vector<float> ncb(C.size());
    for (size_t i = 0; i < C.size(); ++i) ncb[i] = -C[i];
    if (!ctx->pi_split) {
        std::vector<float> P((size_t)d * d);
        e = cudaMemcpy(P.data(), ctx->Pi, P.size() * 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return e;
        std::vector<uint16_t> pis;
        split_operand_sw128(P.data(), d, kPiScale, pis);
        e = cudaMalloc((void **)&ctx->pi_split, pis.size() * 2);
        if (e == cudaSuccess) e = cudaMemcpy(ctx->pi_split, pis.data(), pis.size() * 2, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return e;
    }
    e = upload_vec(&ctx->k4_cells, grid.rec);
    if (e == cudaSuccess) e = upload_vec(&ctx->k4_pool, grid.pool);
    if (e == cudaSuccess) e = upload_vec(&ctx->k4_axis, grid.axis);
    if (e == cudaSuccess) e = upload_vec(&ctx->k4_ncb, ncb);
    if (e != cudaSuccess) return e;
    if (d == 64) return prep_k4<64, 5, 1>(ctx);
    return prep_k4<128, 2, 1>(ctx);
}

cudaError_t launch_encode_k4_grid(const fq_ctx *ctx, const __half *x, int64_t M, RowMap map, float *nu,
                                  uint32_t *codes, cudaStream_t s) {
    if (ctx->d == 64)
        return launch_k4<64, 5, 1>(ctx, x, M, map, nu, codes, s);
    return launch_k4<128, 2, 1>(ctx, x, M, map, nu, codes, s);
}

}  // namespace fq
