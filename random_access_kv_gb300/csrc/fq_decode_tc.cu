// Tensor-core block decoder for k <= 8 [FibQuant §2.3, decoder], full and random-access
// (gather, [FibQuant §1]: any vector decodes on its own from its fixed address).
//
// Each 128-row output tile goes through three steps. At d = 64 (decode_tc) a CTA runs NG row
// groups of 128 threads, one thread per output vector (= TMEM lane), each group taking its tiles
// through the steps in turn; at d = 128 (decode_ws, below) the steps of consecutive tiles run at
// once in separate warps:
//   1. Each thread reads its source row (idx[j] for a gather), its nu and its record, unpacks the
//      d/k indices and writes the concatenated codewords y_hat, split into fp16 halves of
//      2^10 y_hat (hi, lo), as row t of two shared-memory A operands (128-byte swizzle).
//   2. One thread issues Y_hat Pi on the tensor pipe as three fp16 MMAs into a TMEM fp32
//      accumulator: hi*Pi_hi + hi*Pi_lo + lo*Pi_hi, with Pi^T carried as fp16 halves of 2^12 Pi^T
//      (the dropped lo*lo term is below 2^-22 of the result).
//   3. Each thread reads its row back and scales it by nu 2^-22. fp16 output (rounded to nearest
//      even) is staged row by row in the tile's A buffer, in the same 128-byte swizzle, and
//      written by one TMA tensor store per 64-column box; fp32 output is stored row by row.
// With d = 64 and a codebook of at most 512 words (k <= 2), the table is held once per lane
// (word w of lane l at w * 32 + l), so that the random codeword reads of a warp never share a bank.
// Gather indices outside [0, M) give zero rows and set FQ_FLAG_RANGE.
#include <math.h>
#include <string.h>

#include <vector>

#include "fq_bits.cuh"
#include "fq_internal.h"
#include "fq_sm100.cuh"

namespace fq {

namespace {

using namespace sm100;

constexpr int kTileRows = 128;
constexpr float kPiScale = 4096.f;    // 2^12 on Pi^T
constexpr float kYScale = 1024.f;     // 2^10 on the codewords
constexpr float kOutScale = 1.0f / (4096.f * 1024.f);

// Where the codebook halves are read from.
constexpr int kCbGlobal = 0, kCbShared = 1, kCbLanes = 2;

template <int D, int K, int NG, int CBM>
struct DLayout {
    static constexpr int kPiPart = D * D * 2;
    static constexpr int kATile = kTileRows * D * 2;                 // one fp16 A operand
    static constexpr int oPi = 0;
    static constexpr int oA = oPi + 2 * kPiPart;
    static constexpr int oCb = oA + NG * 2 * kATile;
    static constexpr int kCbMax = CBM == kCbShared ? 16384 : CBM == kCbLanes ? 65536 : 0;
    static constexpr int oBar = oCb + kCbMax;
    static constexpr int kBars = 1 + NG;
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;
    static constexpr uint32_t kTmemCols = (NG * D <= 64) ? 64 : (NG * D <= 128) ? 128 : (NG * D <= 256) ? 256 : 512;
};

struct DecParams {
    const float *nu;
    const uint32_t *codes;
    int64_t M;
    const int64_t *idx;       // null: row j
    int64_t n;
    int B;
    int N;
    const uint8_t *pit_split; // [2][D*D] fp16 halves of 2^12 Pi^T, swizzled
    const uint16_t *cb;       // [N][2K] fp16: K hi halves then K lo halves of 2^10 c_n
    const uint32_t *cb_lanes; // the words of cb, each repeated for the 32 lanes (or null)
    void *out;
    uint32_t *flags;
};

// Codeword n's hi and lo halves, K of each.
template <int K>
struct CwHalves {
    uint32_t hi[K > 1 ? K / 2 : 1], lo[K > 1 ? K / 2 : 1];
};

template <int K, int CBM>
__device__ __forceinline__ CwHalves<K> fetch_cw(const uint16_t *cb, uint32_t n, int lane) {
    CwHalves<K> r;
    constexpr bool CB_SMEM = CBM == kCbShared;
    if constexpr (CBM == kCbLanes) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(cb) + lane;
        if constexpr (K == 2) {
            r.hi[0] = w[(2 * n) * 32];
            r.lo[0] = w[(2 * n + 1) * 32];
        } else {
            const uint32_t v = w[n * 32];
            r.hi[0] = v & 0xFFFFu; r.lo[0] = v >> 16;
        }
        return r;
    }
    const uint16_t *p = cb + (size_t)n * 2 * K;
    if constexpr (K == 8) {
        const uint4 h = CB_SMEM ? *reinterpret_cast<const uint4 *>(p) : __ldg(reinterpret_cast<const uint4 *>(p));
        const uint4 l = CB_SMEM ? *reinterpret_cast<const uint4 *>(p + 8) : __ldg(reinterpret_cast<const uint4 *>(p + 8));
        r.hi[0] = h.x; r.hi[1] = h.y; r.hi[2] = h.z; r.hi[3] = h.w;
        r.lo[0] = l.x; r.lo[1] = l.y; r.lo[2] = l.z; r.lo[3] = l.w;
    } else if constexpr (K == 4) {
        const uint4 v = CB_SMEM ? *reinterpret_cast<const uint4 *>(p) : __ldg(reinterpret_cast<const uint4 *>(p));
        r.hi[0] = v.x; r.hi[1] = v.y; r.lo[0] = v.z; r.lo[1] = v.w;
    } else if constexpr (K == 2) {
        const uint2 v = CB_SMEM ? *reinterpret_cast<const uint2 *>(p) : __ldg(reinterpret_cast<const uint2 *>(p));
        r.hi[0] = v.x; r.lo[0] = v.y;
    } else {
        const uint32_t v = CB_SMEM ? *reinterpret_cast<const uint32_t *>(p) : __ldg(reinterpret_cast<const uint32_t *>(p));
        r.hi[0] = v & 0xFFFFu; r.lo[0] = v >> 16;
    }
    return r;
}

template <int D, typename OutT>
__device__ __forceinline__ void store16(OutT *out, int64_t j, int c, const float (&v)[16], float s) {
    if constexpr (sizeof(OutT) == 2) {
        uint4 *dst = reinterpret_cast<uint4 *>(out + j * D + 16 * c);
        uint4 w[2];
        __half2 *h = reinterpret_cast<__half2 *>(w);
#pragma unroll
        for (int q = 0; q < 8; ++q) h[q] = __floats2half2_rn(v[2 * q] * s, v[2 * q + 1] * s);
        dst[0] = w[0];
        dst[1] = w[1];
    } else {
        float4 *dst = reinterpret_cast<float4 *>(out + j * D + 16 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q] * s, v[4 * q + 1] * s, v[4 * q + 2] * s, v[4 * q + 3] * s);
    }
}

// The source row, its scale and its record, loaded ahead of use. With a compile-time B whose
// records are whole words (BS != 0) the record is held in registers; otherwise it is read
// field by field through the bit reader when the A operand is written.
template <int W>
struct RowData {
    int64_t j;
    int64_t row;
    bool live, valid;
    float s;
    uint32_t w[W > 0 ? W : 1];
};

template <int D, int K, int BS, bool NU = true>
__device__ __forceinline__ RowData<(BS ? (D / K) * BS / 32 : 0)> load_row(const DecParams &p, int64_t tile, int t) {
    constexpr int W = BS ? (D / K) * BS / 32 : 0;
    RowData<W> r;
    r.j = tile * kTileRows + t;
    r.live = r.j < p.n;
    r.row = r.live ? (p.idx ? __ldg(p.idx + r.j) : r.j) : 0;
    r.valid = r.live && r.row >= 0 && r.row < p.M;
    r.s = (NU && r.valid) ? __ldg(p.nu + r.row) * kOutScale : 0.f;
    if constexpr (W > 0) {
        const uint32_t *src = p.codes + (r.valid ? r.row : 0) * W;
        if constexpr (W % 4 == 0) {
            if ((reinterpret_cast<uintptr_t>(p.codes) & 15u) == 0) {
#pragma unroll
                for (int q = 0; q < W; q += 4) {
                    const uint4 v = r.valid ? __ldg(reinterpret_cast<const uint4 *>(src + q)) : make_uint4(0, 0, 0, 0);
                    r.w[q] = v.x; r.w[q + 1] = v.y; r.w[q + 2] = v.z; r.w[q + 3] = v.w;
                }
                return r;
            }
        }
#pragma unroll
        for (int q = 0; q < W; ++q) r.w[q] = r.valid ? __ldg(src + q) : 0u;
    }
    return r;
}

// Field b (BS bits) of a register-held record.
template <int BS, int W>
__device__ __forceinline__ uint32_t field(const uint32_t (&w)[W], int b) {
    const int bit = b * BS, q = bit / 32, o = bit % 32;
    uint32_t v;
    if (o + BS <= 32 || q + 1 >= W) v = w[q] >> o;
    else v = __funnelshift_r(w[q], w[q + 1], o);
    return v & ((1u << BS) - 1u);
}

// Row t of the two A operands (fp16 halves of 2^10 y_hat, 128-byte swizzle) from the row's
// record, one 16-byte chunk (8 columns) at a time: the d/k codewords of the record, concatenated.
// A row that is not valid is written as zeros.
template <int D, int K, int CBM, int BS, int W>
__device__ __forceinline__ void build_a_row(const DecParams &p, const RowData<W> &cur, const uint16_t *cb,
                                            uint8_t *a_hi, uint8_t *a_lo, int t) {
    const int R = (D / K) * p.B;
    BitReader rd(p.codes, (BS == 0 && cur.valid) ? cur.row * (int64_t)R : 0, BS == 0 && cur.valid);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
        if (cur.valid) {
            constexpr int BPC = K >= 2 ? 8 / K : 8;      // blocks per chunk
#pragma unroll
            for (int b = 0; b < BPC; ++b) {
                uint32_t i;
                if constexpr (BS != 0) i = field<BS, W>(cur.w, c * BPC + b);
                else i = rd.get(p.B);
                const CwHalves<K> v = fetch_cw<K, CBM>(cb, i, t & 31);
                if constexpr (K >= 2) {
#pragma unroll
                    for (int q = 0; q < K / 2; ++q) {
                        hw[b * (K / 2) + q] = v.hi[q];
                        lw[b * (K / 2) + q] = v.lo[q];
                    }
                } else {
                    hw[b / 2] |= v.hi[0] << (16 * (b & 1));
                    lw[b / 2] |= v.lo[0] << (16 * (b & 1));
                }
            }
        }
        const int kb = c / 8, cc = c % 8;
        const uint32_t off = (uint32_t)(kb * 16384 + t * 128 + ((cc ^ (t & 7)) << 4));
        *reinterpret_cast<uint4 *>(a_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(a_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

// Y_hat Pi^T-split into a 128 x D fp32 accumulator: hi*Pi_hi + hi*Pi_lo + lo*Pi_hi, D/16
// K-steps each (A: 128 rows x D fp16 in 64-column swizzled blocks of 16 KB; B likewise, D rows).
template <int D>
__device__ __forceinline__ void issue_rotation(uint32_t acc, uint32_t ah, uint32_t al, uint32_t pb_hi, uint32_t pb_lo) {
    const uint32_t idesc = idesc_f16_f32(128, D);
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const uint32_t aa = pass == 2 ? al : ah;
        const uint32_t bb = pass == 1 ? pb_lo : pb_hi;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t aoff = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32);
            const uint32_t boff = (uint32_t)((kk >> 2) * (D * 128) + (kk & 3) * 32);
            mma_f16(acc, sdesc_sw128(aa + aoff), sdesc_sw128(bb + boff), idesc, (pass | kk) ? 1u : 0u);
        }
    }
}

template <int D, int K, int NG, int CBM, int BS, typename OutT>
__global__ void __launch_bounds__(NG * 128, 1) decode_tc(const __grid_constant__ CUtensorMap omap, const DecParams p) {
    constexpr bool CB_SMEM = CBM != kCbGlobal;
    constexpr bool TMA_OUT = sizeof(OutT) == 2;
    using L = DLayout<D, K, NG, CBM>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oTmem);
    const uint16_t *cb = CB_SMEM ? reinterpret_cast<const uint16_t *>(sm + L::oCb) : p.cb;

    const int tid = threadIdx.x;
    const int g = tid / 128;
    const int t = tid % 128;
    const int wq = t / 32;
    uint64_t *bar_tab = bars;
    uint64_t *bar_mma = bars + 1 + g;
    uint8_t *a_hi = sm + L::oA + g * 2 * L::kATile;
    uint8_t *a_lo = a_hi + L::kATile;
    const int64_t ntiles = (p.n + kTileRows - 1) / kTileRows;
    const int64_t gstride = (int64_t)gridDim.x * NG;
    const int64_t first = (int64_t)blockIdx.x * NG + g;
    constexpr int W = BS ? (D / K) * BS / 32 : 0;

    if (tid == 0) {
        for (int i = 0; i < L::kBars; ++i) mbar_init(bars + i, 1);
        fence_barrier_init();
    }
    if (tid < 32) tmem_alloc(tmem_slot, L::kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (tid == 0) {
        // A bulk copy moves a multiple of 16 bytes; the table is allocated padded to one.
        const uint32_t cb_bytes = CBM == kCbLanes ? (uint32_t)(p.N * K * 4 * 32)
                                  : CB_SMEM ? ((uint32_t)(p.N * K * 4) + 15u) & ~15u : 0u;
        mbar_arrive_expect_tx(bar_tab, 2u * L::kPiPart + cb_bytes);
        bulk_g2s(sm + L::oPi, p.pit_split, 2u * L::kPiPart, bar_tab);
        if (CB_SMEM)
            bulk_g2s(sm + L::oCb, CBM == kCbLanes ? static_cast<const void *>(p.cb_lanes) : static_cast<const void *>(p.cb),
                     cb_bytes, bar_tab);
        if (TMA_OUT) prefetch_tensormap(&omap);
    }
    // Indices, norms and codes may be written by the previous kernel in the stream.
    griddep_launch_dependents();
    griddep_wait();
    // The first tile's row data is requested before the tables arrive.
    RowData<W> cur = load_row<D, K, BS>(p, first, t);
    bool ok = named_sync_and(1 + g, 128, mbar_wait(bar_tab, 0));

    const uint32_t tmem_acc = tmem_base + (uint32_t)(g * D);
    const uint32_t pb_hi = smem_addr(sm + L::oPi), pb_lo = pb_hi + L::kPiPart;
    OutT *out = reinterpret_cast<OutT *>(p.out);

    int64_t it = 0;
    for (int64_t tile = first; tile < ntiles && ok; tile += gstride, ++it) {
        // Requests for the next tile go out now and land while this one is processed.
        const RowData<W> nxt = load_row<D, K, BS>(p, tile + gstride, t);
        if (cur.live && !cur.valid) atomicOr(p.flags, (uint32_t)FQ_FLAG_RANGE);
        build_a_row<D, K, CBM, BS, W>(p, cur, cb, a_hi, a_lo, t);
        fence_proxy_async_smem();
        named_sync(1 + g, 128);
        if (t == 0) {
            tc_fence_after();
            issue_rotation<D>(tmem_acc, smem_addr(a_hi), smem_addr(a_lo), pb_hi, pb_lo);
            mma_commit(bar_mma);
        }
        ok = named_sync_and(1 + g, 128, mbar_wait(bar_mma, (uint32_t)(it & 1)));
        if (!ok) break;
        tc_fence_after();
        if constexpr (TMA_OUT) {
            // Row t of the output tile into the A buffer the MMA has finished with, then one
            // tensor store per 64-column box (rows past n are clipped by the store).
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
                float v[16];
                tmem_ld16(tmem_acc + ((uint32_t)(32 * wq) << 16) + (uint32_t)(16 * c), v);
                tmem_wait_ld();
                uint32_t w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const __half2 h = __floats2half2_rn(v[2 * q] * cur.s, v[2 * q + 1] * cur.s);
                    w[q] = *reinterpret_cast<const uint32_t *>(&h);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int ch = 2 * c + hh, kb = ch / 8, cc = ch % 8;
                    const uint32_t off = (uint32_t)(kb * 16384 + t * 128 + ((cc ^ (t & 7)) << 4));
                    *reinterpret_cast<uint4 *>(a_hi + off) = make_uint4(w[4 * hh], w[4 * hh + 1], w[4 * hh + 2], w[4 * hh + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(1 + g, 128);
            if (t == 0) {
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) tma_store_2d(&omap, a_hi + kb * 16384, kb * 64, (int)(tile * kTileRows));
                bulk_commit();
                bulk_wait_read0();          // the next tile's A operand overwrites this buffer
            }
        } else {
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
                float v[16];
                tmem_ld16(tmem_acc + ((uint32_t)(32 * wq) << 16) + (uint32_t)(16 * c), v);
                tmem_wait_ld();
                if (cur.live) store16<D, OutT>(out, cur.j, c, v, cur.s);
            }
            tc_fence_before();
        }
        named_sync(1 + g, 128);
        cur = nxt;
    }
    if (!ok && t == 0) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
    if (TMA_OUT && t == 0) bulk_wait_all();   // stores complete before the CTA's memory goes away
    __syncthreads();
    if (!ok) mbar_wait(bar_mma, 0, 1000000ull);
    tc_fence_after();
    if (tid < 32) tmem_dealloc(tmem_base, L::kTmemCols);
}

// ---- d = 128: warp-specialised pipeline -----------------------------------------------------
//
// At d = 128 one A operand pair (hi, lo) is 64 KB and the rotation another 64 KB, so only two
// row groups fit and each ran its phases (A rows, MMAs, read-back and store) one after another.
// Here the phases of consecutive tiles overlap instead, through two A buffers, two TMEM
// accumulators and one output stage (224 KB of shared memory):
//   warps 0-7   two builder groups of 128 threads; group b writes the A rows of the CTA's tiles
//               i = b, b + 2, ... into A buffer b (one thread per row; at k = 8 one 256-bit load
//               per codeword), then arrives on a_full[b];
//   warp 16     one thread issues each tile's three MMAs into accumulator i % 2 once its A rows are
//               written and the accumulator is free, and commits to mma_done[i % 2] (which also
//               frees A buffer i % 2 for the builders);
//   warps 8-15  the read-back: warp 8 + 4h + q reads TMEM lanes 32q .. 32q + 31 (its rows),
//               columns 64h .. 64h + 63, releases the accumulator (acc_empty), scales by nu, and
//               stages fp16 rows for one TMA tensor store per 64-column box (fp32 rows are stored
//               directly). These threads read the row's index and nu themselves, ahead of use.
// The source rows, records and norms of later tiles are requested early enough that no step
// waits on a load issued in the same iteration.
// Every wait is bounded; a wait that gives up sets FQ_FLAG_TIMEOUT and its role stops.
struct WsLayout {
    static constexpr int D = 128;
    static constexpr int kPiPart = D * D * 2;                    // 32 KB
    static constexpr int kATile = kTileRows * D * 2;             // 32 KB: one fp16 operand
    static constexpr int oPi = 0;
    static constexpr int oA = oPi + 2 * kPiPart;                 // two (hi, lo) buffers
    static constexpr int oOut = oA + 2 * 2 * kATile;             // the fp16 output stage
    static constexpr int oBar = oOut + kATile;
    static constexpr int kBars = 7;                              // tables, a_full[2], mma_done[2], acc_empty[2]
    static constexpr int oTmem = oBar + kBars * 8;
    static constexpr int kBytes = oTmem + 16 + 1024;
    static constexpr uint32_t kTmemCols = 2 * D;
};
constexpr int kWsEpiWarp = 8, kWsMmaWarp = 16, kWsThreads = 17 * 32, kWsEpiThreads = 256;

// The source row of output row j: its gather index, or j itself. Rows past n read the last index
// (a valid address); whether a row is live and valid is decided where the value is used, so that
// nothing waits on the load in the iteration that issues it.
__device__ __forceinline__ int64_t src_row(const DecParams &p, int64_t j) {
    return p.idx ? __ldg(p.idx + (j < p.n ? j : p.n - 1)) : j;
}

__device__ __forceinline__ bool row_valid(const DecParams &p, int64_t j, int64_t row) {
    return j < p.n && row >= 0 && row < p.M;
}

// A record held in registers (W words; none when fields are read at run time).
template <int W>
struct Rec {
    uint32_t w[W > 0 ? W : 1];
};

template <int W>
__device__ __forceinline__ Rec<W> load_rec(const DecParams &p, int64_t row, bool valid) {
    Rec<W> r;
#pragma unroll
    for (int q = 0; q < (W > 0 ? W : 1); ++q) r.w[q] = 0u;
    if constexpr (W > 0) {
        const uint32_t *src = p.codes + (valid ? row : 0) * W;
#pragma unroll
        for (int q = 0; q < W; ++q) r.w[q] = valid ? __ldg(src + q) : 0u;
    }
    return r;
}

// 32 bytes (one sector) from read-only global memory in one 256-bit load, not kept in L1.
// The address must be 32-byte aligned.
__device__ __forceinline__ void ld_nc_v8(const void *src, uint32_t (&r)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(src));
}

// k = 8 A rows: each codeword's 32 bytes (fp16 hi half, then lo half) are one sector, read by one
// 256-bit load and written as one 16-byte chunk of each A operand. Eight codewords are in flight
// at a time. A row that is not valid is written as zeros.
template <int BS, int W>
__device__ __forceinline__ void build_k8_row(const DecParams &p, int64_t row, bool valid, const Rec<W> &rec,
                                             uint8_t *a_hi, uint8_t *a_lo, int t) {
    constexpr int D = 128, K = 8;
    BitReader rd(p.codes, (BS == 0 && valid) ? row * (int64_t)((D / K) * p.B) : 0, BS == 0 && valid);
#pragma unroll
    for (int c0 = 0; c0 < D / 8; c0 += 8) {
        uint32_t v[8][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
#pragma unroll
            for (int m = 0; m < 8; ++m) v[c][m] = 0u;
            if (valid) {
                uint32_t i;
                if constexpr (BS != 0) i = field<BS, W>(rec.w, c0 + c);
                else i = rd.get(p.B);
                ld_nc_v8(p.cb + (size_t)i * 2 * K, v[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int ch = c0 + c, kb = ch / 8, cc = ch % 8;
            const uint32_t off = (uint32_t)(kb * 16384 + t * 128 + ((cc ^ (t & 7)) << 4));
            *reinterpret_cast<uint4 *>(a_hi + off) = make_uint4(v[c][0], v[c][1], v[c][2], v[c][3]);
            *reinterpret_cast<uint4 *>(a_lo + off) = make_uint4(v[c][4], v[c][5], v[c][6], v[c][7]);
        }
    }
}

template <int K, int BS, typename OutT>
__global__ void __launch_bounds__(kWsThreads, 1) decode_ws(const __grid_constant__ CUtensorMap omap, const DecParams p) {
    constexpr int D = 128;
    constexpr bool TMA_OUT = sizeof(OutT) == 2;
    constexpr int W = BS ? (D / K) * BS / 32 : 0;
    using L = WsLayout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
    uint64_t *bar_tab = bars, *a_full = bars + 1, *mma_done = bars + 3, *acc_empty = bars + 5;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oTmem);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int64_t ntiles = (p.n + kTileRows - 1) / kTileRows;
    const int64_t first = blockIdx.x, gstride = gridDim.x;

    if (tid == 0) {
        mbar_init(bar_tab, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(a_full + b, 1);
            mbar_init(mma_done + b, 1);
            mbar_init(acc_empty + b, 8);                 // one arrival per read-back warp
        }
        fence_barrier_init();
    }
    if (warp == kWsMmaWarp) tmem_alloc(tmem_slot, L::kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_tab, 2u * L::kPiPart);
        bulk_g2s(sm + L::oPi, p.pit_split, 2u * L::kPiPart, bar_tab);
        if (TMA_OUT) prefetch_tensormap(&omap);
    }
    // Indices, norms and codes may be written by the previous kernel in the stream.
    griddep_launch_dependents();
    griddep_wait();

    bool ok = true;
    if (warp < kWsEpiWarp) {
        // Builder thread t of group b writes row t of the group's tiles. Source rows are read two
        // of the group's tiles ahead and records one ahead.
        const int b = warp / 4, t = tid % 128;
        uint8_t *a_hi = sm + L::oA + b * 2 * L::kATile;
        uint8_t *a_lo = a_hi + L::kATile;
        auto jrow = [&](int64_t i) { return (first + i * gstride) * kTileRows + t; };
        int64_t row_c = src_row(p, jrow(b)), row_n = src_row(p, jrow(b + 2));
        Rec<W> rec_c = load_rec<W>(p, row_c, row_valid(p, jrow(b), row_c));
        for (int64_t i = b; first + i * gstride < ntiles; i += 2) {
            const Rec<W> rec_n = load_rec<W>(p, row_n, row_valid(p, jrow(i + 2), row_n));
            const int64_t row_nn = src_row(p, jrow(i + 4));
            const bool valid = row_valid(p, jrow(i), row_c);
            if (jrow(i) < p.n && !valid) atomicOr(p.flags, (uint32_t)FQ_FLAG_RANGE);
            if (i >= 2) {
                // The MMAs of tile i - 2 have read this buffer.
                ok = named_sync_and(1 + b, 128, mbar_wait(mma_done + b, (uint32_t)(((i >> 1) - 1) & 1)));
                if (!ok) break;
            }
            if constexpr (K == 8) {
                build_k8_row<BS, W>(p, row_c, valid, rec_c, a_hi, a_lo, t);
            } else {
                RowData<W> rd;
                rd.j = jrow(i);
                rd.row = row_c;
                rd.live = rd.j < p.n;
                rd.valid = valid;
                rd.s = 0.f;
#pragma unroll
                for (int q = 0; q < (W > 0 ? W : 1); ++q) rd.w[q] = rec_c.w[q];
                build_a_row<D, K, kCbGlobal, BS, W>(p, rd, p.cb, a_hi, a_lo, t);
            }
            fence_proxy_async_smem();
            named_sync(1 + b, 128);
            if (t == 0) mbar_arrive(a_full + b);
            rec_c = rec_n;
            row_c = row_n;
            row_n = row_nn;
        }
    } else if (warp < kWsMmaWarp) {
        // Read-back warp 8 + 4h + q: rows 32q .. 32q + 31 (TMEM lanes), columns 64h .. 64h + 63.
        const int et = tid - kWsEpiWarp * 32, wq = warp % 4, h = (warp - kWsEpiWarp) / 4;
        const int e = 32 * wq + lane;                    // the row
        uint8_t *stage = sm + L::oOut;
        OutT *out = reinterpret_cast<OutT *>(p.out);
        // Source rows two tiles ahead, nu one tile ahead; the scale is formed where it is used.
        auto jrow = [&](int64_t i) { return (first + i * gstride) * kTileRows + e; };
        int64_t row_n = src_row(p, jrow(1));
        const int64_t row0 = src_row(p, jrow(0));
        float nu_c = row_valid(p, jrow(0), row0) ? __ldg(p.nu + row0) : 0.f;
        for (int64_t i = 0; first + i * gstride < ntiles; ++i) {
            const int b = (int)(i & 1);
            const int64_t tile = first + i * gstride;
            const float nu_n = row_valid(p, jrow(i + 1), row_n) ? __ldg(p.nu + row_n) : 0.f;
            const int64_t row_nn = src_row(p, jrow(i + 2));
            const float sc = nu_c * kOutScale;
            const int64_t jc = jrow(i);
            const bool w = mbar_wait(mma_done + b, (uint32_t)((i >> 1) & 1));
            if (TMA_OUT && et == 0) bulk_wait_read0();   // the previous tile's store has read the stage
            ok = named_sync_and(3, kWsEpiThreads, w);
            if (!ok) break;
            tc_fence_after();
            const uint32_t acc = tmem_base + (uint32_t)(b * D + 64 * h) + ((uint32_t)(32 * wq) << 16);
            uint32_t r[4][16];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16_nowait(acc + (uint32_t)(16 * q), r[q]);
            tmem_wait_ld();
            // This warp's reads of the accumulator are done.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + b);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float v[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) v[m] = __uint_as_float(r[q][m]);
                if constexpr (TMA_OUT) {
                    uint32_t hw[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const __half2 hv = __floats2half2_rn(v[2 * m] * sc, v[2 * m + 1] * sc);
                        hw[m] = *reinterpret_cast<const uint32_t *>(&hv);
                    }
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int cc = 2 * q + hh;               // 16-byte chunk within box h
                        const uint32_t off = (uint32_t)(h * 16384 + e * 128 + ((cc ^ (e & 7)) << 4));
                        *reinterpret_cast<uint4 *>(stage + off) =
                            make_uint4(hw[4 * hh], hw[4 * hh + 1], hw[4 * hh + 2], hw[4 * hh + 3]);
                    }
                } else {
                    if (jc < p.n) store16<D, OutT>(out, jc, 4 * h + q, v, sc);
                }
            }
            if constexpr (TMA_OUT) {
                fence_proxy_async_smem();
                named_sync(3, kWsEpiThreads);
                if (et == 0) {
                    // Rows past n are clipped by the store.
                    tma_store_2d(&omap, stage, 0, (int)(tile * kTileRows));
                    tma_store_2d(&omap, stage + 16384, 64, (int)(tile * kTileRows));
                    bulk_commit();
                }
            }
            nu_c = nu_n;
            row_n = row_nn;
        }
        if (TMA_OUT && et == 0) bulk_wait_all();         // stores complete before the CTA's memory goes away
    } else if (lane == 0) {
        const uint32_t pb_hi = smem_addr(sm + L::oPi), pb_lo = pb_hi + L::kPiPart;
        uint32_t issued0 = 0u, issued1 = 0u;         // tiles issued into accumulator 0 and 1
        ok = mbar_wait(bar_tab, 0);
        for (int64_t i = 0; ok && first + i * gstride < ntiles; ++i) {
            const int b = (int)(i & 1);
            ok = mbar_wait(a_full + b, (uint32_t)((i >> 1) & 1));
            // The read-back of tile i - 2 has left accumulator b.
            if (ok && i >= 2) ok = mbar_wait(acc_empty + b, (uint32_t)(((i >> 1) - 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const uint32_t ab = smem_addr(sm + L::oA + b * 2 * L::kATile);
            issue_rotation<D>(tmem_base + (uint32_t)(b * D), ab, ab + L::kATile, pb_hi, pb_lo);
            mma_commit(mma_done + b);
            if (b) ++issued1;
            else ++issued0;
        }
        // Every issued MMA has finished before the tensor memory is released.
        if (issued0) mbar_wait(mma_done, (issued0 - 1u) & 1u, 1000000ull);
        if (issued1) mbar_wait(mma_done + 1, (issued1 - 1u) & 1u, 1000000ull);
    }
    if (!ok) atomicOr(p.flags, (uint32_t)FQ_FLAG_TIMEOUT);
    __syncthreads();
    tc_fence_after();
    if (warp == kWsMmaWarp) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int D, int K>
constexpr int groups() { return D == 64 ? 4 : 2; }

template <int D, int K>
constexpr int cb_mode() { return K <= 4 ? kCbShared : kCbGlobal; }

// The lane-replicated table fits its 64 KB slot beside four d = 64 row groups.
template <int D, int K>
constexpr bool lanes_possible() { return D == 64 && K <= 2; }

template <int D, int K, int CBM, int BS, typename OutT>
cudaError_t launch_dkm(const fq_ctx *ctx, const DecParams &p, cudaStream_t s) {
    constexpr int NG = D == 128 ? 1 : groups<D, K>();      // d = 128: one pipeline per CTA
    CUtensorMap omap;
    memset(&omap, 0, sizeof(omap));
    if (sizeof(OutT) == 2 && !encode_rows_tensor_map(&omap, p.out, p.n, D)) return cudaErrorInvalidValue;
    const int64_t ntiles = (p.n + kTileRows - 1) / kTileRows;
    int64_t grid = (ntiles + NG - 1) / NG;
    if (grid > ctx->num_sms) grid = ctx->num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (D == 128) {
        cfg.blockDim = dim3(kWsThreads);
        cfg.dynamicSmemBytes = WsLayout::kBytes;
        return cudaLaunchKernelEx(&cfg, decode_ws<K, BS, OutT>, omap, p);
    } else {
        cfg.blockDim = dim3(NG * 128);
        cfg.dynamicSmemBytes = DLayout<D, K, NG, CBM>::kBytes;
        return cudaLaunchKernelEx(&cfg, decode_tc<D, K, NG, CBM, BS, OutT>, omap, p);
    }
}

template <int D, int K, int BS, typename OutT>
cudaError_t launch_dk(const fq_ctx *ctx, const DecParams &p, cudaStream_t s) {
    if constexpr (lanes_possible<D, K>())
        if (p.cb_lanes) return launch_dkm<D, K, kCbLanes, BS, OutT>(ctx, p, s);
    return launch_dkm<D, K, cb_mode<D, K>(), BS, OutT>(ctx, p, s);
}

template <int D, int K, int CBM, int BS>
cudaError_t prep_dkm() {
    if constexpr (D == 128) {
        static_assert(WsLayout::kBytes <= 227 * 1024, "shared memory budget");
        cudaError_t e = cudaFuncSetAttribute(decode_ws<K, BS, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             WsLayout::kBytes);
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(decode_ws<K, BS, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    WsLayout::kBytes);
    }
    constexpr int NG = groups<D, K>();
    using L = DLayout<D, K, NG, CBM>;
    static_assert(L::kBytes <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(decode_tc<D, K, NG, CBM, BS, __half>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_tc<D, K, NG, CBM, BS, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kBytes);
}

template <int D, int K, int BS>
cudaError_t prep_dk(bool lanes) {
    if constexpr (lanes_possible<D, K>())
        if (lanes) return prep_dkm<D, K, kCbLanes, BS>();
    return prep_dkm<D, K, cb_mode<D, K>(), BS>();
}

// Record widths with a compile-time field size: (d, k, B) of the synthetic workloads, whose
// records are whole 32-bit words. Everything else reads its fields at run time.
constexpr int kStatic[][3] = {{64, 2, 4}, {64, 2, 8}, {64, 4, 10}, {128, 8, 12}};

int static_bits(int d, int k, int B) {
    for (const auto &c : kStatic)
        if (c[0] == d && c[1] == k && c[2] == B) return B;
    return 0;
}

}  // namespace

bool decode_tc_supported(const fq_ctx *ctx) {
    if (!(ctx->d == 64 || ctx->d == 128)) return false;
    if (!(ctx->k == 1 || ctx->k == 2 || ctx->k == 4 || ctx->k == 8)) return false;
    // Codebooks that live in shared memory must fit its 16 KB slot.
    if (ctx->k <= 4 && (size_t)ctx->N * ctx->k * 4 > 16384) return false;
    return true;
}

cudaError_t prepare_decode_tc(fq_ctx *ctx) {
    const int d = ctx->d, k = ctx->k, N = ctx->N;
    std::vector<float> P((size_t)d * d), PT((size_t)d * d), C((size_t)N * k);
    cudaError_t e = cudaMemcpy(P.data(), ctx->Pi, P.size() * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(C.data(), ctx->C, C.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    for (int a = 0; a < d; ++a)
        for (int b = 0; b < d; ++b) PT[(size_t)a * d + b] = P[(size_t)b * d + a];
    std::vector<uint16_t> pts;
    split_operand_sw128(PT.data(), d, kPiScale, pts);
    std::vector<uint16_t> cb((size_t)N * 2 * k);
    for (int n = 0; n < N; ++n)
        for (int q = 0; q < k; ++q) {
            const float v = C[(size_t)n * k + q] * kYScale;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            memcpy(&cb[(size_t)n * 2 * k + q], &hi, 2);
            memcpy(&cb[(size_t)n * 2 * k + k + q], &lo, 2);
        }
    e = cudaMalloc((void **)&ctx->pit_split, pts.size() * 2);
    if (e == cudaSuccess) e = cudaMemcpy(ctx->pit_split, pts.data(), pts.size() * 2, cudaMemcpyHostToDevice);
    // Padded to a multiple of 16 bytes: the kernel bulk-copies the whole table (N k = 2 gives 8 bytes).
    const size_t cb_alloc = (cb.size() * 2 + 15) & ~(size_t)15;
    if (e == cudaSuccess) e = cudaMalloc((void **)&ctx->cb_split, cb_alloc);
    if (e == cudaSuccess) e = cudaMemset(ctx->cb_split, 0, cb_alloc);
    if (e == cudaSuccess) e = cudaMemcpy(ctx->cb_split, cb.data(), cb.size() * 2, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return e;
    // Lane-replicated copy of the table's 32-bit words (d = 64, k <= 2, N k <= 512 words).
    const bool lanes = d == 64 && k <= 2 && (size_t)N * k <= 512;
    if (lanes) {
        std::vector<uint32_t> words((size_t)N * k), rep((size_t)N * k * 32);
        memcpy(words.data(), cb.data(), words.size() * 4);
        for (size_t w = 0; w < words.size(); ++w)
            for (int l = 0; l < 32; ++l) rep[w * 32 + l] = words[w];
        e = cudaMalloc((void **)&ctx->cb_lanes, rep.size() * 4);
        if (e == cudaSuccess) e = cudaMemcpy(ctx->cb_lanes, rep.data(), rep.size() * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return e;
    }
    {
        cudaError_t es = cudaSuccess;
        if (static_bits(d, k, ctx->B) == 4) es = prep_dk<64, 2, 4>(lanes);
        if (static_bits(d, k, ctx->B) == 8) es = prep_dk<64, 2, 8>(lanes);
        if (static_bits(d, k, ctx->B) == 10) es = prep_dk<64, 4, 10>(lanes);
        if (static_bits(d, k, ctx->B) == 12) es = prep_dk<128, 8, 12>(lanes);
        if (es != cudaSuccess) return es;
    }
#define PREP(D, K) prep_dk<D, K, 0>(lanes)
    if (d == 64) {
        if (k == 1) return PREP(64, 1);
        if (k == 2) return PREP(64, 2);
        if (k == 4) return PREP(64, 4);
        return PREP(64, 8);
    }
    if (k == 1) return PREP(128, 1);
    if (k == 2) return PREP(128, 2);
    if (k == 4) return PREP(128, 4);
    return PREP(128, 8);
#undef PREP
}

cudaError_t launch_decode_tc(const fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                             const int64_t *idx, int64_t n, void *out, bool out_f32, cudaStream_t s) {
    DecParams p;
    p.nu = nu;
    p.codes = codes;
    p.M = M;
    p.idx = idx;
    p.n = n;
    p.B = ctx->B;
    p.N = ctx->N;
    p.pit_split = ctx->pit_split;
    p.cb = ctx->cb_split;
    p.cb_lanes = ctx->cb_lanes;
    p.out = out;
    p.flags = ctx->flags;
#define CALLB(D, K, BS) (out_f32 ? launch_dk<D, K, BS, float>(ctx, p, s) : launch_dk<D, K, BS, __half>(ctx, p, s))
    switch (static_bits(ctx->d, ctx->k, ctx->B)) {
        case 4: return CALLB(64, 2, 4);
        case 8: return CALLB(64, 2, 8);
        case 10: return CALLB(64, 4, 10);
        case 12: return CALLB(128, 8, 12);
        default: break;
    }
#undef CALLB
#define CALL(D, K) (out_f32 ? launch_dk<D, K, 0, float>(ctx, p, s) : launch_dk<D, K, 0, __half>(ctx, p, s))
    if (ctx->d == 64) {
        if (ctx->k == 1) return CALL(64, 1);
        if (ctx->k == 2) return CALL(64, 2);
        if (ctx->k == 4) return CALL(64, 4);
        return CALL(64, 8);
    }
    if (ctx->k == 1) return CALL(128, 1);
    if (ctx->k == 2) return CALL(128, 2);
    if (ctx->k == 4) return CALL(128, 4);
    return CALL(128, 8);
#undef CALL
}

}  // namespace fq
