// Iterated-map archive of symbol streams ("Fractal KV-Cache Archives", Method 1): encode / append,
// full decode and random access kernels and their launches (the C ABI is in fa_api.cu).
//
// Each segment of L symbols is independent (it starts at the origin), so one device thread owns one
// segment (encode, decode) or one lookup (random access). The work is a chain of dependent fp64
// steps per thread: GB300 runs fp64 at a small fraction of its fp32 rate, so these kernels are
// bound by the fp64 pipe, not by memory (2 bytes per symbol in, 16 bytes per segment out).
//   * forward step, per coordinate: t = p - V, then p = r t + V as one fused multiply-add (two fp64
//     instructions, one rounding fewer than the three-operation form, so the error bound behind
//     the segment length still holds); a fixed instruction sequence makes anchors identical
//     whatever the split of a stream into append calls;
//   * backward step: the cell is found in fp32 (the angle of the point rounded to the nearest
//     vertex; the cells are disjoint with a margin the context guarantees to be at least 2e-5, far
//     above fp32 error), the point is checked to lie within r + 3/4 of the margin of that cell's
//     centre, then the map is inverted in fp64 as p = V + (p - V) / r with the quotient taken as a
//     fused multiply by 1/r. The fp32 copy of the point is cut from the fp64 bits with integer
//     instructions, which measured faster in these kernels than the hardware fp64-to-fp32
//     conversion.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"

namespace {

using fa::kMaxSegment;
using fa::kThreads;
constexpr uint16_t kBad = 0xFFFFu;

struct Tables {
    const double2 *V;
    const float2 *Cf;
    int N;
    int L;
    double r;
    double rinv;
    float scaleN;
    float lim2;
    uint32_t *flags;
};

Tables tables_of(const fa_ctx *c) {
    return Tables{c->V, c->Cf, c->N, c->L, c->r, c->rinv, c->scaleN, c->lim2, c->flags};
}

__device__ __forceinline__ void forward_step(double &x, double &y, double2 v, double r) {
    x = __fma_rn(r, __dsub_rn(x, v.x), v.x);
    y = __fma_rn(r, __dsub_rn(y, v.y), v.y);
}

__device__ __forceinline__ void backward_step(double &x, double &y, double2 v, double rinv) {
    x = __fma_rn(__dsub_rn(x, v.x), rinv, v.x);
    y = __fma_rn(__dsub_rn(y, v.y), rinv, v.y);
}

// x as an fp32 number with its mantissa truncated to 23 bits (relative error below 2^-23), from
// the IEEE-754 fields: magnitudes below the fp32 normal range become zero; infinities and NaNs stay
// infinities and NaNs.
__device__ __forceinline__ float to_f32_trunc(double x) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(x);
    const uint32_t hi = (uint32_t)(b >> 32);
    const uint32_t sign = hi & 0x80000000u;
    const int e = (int)((hi >> 20) & 0x7ffu) - 1023 + 127;
    const uint32_t m = (uint32_t)(b >> 29) & 0x7fffffu;
    if (e <= 0) return __uint_as_float(sign);
    if (e >= 255) return __uint_as_float(sign | 0x7f800000u | (m ? 0x400000u : 0u));
    return __uint_as_float(sign | ((uint32_t)e << 23) | m);
}

// The symbol whose cell holds (x, y); sets `bad` when the point is not within reach of that cell
// (NaN included). Returns the vertex in v.
__device__ __forceinline__ int find_cell(double x, double y, const Tables &t, double2 &v, bool &bad) {
    const float fx = to_f32_trunc(x), fy = to_f32_trunc(y);
    int c = __float2int_rn(atan2f(fy, fx) * t.scaleN);
    if (c < 0) c += t.N;
    c = min(max(c, 0), t.N - 1);
    const float2 ctr = __ldg(t.Cf + c);
    const float dx = fx - ctr.x, dy = fy - ctr.y;
    if (!(fmaf(dx, dx, dy * dy) <= t.lim2)) bad = true;
    v = __ldg(t.V + c);
    return c;
}

// One thread per touched segment (stream q, segment s0 + j): continue or start the segment with the
// appended symbols at positions [max(s L, T_old), min(s L + L, T_old + n_new)).
__global__ void __launch_bounds__(kThreads)
archive_encode(Tables t, const uint16_t *__restrict__ sym, int64_t n_streams, int64_t n_new, int64_t S_cap,
               int64_t T_old, int64_t s0, int64_t n_seg, double2 *__restrict__ anchors) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_streams * n_seg) return;
    const int64_t q = i / n_seg, s = s0 + (i - q * n_seg);
    int64_t lo = s * t.L;
    int64_t hi = lo + t.L;
    if (hi > T_old + n_new) hi = T_old + n_new;
    double2 *a = anchors + q * S_cap + s;
    double x = 0.0, y = 0.0;
    if (lo < T_old) {               // the partial last segment continues from its stored point
        const double2 p = *a;
        x = p.x;
        y = p.y;
        lo = T_old;
    }
    const uint16_t *row = sym + q * n_new;
    auto src = [&](int64_t p) -> uint32_t { return row[p - T_old]; };   // the symbol at position p
    bool bad = false;
    // The loads of a step do not depend on the point, so they run ahead of the fp64 chain: the
    // symbol two steps ahead and the vertex one step ahead.
    auto vertex = [&](uint32_t c) {
        if (c >= (uint32_t)t.N) {
            bad = true;
            c = 0;
        }
        return __ldg(t.V + c);
    };
    uint32_t c_next = lo + 1 < hi ? src(lo + 1) : 0u;
    double2 v = lo < hi ? vertex(src(lo)) : make_double2(0.0, 0.0);
    for (int64_t pos = lo; pos < hi; ++pos) {
        const double2 vc = v;
        if (pos + 1 < hi) {
            v = vertex(c_next);
            if (pos + 2 < hi) c_next = src(pos + 2);
        }
        forward_step(x, y, vc, t.r);
    }
    if (bad) {
        x = y = __longlong_as_double(0x7ff8000000000000LL);
        atomicOr(t.flags, (uint32_t)FA_FLAG_SYMBOL);
    }
    *a = make_double2(x, y);
}

// One thread per segment: every symbol, from the last position back to the first.
__global__ void __launch_bounds__(kThreads)
archive_decode(Tables t, const double2 *__restrict__ anchors, int64_t n_streams, int64_t S_cap, int64_t T,
               int64_t S, uint16_t *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_streams * S) return;
    const int64_t q = i / S, s = i - q * S;
    const int len = (int)min((int64_t)t.L, T - s * t.L);
    const double2 p = anchors[q * S_cap + s];
    double x = p.x, y = p.y;
    uint16_t *o = out + q * T + s * t.L;
    bool bad = false;
    for (int k = len - 1; k >= 0; --k) {
        double2 v;
        const int c = find_cell(x, y, t, v, bad);
        o[k] = bad ? kBad : (uint16_t)c;
        if (k) backward_step(x, y, v, t.rinv);
    }
    if (bad) atomicOr(t.flags, (uint32_t)FA_FLAG_CORRUPT);
}

// Random access: backward from each lookup's segment anchor down to the wanted position only.
//
// A lookup needs between 0 and L - 1 backward steps, so one lookup per thread would leave most lanes
// of a warp idle while the longest walk finishes, and every fp64 instruction costs the pipe the same
// whatever its active lanes. Instead each warp owns a run of `per_warp` lookups as a queue:
//   1. the warp turns every position of its run into (anchor index, walk length, target) in shared
//      memory, all lanes together, so the integer divisions run convergent;
//   2. a lane that answers its lookup takes the next one from the queue for the following round, so
//      the fp64 backward step of each round is shared by most lanes (for walks of 0 .. 6 steps a lane
//      walks in 3 of every 4 rounds, and the queue keeps about 4/5 of the lanes busy to the end);
//   3. each lane keeps the next lookup's anchor load in flight (slot A) and holds the one after as a
//      queue index (slot B); B slots are handed out once per round through a warp ballot.
constexpr int kAccessMinPerLane = 4;
constexpr int kAccessMaxPerLane = 16;
constexpr int kAccessWarpsPerSm = 24;
constexpr int kAccessOutOfRange = -1;

__global__ void __launch_bounds__(kThreads)
archive_access(Tables t, const double2 *__restrict__ anchors, int64_t n_streams, int64_t T_cap, int64_t S_cap,
               int64_t T, const int64_t *__restrict__ pos, int64_t n, int per_warp, uint16_t *__restrict__ out) {
    extern __shared__ __align__(16) unsigned char access_smem[];
    const int lane = threadIdx.x & 31, warp_in_block = threadIdx.x >> 5;
    const int64_t begin = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * per_warp;
    if (begin >= n) return;                                      // uniform over the warp
    const int cnt = (int)min((int64_t)per_warp, n - begin);
    int64_t *seg = reinterpret_cast<int64_t *>(access_smem) + (size_t)warp_in_block * per_warp;
    uint16_t *walk = reinterpret_cast<uint16_t *>(reinterpret_cast<int64_t *>(access_smem) + (size_t)(kThreads / 32) * per_warp)
                     + (size_t)warp_in_block * per_warp;

    // 1. positions -> (anchor index or kAccessOutOfRange, first position k | target off << 8)
    for (int j = lane; j < cnt; j += 32) {
        const int64_t g = pos[begin + j];
        const int64_t q = g >= 0 ? g / T_cap : -1;
        const int64_t tt = g - q * T_cap;
        if (g < 0 || q >= n_streams || tt >= T) {
            seg[j] = kAccessOutOfRange;
            walk[j] = 0;
        } else {
            const int64_t s = tt / t.L;
            seg[j] = q * S_cap + s;
            walk[j] = (uint16_t)((min((int64_t)t.L, T - s * t.L) - 1) | ((tt - s * t.L) << 8));
        }
    }
    __syncwarp();

    const unsigned below = (1u << lane) - 1u;
    int head = 0;                                                // next unclaimed queue entry (warp-uniform)
    int b = -1;                                                  // slot B: a queue entry, or -1
    auto refill = [&]() {
        const bool need = b < 0;
        const unsigned mask = __ballot_sync(0xffffffffu, need);
        const int idx = head + __popc(mask & below);
        if (need && idx < cnt) b = idx;
        head += __popc(mask);
    };

    double2 a_anchor = make_double2(0.0, 0.0);                   // slot A: anchor load in flight
    int a = -1;
    int64_t a_seg = 0;
    auto promote = [&]() {                                       // A <- B
        a = b;
        b = -1;
        if (a >= 0) {
            a_seg = seg[a];
            if (a_seg != kAccessOutOfRange) a_anchor = anchors[a_seg];
        }
    };

    double x = 0.0, y = 0.0;                                     // the current lookup
    int cur = 0, k = 0, off = 0;
    bool bad = false, corrupt = false, range = false;
    auto take = [&]() -> bool {                                  // current <- A; false if none
        while (a >= 0) {
            cur = a;
            if (a_seg == kAccessOutOfRange) {                    // answered without a walk
                out[begin + cur] = kBad;
                range = true;
                promote();
                continue;
            }
            const int w = walk[cur];
            x = a_anchor.x;
            y = a_anchor.y;
            k = w & 0xff;
            off = w >> 8;
            bad = false;
            promote();
            return true;
        }
        return false;
    };

    refill();
    promote();
    refill();
    bool has = take();
    refill();
    // Every round either moves some lane one step down its walk or hands out queued lookups, so the
    // loop ends by itself; the cap only bounds it for the record.
    const int cap = (per_warp + 4) * (kMaxSegment + 2);
    for (int round = 0; round < cap && __any_sync(0xffffffffu, has || a >= 0 || b >= 0); ++round) {
        if (!has) {
            if (a < 0 && b >= 0) promote();
            has = take();
        }
        if (has) {
            double2 v;
            const int c = find_cell(x, y, t, v, bad);
            if (k > off) {
                backward_step(x, y, v, t.rinv);
                --k;
            } else {                                             // answered: the next lookup starts next round
                out[begin + cur] = bad ? kBad : (uint16_t)c;
                corrupt |= bad;
                has = take();
            }
        }
        refill();
    }
    if (corrupt) atomicOr(t.flags, (uint32_t)FA_FLAG_CORRUPT);
    if (range) atomicOr(t.flags, (uint32_t)FA_FLAG_RANGE);
}

unsigned blocks_for(int64_t threads) { return (unsigned)((threads + kThreads - 1) / kThreads); }

}  // namespace

namespace fa {

cudaError_t launch_encode(const fa_ctx *c, const uint16_t *sym, int64_t n_streams, int64_t n_new, int64_t S_cap,
                          int64_t T_old, int64_t s0, int64_t n_seg, double *anchors, cudaStream_t s) {
    archive_encode<<<blocks_for(n_streams * n_seg), kThreads, 0, s>>>(tables_of(c), sym, n_streams, n_new, S_cap,
                                                                     T_old, s0, n_seg,
                                                                     reinterpret_cast<double2 *>(anchors));
    return cudaGetLastError();
}

cudaError_t launch_decode(const fa_ctx *c, const double *anchors, int64_t n_streams, int64_t S_cap, int64_t T,
                          int64_t S, uint16_t *out, cudaStream_t s) {
    archive_decode<<<blocks_for(n_streams * S), kThreads, 0, s>>>(
        tables_of(c), reinterpret_cast<const double2 *>(anchors), n_streams, S_cap, T, S, out);
    return cudaGetLastError();
}

cudaError_t launch_access(const fa_ctx *c, const double *anchors, int64_t n_streams, int64_t T_cap, int64_t S_cap,
                          int64_t T, const int64_t *pos, int64_t n, uint16_t *out, cudaStream_t s) {
    // Queue length per warp: enough warps for about kAccessWarpsPerSm per SM, 4 to 16 lookups per lane.
    int64_t per_lane = (n + 32LL * c->num_sms * kAccessWarpsPerSm - 1) / (32LL * c->num_sms * kAccessWarpsPerSm);
    per_lane = per_lane < kAccessMinPerLane ? kAccessMinPerLane : (per_lane > kAccessMaxPerLane ? kAccessMaxPerLane : per_lane);
    const int per_warp = (int)(32 * per_lane);
    const int64_t warps = (n + per_warp - 1) / per_warp;
    const size_t smem = (size_t)(kThreads / 32) * per_warp * (sizeof(int64_t) + sizeof(uint16_t));
    archive_access<<<blocks_for(warps * 32), kThreads, smem, s>>>(tables_of(c), reinterpret_cast<const double2 *>(anchors),
                                                                  n_streams, T_cap, S_cap, T, pos, n, per_warp, out);
    return cudaGetLastError();
}

}  // namespace fa
