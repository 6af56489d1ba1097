// Fused decode-into-attention [FibQuant §5: the fixed-address, random-access interface lets
// decompression run inside the attention kernel]. A query q attends over the T cached keys and
// values of its group straight from the code store; no decoded vector is written anywhere.
//
// With y_t = concat_b c_{i_tb} the rotated-domain decode and x_hat_t = nu_t Pi^T y_t [FibQuant §2.3]:
//
//   q . k_hat_t = nu_t (Pi q) . y_t = nu_t sum_b (Pi q)_b . c_{i_tb}          (scores)
//   o = Pi^T ( sum_t p_t nu^V_t y^V_t ) / sum_t p_t,  p_t = exp(s_t - max s)  (values)
//
// k <= 8: a CTA rotates the query once and, when it fits in shared memory, builds the per-query
// table L[n][b] = (Pi q)_b . c_n, so a key costs d/k table reads; otherwise the score takes the
// k-term dot product with the codeword. Values accumulate in the rotated domain and Pi^T is
// applied once per query. k = d: the rotated codebook rows Pi^T c_n (L2-resident) serve both the
// dot products and the value sums, so neither rotation is needed.
//
// Grouped queries. The QG queries of one cached group that a cluster serves (QG = 1 or 4) share
// every record read, index unpack and codeword read; each has its own rotated query, score table,
// partial scores, softmax state and value sums.
//
// Work split. The tokens of a query are divided over the S CTAs of a thread-block cluster; the
// warps of a CTA take 32-token tiles round-robin, each with its own online softmax (max, sum, z).
// The warps' partial results merge through shared memory, the CTAs' through distributed shared
// memory at CTA rank 0, which writes the output. There is no global scratch and one launch.
//
// Lane mapping (k <= 8), nb = d/k blocks: a tile is 32 tokens x nb blocks, processed 32 (token,
// block) pairs per step. nb >= 32: a step is nb/32-th of one token, lane l takes blocks l + 32 s.
// nb < 32: a step covers 32/nb tokens, lane l takes block l % nb of token group l / nb. Table rows
// are laid out [n][lane slot] (pitch max(nb, 32), duplicated across token groups), so the lanes of
// a step read 32 distinct banks. Per-lane partial scores are combined by a transposed butterfly
// (nb - 1 or 31 shuffles per tile) that leaves each lane with one token's score. Records are staged
// per warp in shared memory by cp.async, double-buffered one tile ahead.
// Kernel of the fused decode-into-attention, shared by the translation units that instantiate it
// (one query per cluster, and grouped queries). Host-side planning and launch are in fq_attend.cu.
#pragma once

#include <math.h>

#include <type_traits>

#include "fq_internal.h"
#include "fq_sm100.cuh"

namespace fq {
namespace attend_detail {

using namespace sm100;

constexpr int kMaxWarps = 16;
constexpr int kMinWarps = 4;
constexpr int kMaxSplit = 8;

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int Pending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(Pending) : "memory");
}

// A float in the shared memory of cluster CTA `rank`, at the offset of `p` in this CTA.
__device__ __forceinline__ float ld_cluster(const float *p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Each lane holds NP partial sums; afterwards lane l holds the sum over its aligned group of NP
// lanes of partial l % NP (recursive halving: each stage keeps half the values, adds the
// partner's copy of that half).
template <int NP>
__device__ __forceinline__ float transpose_sum(float (&v)[NP], int lane) {
#pragma unroll
    for (int h = NP / 2; h >= 1; h >>= 1) {
        const bool up = lane & h;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
    }
    return v[0];
}

// B-bit field at bit p of a staged word array. ONE: the field lies within one word (B divides
// 32 and the tile's fields start on multiples of B); otherwise it may straddle two words.
template <bool ONE>
__device__ __forceinline__ uint32_t field(const uint32_t *w, int p, uint32_t mask) {
    if constexpr (ONE)
        return (w[p >> 5] >> (p & 31)) & mask;
    else
        return __funnelshift_r(w[p >> 5], w[(p >> 5) + 1], p & 31) & mask;
}

// Codebook rows in shared memory. For k = 8 a row is two 16-byte halves; storing them swapped in
// rows with bit 2 of n set spreads the halves that the lanes of a quarter-warp read over all eight
// 4-bank groups (unswizzled, every first half falls in an even group).
template <int K>
__device__ __forceinline__ int codeword_slot(int n, int half) {
    return K == 8 ? n * 8 + 4 * (half ^ ((n >> 2) & 1)) : n * K + 4 * half;
}

template <int K>
__device__ __forceinline__ void load_codeword(const float *Cs, uint32_t n, float (&v)[K]) {
    if constexpr (K == 1) {
        v[0] = Cs[n];
    } else if constexpr (K == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(Cs + 2 * n);
        v[0] = a.x, v[1] = a.y;
    } else {
#pragma unroll
        for (int h = 0; h < K / 4; ++h) {
            const float4 a = *reinterpret_cast<const float4 *>(Cs + codeword_slot<K>(n, h));
            v[4 * h] = a.x, v[4 * h + 1] = a.y, v[4 * h + 2] = a.z, v[4 * h + 3] = a.w;
        }
    }
}

struct AttendArgs {
    const float *nu;
    const uint32_t *codes;
    const __half *q;       // [nq x D]
    float *out;            // [nq x D]
    const float *C;        // [N x K] (k <= 8) or the rotated codebook [N x D] (k = d)
    const float *Pi;       // [D x D]
    int64_t T, k_row0, v_row0, stride, q_per_group;
    float scale;
    int N, B, R;
    int split;             // CTAs per query = cluster size
    int buf_words;         // staging words per buffer
};

// Shared memory (floats), per served query: q[D], q~[D], the cluster slot {max, sum, -, -}, z[D],
// per-warp max[16], sum[16] and z[16 x D]; then the codebook (k <= 8), the score tables (if used,
// one per query), and per warp two staging buffers {nu of 32 keys, nu of 32 values, key record
// words, value record words}.
template <int D, int K, bool LUT, int QG>
__global__ void __launch_bounds__(QG == 1 ? kMaxWarps * 32 : 256)
attend_kernel(const AttendArgs a) {
    constexpr bool FULL = (K == D);
    constexpr int NB = D / K;
    constexpr int SPT = (NB >= 32) ? NB / 32 : 1;      // steps per token
    constexpr int TPS = (NB >= 32) ? 1 : 32 / NB;      // tokens per step
    constexpr int NP = (NB >= 32) ? 32 : (FULL ? 32 : NB);  // partial sums per lane
    constexpr int LP = (NB >= 32) ? NB : 32;           // score table pitch
    constexpr int ZA = FULL ? D / 32 : K * SPT;        // value accumulators per lane
    constexpr int QR = FULL ? D / 32 : (LUT ? 1 : K * SPT);   // query coordinates per lane

    extern __shared__ __align__(16) float sm[];
    float *qs = sm;                               // [QG][D]
    float *qt = qs + QG * D;                      // [QG][D]
    float *cm = qt + QG * D;                      // [QG][4]
    float *cz = cm + QG * 4;                      // [QG][D]
    float *wm = cz + QG * D;                      // [QG][kMaxWarps]
    float *wl = wm + QG * kMaxWarps;              // [QG][kMaxWarps]
    float *wz = wl + QG * kMaxWarps;              // [QG][kMaxWarps][D]
    float *Cs = wz + QG * kMaxWarps * D;
    float *Ls = Cs + (FULL ? 0 : a.N * K);        // [QG][N][LP]
    uint32_t *stage = reinterpret_cast<uint32_t *>(Ls + (LUT ? QG * a.N * LP : 0));

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const int64_t q0 = (int64_t)(blockIdx.x / a.split) * QG;   // first served query
    const int64_t group = q0 / a.q_per_group;
    const int N = a.N, B = a.B, R = a.R;
    const uint32_t mask = (uint32_t)N - 1u;
    const int64_t T = a.T;
    const int NLP = N * LP;

    // This CTA's tiles, dealt to its warps round-robin.
    const int64_t n_tiles = (T + 31) / 32;
    const int64_t tile_lo = n_tiles * rank / a.split, tile_hi = n_tiles * (rank + 1) / a.split;
    const int64_t kbase = a.k_row0 + group * a.stride, vbase = a.v_row0 + group * a.stride;
    const int RW = R + 2;
    uint32_t *my_stage = stage + (int64_t)warp * 2 * a.buf_words;

    auto issue = [&](int64_t tile, int buf) {
        uint32_t *st = my_stage + buf * a.buf_words;
        const int64_t t0 = tile * 32;
        const int nv = T - t0 < 32 ? (int)(T - t0) : 32;
        const int64_t kr = kbase + t0, vr = vbase + t0;
        if (lane < nv) {
            cp_async4(st + lane, a.nu + kr + lane);
            cp_async4(st + 32 + lane, a.nu + vr + lane);
        }
        const int64_t kw0 = (kr * R) >> 5, kw1 = ((kr + nv) * R - 1) >> 5;
        for (int64_t w = kw0 + lane; w <= kw1; w += 32) cp_async4(st + 64 + (w - kw0), a.codes + w);
        const int64_t vw0 = (vr * R) >> 5, vw1 = ((vr + nv) * R - 1) >> 5;
        for (int64_t w = vw0 + lane; w <= vw1; w += 32) cp_async4(st + 64 + RW + (w - vw0), a.codes + w);
        cp_async_commit();
    };

    // The first tile's records are requested before the tables are built, to overlap their latency.
    int64_t tile = tile_lo + warp;
    if (tile < tile_hi) issue(tile, 0);

    for (int i = threadIdx.x; i < QG * D; i += blockDim.x) qs[i] = __half2float(a.q[q0 * D + i]);
    if constexpr (!FULL)
        for (int i = threadIdx.x; i < N * K; i += blockDim.x)
            Cs[K == 8 ? codeword_slot<K>(i / 8, (i / 4) & 1) + (i & 3) : i] = __ldg(a.C + i);
    __syncthreads();
    if constexpr (!FULL) {
        // q~ = Pi q for every served query: 8 consecutive threads per (query, row), each a
        // contiguous chunk of the row, all of a thread's loads in flight together.
        constexpr int TPR = 8, CH = D / TPR;
        for (int rr = threadIdx.x / TPR; rr < QG * D; rr += (int)blockDim.x / TPR) {
            const int qi = rr / D, i = rr % D, part = threadIdx.x % TPR;
            const float4 *prow = reinterpret_cast<const float4 *>(a.Pi + (int64_t)i * D + part * CH);
            const float *qq = qs + qi * D + part * CH;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < CH / 4; ++j) {
                const float4 p = __ldg(prow + j);
                acc = fmaf(p.x, qq[4 * j], acc);
                acc = fmaf(p.y, qq[4 * j + 1], acc);
                acc = fmaf(p.z, qq[4 * j + 2], acc);
                acc = fmaf(p.w, qq[4 * j + 3], acc);
            }
#pragma unroll
            for (int o = TPR / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (part == 0) qt[qi * D + i] = acc;
        }
        __syncthreads();
        if constexpr (LUT) {
            for (int e = threadIdx.x; e < QG * NLP; e += blockDim.x) {
                const int qi = e / NLP, n = (e % NLP) / LP, slot = e % LP;
                const int b = (NB >= 32) ? slot : slot % NB;
                float c[K];
                load_codeword<K>(Cs, n, c);
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < K; ++j) acc = fmaf(qt[qi * D + b * K + j], c[j], acc);
                Ls[e] = acc;
            }
            __syncthreads();
        }
    }

    // Each lane's query coordinates: k <= 8 without a table, its blocks of q~; k = d, q itself.
    float qreg[QG][QR];
#pragma unroll
    for (int qi = 0; qi < QG; ++qi) {
        if constexpr (FULL) {
#pragma unroll
            for (int s = 0; s < D / 32; ++s) qreg[qi][s] = qs[qi * D + s * 32 + lane];
        } else if constexpr (!LUT) {
#pragma unroll
            for (int s = 0; s < SPT; ++s) {
                const int b = (NB >= 32) ? s * 32 + lane : lane % NB;
#pragma unroll
                for (int j = 0; j < K; ++j) qreg[qi][s * K + j] = qt[qi * D + b * K + j];
            }
        } else {
            qreg[qi][0] = 0.f;
        }
    }

    float m[QG], l[QG], z[QG][ZA];
#pragma unroll
    for (int qi = 0; qi < QG; ++qi) {
        m[qi] = -INFINITY;
        l[qi] = 0.f;
#pragma unroll
        for (int j = 0; j < ZA; ++j) z[qi][j] = 0.f;
    }

    for (int it = 0; tile < tile_hi; ++it, tile += nwarps) {
        const int buf = it & 1;
        if (tile + nwarps < tile_hi) {
            issue(tile + nwarps, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        const uint32_t *st = my_stage + buf * a.buf_words;
        const float *kn = reinterpret_cast<const float *>(st);
        const float *vn = kn + 32;
        const uint32_t *kw = st + 64, *vw = st + 64 + RW;
        const int64_t t0 = tile * 32;
        const int nv = T - t0 < 32 ? (int)(T - t0) : 32;
        const int ko = (int)(((kbase + t0) * R) & 31), vo = (int)(((vbase + t0) * R) & 31);
        const bool one_word = (32 % B == 0) && ((ko | vo) % B == 0);

        // Scores.
        float part[QG][NP];
#pragma unroll
        for (int qi = 0; qi < QG; ++qi)
#pragma unroll
            for (int p = 0; p < NP; ++p) part[qi][p] = 0.f;
        if constexpr (FULL) {
            const uint32_t my_idx = field<false>(kw, ko + lane * R, mask);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float *c = a.C + (int64_t)__shfl_sync(0xffffffffu, my_idx, t) * D;
                float cv[D / 32];
#pragma unroll
                for (int s = 0; s < D / 32; ++s) cv[s] = __ldg(c + s * 32 + lane);
#pragma unroll
                for (int qi = 0; qi < QG; ++qi) {
                    float acc = 0.f;
#pragma unroll
                    for (int s = 0; s < D / 32; ++s) acc = fmaf(qreg[qi][s], cv[s], acc);
                    part[qi][t] = acc;
                }
            }
        } else {
            auto scores = [&](auto one) {
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int t = (NB >= 32) ? j / SPT : j * TPS + lane / NB;
                    const int s = (NB >= 32) ? j % SPT : 0;
                    const int b = (NB >= 32) ? s * 32 + lane : lane % NB;
                    const uint32_t idx = field<decltype(one)::value>(kw, ko + t * R + b * B, mask);
                    if constexpr (LUT) {
                        const int col = (int)idx * LP + ((NB >= 32) ? b : lane);
#pragma unroll
                        for (int qi = 0; qi < QG; ++qi) part[qi][(NB >= 32) ? t : j] += Ls[qi * NLP + col];
                    } else {
                        float c[K];
                        load_codeword<K>(Cs, idx, c);
#pragma unroll
                        for (int qi = 0; qi < QG; ++qi) {
                            float v = 0.f;
#pragma unroll
                            for (int jj = 0; jj < K; ++jj) v = fmaf(qreg[qi][s * K + jj], c[jj], v);
                            part[qi][(NB >= 32) ? t : j] += v;
                        }
                    }
                }
            };
            if (one_word) scores(std::true_type{});
            else scores(std::false_type{});
        }
        const int tok = (NB >= 32 || FULL) ? lane : (lane % NB) * TPS + lane / NB;
        const bool valid = tok < nv;

        // Online softmax over this tile, per served query.
        float w[QG];
#pragma unroll
        for (int qi = 0; qi < QG; ++qi) {
            const float dot = transpose_sum<NP>(part[qi], lane);
            const float sc = valid ? a.scale * kn[tok] * dot : -INFINITY;
            const float m_new = fmaxf(m[qi], warp_max(sc));
            const float alpha = expf(m[qi] - m_new);
            const float p = valid ? expf(sc - m_new) : 0.f;
            l[qi] = l[qi] * alpha + warp_sum(p);
            m[qi] = m_new;
            w[qi] = valid ? p * vn[tok] : 0.f;
#pragma unroll
            for (int j = 0; j < ZA; ++j) z[qi][j] *= alpha;
        }

        // Values.
        if constexpr (FULL) {
            const uint32_t my_idx = field<false>(vw, vo + lane * R, mask);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float *c = a.C + (int64_t)__shfl_sync(0xffffffffu, my_idx, t) * D;
                float cv[D / 32];
#pragma unroll
                for (int s = 0; s < D / 32; ++s) cv[s] = __ldg(c + s * 32 + lane);
#pragma unroll
                for (int qi = 0; qi < QG; ++qi) {
                    const float wt = __shfl_sync(0xffffffffu, w[qi], t);
#pragma unroll
                    for (int s = 0; s < D / 32; ++s) z[qi][s] = fmaf(wt, cv[s], z[qi][s]);
                }
            }
        } else {
            auto values = [&](auto one) {
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int t = (NB >= 32) ? j / SPT : j * TPS + lane / NB;
                    const int s = (NB >= 32) ? j % SPT : 0;
                    const int b = (NB >= 32) ? s * 32 + lane : lane % NB;
                    const int src = (NB >= 32) ? t : (lane / NB) * NB + j;
                    const uint32_t idx = field<decltype(one)::value>(vw, vo + t * R + b * B, mask);
                    float c[K];
                    load_codeword<K>(Cs, idx, c);
#pragma unroll
                    for (int qi = 0; qi < QG; ++qi) {
                        const float wt = __shfl_sync(0xffffffffu, w[qi], src);
#pragma unroll
                        for (int jj = 0; jj < K; ++jj) z[qi][s * K + jj] = fmaf(wt, c[jj], z[qi][s * K + jj]);
                    }
                }
            };
            if (one_word) values(std::true_type{});
            else values(std::false_type{});
        }
        __syncwarp();   // the next issue overwrites this buffer
    }

    // Warp results -> shared memory (token groups of one block summed first when nb < 32).
#pragma unroll
    for (int qi = 0; qi < QG; ++qi) {
        if constexpr (!FULL && NB < 32) {
#pragma unroll
            for (int o = NB; o < 32; o <<= 1)
#pragma unroll
                for (int j = 0; j < ZA; ++j) z[qi][j] += __shfl_xor_sync(0xffffffffu, z[qi][j], o);
        }
        float *wzq = wz + (qi * kMaxWarps + warp) * D;
        if constexpr (FULL) {
#pragma unroll
            for (int s = 0; s < D / 32; ++s) wzq[s * 32 + lane] = z[qi][s];
        } else if constexpr (NB >= 32) {
#pragma unroll
            for (int s = 0; s < SPT; ++s)
#pragma unroll
                for (int j = 0; j < K; ++j) wzq[(s * 32 + lane) * K + j] = z[qi][s * K + j];
        } else if (lane < NB) {
#pragma unroll
            for (int j = 0; j < K; ++j) wzq[lane * K + j] = z[qi][j];
        }
        if (lane == 0) {
            wm[qi * kMaxWarps + warp] = m[qi];
            wl[qi * kMaxWarps + warp] = l[qi];
        }
    }
    __syncthreads();
    for (int o = threadIdx.x; o < QG * D; o += blockDim.x) {
        const int qi = o / D, i = o % D;
        float M = -INFINITY;
        for (int w = 0; w < nwarps; ++w) M = fmaxf(M, wm[qi * kMaxWarps + w]);
        float L = 0.f, Z = 0.f;
        if (M > -INFINITY) {
            for (int w = 0; w < nwarps; ++w) {
                const float f = expf(wm[qi * kMaxWarps + w] - M);
                L = fmaf(f, wl[qi * kMaxWarps + w], L);
                Z = fmaf(f, wz[(qi * kMaxWarps + w) * D + i], Z);
            }
        }
        cz[qi * D + i] = Z;
        if (i == 0) {
            cm[qi * 4] = M;
            cm[qi * 4 + 1] = L;
        }
    }
    cluster_sync();
    if (rank == 0) {
        for (int o = threadIdx.x; o < QG * D; o += blockDim.x) {
            const int qi = o / D, i = o % D;
            float M = -INFINITY;
            for (int r = 0; r < a.split; ++r) M = fmaxf(M, ld_cluster(cm + qi * 4, r));
            float L = 0.f, Z = 0.f;
            for (int r = 0; r < a.split; ++r) {
                const float Mr = ld_cluster(cm + qi * 4, r);
                const float f = Mr > -INFINITY ? expf(Mr - M) : 0.f;
                L = fmaf(f, ld_cluster(cm + qi * 4 + 1, r), L);
                Z = fmaf(f, ld_cluster(cz + qi * D + i, r), Z);
            }
            qs[qi * D + i] = Z / L;
        }
    }
    cluster_sync();   // every CTA's slots have been read; rank 0's qs holds z / sum
    if (rank != 0) return;
    if constexpr (FULL) {
        for (int o = threadIdx.x; o < QG * D; o += blockDim.x) a.out[q0 * D + o] = qs[o];
    } else {
        // o = Pi^T (z / sum): 8 row ranges per (query, output column), partial sums through wz.
        constexpr int PARTS = 8, ROWS = D / PARTS;
        for (int o = threadIdx.x; o < QG * D * PARTS; o += blockDim.x) {
            const int part = o / (QG * D), qj = o % (QG * D), qi = qj / D, j = qj % D;
            float acc = 0.f;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int i = part * ROWS + r;
                acc = fmaf(__ldg(a.Pi + (int64_t)i * D + j), qs[qi * D + i], acc);
            }
            wz[part * QG * D + qj] = acc;
        }
        __syncthreads();
        for (int o = threadIdx.x; o < QG * D; o += blockDim.x) {
            float acc = 0.f;
#pragma unroll
            for (int part = 0; part < PARTS; ++part) acc += wz[part * QG * D + o];
            a.out[q0 * D + o] = acc;
        }
    }
}

template <int D, int K, bool LUT, int QG>
const void *kernel_of() { return reinterpret_cast<const void *>(&attend_kernel<D, K, LUT, QG>); }

template <int QG>
const void *select_kernel_q(int d, int k, bool lut) {
#define FQ_ATTEND_CASE(DD, KK) \
    if (d == DD && k == KK) return lut ? kernel_of<DD, KK, true, QG>() : kernel_of<DD, KK, false, QG>();
    FQ_ATTEND_CASE(64, 1)
    FQ_ATTEND_CASE(64, 2)
    FQ_ATTEND_CASE(64, 4)
    FQ_ATTEND_CASE(64, 8)
    FQ_ATTEND_CASE(128, 1)
    FQ_ATTEND_CASE(128, 2)
    FQ_ATTEND_CASE(128, 4)
    FQ_ATTEND_CASE(128, 8)
#undef FQ_ATTEND_CASE
    if (d == 64 && k == 64) return kernel_of<64, 64, false, QG>();
    return nullptr;
}

}  // namespace attend_detail

// The kernel serving QG = 4 queries per cluster (fq_attend_gqa.cu).
const void *attend_kernel_gqa(int d, int k, bool lut);

}  // namespace fq
