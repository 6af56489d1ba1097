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
#include <math.h>

#include <algorithm>
#include <type_traits>

#include "fq_internal.h"
#include "fq_sm100.cuh"

namespace fq {
namespace {

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

// Shared memory (floats): q[D], q~[D], cluster slot {max, sum, -, -} and z[D], per-warp max[16],
// sum[16], z[16 x D], then the codebook (k <= 8), the score table (if used), and per warp two
// staging buffers {nu of 32 keys, nu of 32 values, key record words, value record words}.
template <int D, int K, bool LUT>
__global__ void __launch_bounds__(kMaxWarps * 32)
attend_kernel(const AttendArgs a) {
    constexpr bool FULL = (K == D);
    constexpr int NB = D / K;
    constexpr int SPT = (NB >= 32) ? NB / 32 : 1;      // steps per token
    constexpr int TPS = (NB >= 32) ? 1 : 32 / NB;      // tokens per step
    constexpr int NP = (NB >= 32) ? 32 : (FULL ? 32 : NB);  // partial sums per lane
    constexpr int LP = (NB >= 32) ? NB : 32;           // score table pitch
    constexpr int ZA = FULL ? D / 32 : K * SPT;        // value accumulators per lane

    extern __shared__ __align__(16) float sm[];
    float *qs = sm;
    float *qt = qs + D;
    float *cm = qt + D;
    float *cz = cm + 4;
    float *wm = cz + D;
    float *wl = wm + kMaxWarps;
    float *wz = wl + kMaxWarps;
    float *Cs = wz + kMaxWarps * D;
    float *Ls = Cs + (FULL ? 0 : a.N * K);
    uint32_t *stage = reinterpret_cast<uint32_t *>(Ls + (LUT ? a.N * LP : 0));

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const int64_t query = blockIdx.x / a.split;
    const int64_t group = query / a.q_per_group;
    const int N = a.N, B = a.B, R = a.R;
    const uint32_t mask = (uint32_t)N - 1u;
    const int64_t T = a.T;

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

    for (int i = threadIdx.x; i < D; i += blockDim.x) qs[i] = __half2float(a.q[query * D + i]);
    if constexpr (!FULL)
        for (int i = threadIdx.x; i < N * K; i += blockDim.x)
            Cs[K == 8 ? codeword_slot<K>(i / 8, (i / 4) & 1) + (i & 3) : i] = __ldg(a.C + i);
    __syncthreads();
    if constexpr (!FULL) {
        // q~ = Pi q: tpr consecutive threads per row (whole warps), each a contiguous chunk of it,
        // with all of a thread's loads in flight together.
        int tpr = 1;
        while (tpr < 8 && 2 * tpr * D <= (int)blockDim.x) tpr *= 2;
        if ((int)threadIdx.x < tpr * D) {
            const int i = threadIdx.x / tpr, part = threadIdx.x % tpr, chunk = D / tpr;
            const float4 *prow = reinterpret_cast<const float4 *>(a.Pi + (int64_t)i * D + part * chunk);
            const float *qq = qs + part * chunk;
            float acc = 0.f;
#pragma unroll 8
            for (int j = 0; j < chunk / 4; ++j) {
                const float4 p = __ldg(prow + j);
                acc = fmaf(p.x, qq[4 * j], acc);
                acc = fmaf(p.y, qq[4 * j + 1], acc);
                acc = fmaf(p.z, qq[4 * j + 2], acc);
                acc = fmaf(p.w, qq[4 * j + 3], acc);
            }
            for (int o = tpr / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (part == 0) qt[i] = acc;
        }
        __syncthreads();
        if constexpr (LUT) {
            for (int e = threadIdx.x; e < N * LP; e += blockDim.x) {
                const int n = e / LP, slot = e % LP;
                const int b = (NB >= 32) ? slot : slot % NB;
                float c[K];
                load_codeword<K>(Cs, n, c);
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < K; ++j) acc = fmaf(qt[b * K + j], c[j], acc);
                Ls[e] = acc;
            }
            __syncthreads();
        }
    }

    // The lane's query coordinates: k <= 8 without a table: its blocks of q~; k = d: q itself.
    float qreg[FULL ? D / 32 : (LUT ? 1 : K * SPT)];
    if constexpr (FULL) {
#pragma unroll
        for (int s = 0; s < D / 32; ++s) qreg[s] = qs[s * 32 + lane];
    } else if constexpr (!LUT) {
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            const int b = (NB >= 32) ? s * 32 + lane : lane % NB;
#pragma unroll
            for (int j = 0; j < K; ++j) qreg[s * K + j] = qt[b * K + j];
        }
    }

    float m = -INFINITY, l = 0.f;
    float z[ZA];
#pragma unroll
    for (int j = 0; j < ZA; ++j) z[j] = 0.f;

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
        float part[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) part[p] = 0.f;
        if constexpr (FULL) {
            const uint32_t my_idx = field<false>(kw, ko + lane * R, mask);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float *c = a.C + (int64_t)__shfl_sync(0xffffffffu, my_idx, t) * D;
                float acc = 0.f;
#pragma unroll
                for (int s = 0; s < D / 32; ++s) acc = fmaf(qreg[s], __ldg(c + s * 32 + lane), acc);
                part[t] = acc;
            }
        } else {
            auto scores = [&](auto one_word) {
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int t = (NB >= 32) ? j / SPT : j * TPS + lane / NB;
                const int s = (NB >= 32) ? j % SPT : 0;
                const int b = (NB >= 32) ? s * 32 + lane : lane % NB;
                const uint32_t idx = field<decltype(one_word)::value>(kw, ko + t * R + b * B, mask);
                float v;
                if constexpr (LUT) {
                    v = Ls[idx * LP + ((NB >= 32) ? b : lane)];
                } else {
                    float c[K];
                    load_codeword<K>(Cs, idx, c);
                    v = 0.f;
#pragma unroll
                    for (int jj = 0; jj < K; ++jj) v = fmaf(qreg[s * K + jj], c[jj], v);
                }
                part[(NB >= 32) ? t : j] += v;
            }
            };
            if (one_word) scores(std::true_type{});
            else scores(std::false_type{});
        }
        const float dot = transpose_sum<NP>(part, lane);
        const int tok = (NB >= 32 || FULL) ? lane : (lane % NB) * TPS + lane / NB;
        const bool valid = tok < nv;
        const float sc = valid ? a.scale * kn[tok] * dot : -INFINITY;

        // Online softmax over this tile.
        const float m_new = fmaxf(m, warp_max(sc));
        const float alpha = expf(m - m_new);
        const float p = valid ? expf(sc - m_new) : 0.f;
        l = l * alpha + warp_sum(p);
        m = m_new;
        const float w = valid ? p * vn[tok] : 0.f;
#pragma unroll
        for (int j = 0; j < ZA; ++j) z[j] *= alpha;

        // Values.
        if constexpr (FULL) {
            const uint32_t my_idx = field<false>(vw, vo + lane * R, mask);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float wt = __shfl_sync(0xffffffffu, w, t);
                const float *c = a.C + (int64_t)__shfl_sync(0xffffffffu, my_idx, t) * D;
#pragma unroll
                for (int s = 0; s < D / 32; ++s) z[s] = fmaf(wt, __ldg(c + s * 32 + lane), z[s]);
            }
        } else {
            auto values = [&](auto one_word) {
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int t = (NB >= 32) ? j / SPT : j * TPS + lane / NB;
                const int s = (NB >= 32) ? j % SPT : 0;
                const int b = (NB >= 32) ? s * 32 + lane : lane % NB;
                const int src = (NB >= 32) ? t : (lane / NB) * NB + j;
                const float wt = __shfl_sync(0xffffffffu, w, src);
                const uint32_t idx = field<decltype(one_word)::value>(vw, vo + t * R + b * B, mask);
                float c[K];
                load_codeword<K>(Cs, idx, c);
#pragma unroll
                for (int jj = 0; jj < K; ++jj) z[s * K + jj] = fmaf(wt, c[jj], z[s * K + jj]);
            }
            };
            if (one_word) values(std::true_type{});
            else values(std::false_type{});
        }
        __syncwarp();   // the next issue overwrites this buffer
    }

    // Warp results -> shared memory (token groups of one block summed first when nb < 32).
    if constexpr (!FULL && NB < 32) {
#pragma unroll
        for (int o = NB; o < 32; o <<= 1)
#pragma unroll
            for (int j = 0; j < ZA; ++j) z[j] += __shfl_xor_sync(0xffffffffu, z[j], o);
    }
    if constexpr (FULL) {
#pragma unroll
        for (int s = 0; s < D / 32; ++s) wz[warp * D + s * 32 + lane] = z[s];
    } else if constexpr (NB >= 32) {
#pragma unroll
        for (int s = 0; s < SPT; ++s)
#pragma unroll
            for (int j = 0; j < K; ++j) wz[warp * D + (s * 32 + lane) * K + j] = z[s * K + j];
    } else if (lane < NB) {
#pragma unroll
        for (int j = 0; j < K; ++j) wz[warp * D + lane * K + j] = z[j];
    }
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
    __syncthreads();
    if (threadIdx.x < D) {
        const int i = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < nwarps; ++w) M = fmaxf(M, wm[w]);
        float L = 0.f, Z = 0.f;
        if (M > -INFINITY) {
            for (int w = 0; w < nwarps; ++w) {
                const float f = expf(wm[w] - M);
                L = fmaf(f, wl[w], L);
                Z = fmaf(f, wz[w * D + i], Z);
            }
        }
        cz[i] = Z;
        if (i == 0) {
            cm[0] = M;
            cm[1] = L;
        }
    }
    cluster_sync();
    if (rank == 0 && threadIdx.x < D) {
        const int i = threadIdx.x;
        float M = -INFINITY;
        for (int r = 0; r < a.split; ++r) M = fmaxf(M, ld_cluster(cm, r));
        float L = 0.f, Z = 0.f;
        for (int r = 0; r < a.split; ++r) {
            const float Mr = ld_cluster(cm, r);
            const float f = Mr > -INFINITY ? expf(Mr - M) : 0.f;
            L = fmaf(f, ld_cluster(cm + 1, r), L);
            Z = fmaf(f, ld_cluster(cz + i, r), Z);
        }
        qs[i] = Z / L;
    }
    cluster_sync();   // every CTA's slots have been read; rank 0's qs holds z / sum
    if (rank != 0) return;
    if constexpr (FULL) {
        if (threadIdx.x < D) a.out[query * D + threadIdx.x] = qs[threadIdx.x];
    } else {
        // o = Pi^T (z / sum): `parts` row ranges per output column, partial sums through wz.
        int parts = 1;
        while (parts < 8 && 2 * parts * D <= (int)blockDim.x) parts *= 2;
        if ((int)threadIdx.x < parts * D) {
            const int j = threadIdx.x % D, part = threadIdx.x / D, rows = D / parts;
            float o = 0.f;
#pragma unroll 8
            for (int r = 0; r < rows; ++r) {
                const int i = part * rows + r;
                o = fmaf(__ldg(a.Pi + (int64_t)i * D + j), qs[i], o);
            }
            wz[part * D + j] = o;
        }
        __syncthreads();
        if (threadIdx.x < D) {
            float o = 0.f;
            for (int part = 0; part < parts; ++part) o += wz[part * D + threadIdx.x];
            a.out[query * D + threadIdx.x] = o;
        }
    }
}

template <int D, int K, bool LUT>
const void *kernel_of() { return reinterpret_cast<const void *>(&attend_kernel<D, K, LUT>); }

const void *select_kernel(int d, int k, bool lut) {
#define FQ_ATTEND_CASE(DD, KK)                                                            \
    if (d == DD && k == KK) return lut ? kernel_of<DD, KK, true>() : kernel_of<DD, KK, false>();
    FQ_ATTEND_CASE(64, 1)
    FQ_ATTEND_CASE(64, 2)
    FQ_ATTEND_CASE(64, 4)
    FQ_ATTEND_CASE(64, 8)
    FQ_ATTEND_CASE(128, 1)
    FQ_ATTEND_CASE(128, 2)
    FQ_ATTEND_CASE(128, 4)
    FQ_ATTEND_CASE(128, 8)
#undef FQ_ATTEND_CASE
    if (d == 64 && k == 64) return kernel_of<64, 64, false>();
    return nullptr;
}

int buf_words(int R) { return (2 * (R + 2) + 64 + 3) & ~3; }

size_t table_bytes(const fq_ctx *c, bool lut) {
    const int d = c->d, k = c->k, nb = d / k;
    size_t f = 3 * (size_t)d + 4 + 2 * kMaxWarps + (size_t)kMaxWarps * d;
    if (k != d) f += (size_t)c->N * k;
    if (lut) f += (size_t)c->N * (nb >= 32 ? nb : 32);
    return f * sizeof(float);
}

}  // namespace

cudaError_t prepare_attend(fq_ctx *c) {
    c->attend_nwarps = 0;
    const size_t per_warp = 2 * (size_t)buf_words(c->R) * sizeof(uint32_t);
    const size_t limit = (size_t)c->smem_optin;
    const bool lut = c->k != c->d && table_bytes(c, true) + kMaxWarps * per_warp <= limit;
    const size_t tables = table_bytes(c, lut);
    if (tables + kMinWarps * per_warp > limit) return cudaSuccess;   // fq_attend reports FQ_EINVAL
    const int nwarps = (int)std::min<size_t>(kMaxWarps, (limit - tables) / per_warp);
    const size_t smem = tables + nwarps * per_warp;
    const void *fn = select_kernel(c->d, c->k, lut);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // Co-resident CTAs for each cluster size (registers, shared memory and cluster placement all
    // counted by the runtime's occupancy query); 0 where the size cannot be placed.
    int max_split = 0;
    for (int s = 1; s <= kMaxSplit; ++s) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(s);
        cfg.blockDim = dim3(32 * nwarps);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = s;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (e != cudaSuccess) return e;
        c->attend_slots[s] = n * s;
        if (n > 0) max_split = s;
    }
    if (!max_split) return cudaSuccess;
    c->attend_lut = lut;
    c->attend_nwarps = nwarps;
    c->attend_smem = smem;
    c->attend_max_split = max_split;
    return cudaSuccess;
}

int attend_split(const fq_ctx *c, int64_t n_queries, int64_t T) {
    const int64_t n_tiles = (T + 31) / 32;
    // Minimise waves x (tokens per CTA + fixed per-CTA cost in token units).
    const int nb = c->d / c->k;
    const double fixed = 64.0 + (c->attend_lut ? (double)c->N * (nb >= 32 ? nb : 32) / nb / 2 : 0.0);
    int best = 1;
    double best_cost = 0;
    for (int s = 1; s <= c->attend_max_split && s <= n_tiles; ++s) {
        const int64_t slots = c->attend_slots[s];
        if (slots <= 0) continue;
        const int64_t ctas = n_queries * s;
        const double waves = (double)((ctas + slots - 1) / slots);
        const double cost = waves * ((double)T / s + fixed);
        if (best_cost == 0 || cost < best_cost * 0.98) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

cudaError_t launch_attend(const fq_ctx *c, const float *nu, const uint32_t *codes, const __half *q,
                          int64_t n_queries, int64_t q_per_group, int64_t T, int64_t k_row0, int64_t v_row0,
                          int64_t stride, float scale, float *out, cudaStream_t s) {
    const int split = attend_split(c, n_queries, T);
    AttendArgs a;
    a.nu = nu;
    a.codes = codes;
    a.q = q;
    a.out = out;
    a.C = c->k == c->d ? c->Crot : c->C;
    a.Pi = c->Pi;
    a.T = T;
    a.k_row0 = k_row0;
    a.v_row0 = v_row0;
    a.stride = stride;
    a.q_per_group = q_per_group;
    a.scale = scale;
    a.N = c->N;
    a.B = c->B;
    a.R = c->R;
    a.split = split;
    a.buf_words = buf_words(c->R);
    const void *fn = select_kernel(c->d, c->k, c->attend_lut);
    if (!fn) return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_queries * split));
    cfg.blockDim = dim3(32 * c->attend_nwarps);
    cfg.dynamicSmemBytes = c->attend_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace fq
