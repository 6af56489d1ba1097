// Host side of the fused decode-into-attention: launch plans (how many queries a cluster serves,
// whether the score tables fit, warps per CTA, cluster size) and the launch. The kernel and its
// description are in fq_attend_kernel.cuh.
#include <algorithm>

#include "fq_attend_kernel.cuh"

namespace fq {
namespace {

using attend_detail::kMaxSplit;
using attend_detail::kMaxWarps;
using attend_detail::kMinWarps;

const void *select_kernel(int d, int k, bool lut, int qg) {
    return qg == 1 ? attend_detail::select_kernel_q<1>(d, k, lut) : attend_kernel_gqa(d, k, lut);
}

int buf_words(int R) { return (2 * (R + 2) + 64 + 3) & ~3; }

size_t table_bytes(const fq_ctx *c, bool lut, int qg) {
    const int d = c->d, k = c->k, nb = d / k;
    size_t f = (size_t)qg * (3 * d + 4 + 2 * kMaxWarps + (size_t)kMaxWarps * d);
    if (k != d) f += (size_t)c->N * k;
    if (lut) f += (size_t)qg * c->N * (nb >= 32 ? nb : 32);
    return f * sizeof(float);
}

// One plan: QG queries per cluster (plan 0: 1, plan 1: 4).
cudaError_t make_plan(fq_ctx *c, int pi) {
    const int qg = pi == 0 ? 1 : 4;
    const int max_warps = qg == 1 ? kMaxWarps : 8;
    AttendPlan &P = c->attend[pi];
    P.nwarps = 0;
    const size_t per_warp = 2 * (size_t)buf_words(c->R) * sizeof(uint32_t);
    const size_t limit = (size_t)c->smem_optin;
    const bool lut = c->k != c->d && table_bytes(c, true, qg) + max_warps * per_warp <= limit;
    const size_t tables = table_bytes(c, lut, qg);
    if (tables + kMinWarps * per_warp > limit) return cudaSuccess;   // this plan does not fit
    const int nwarps = (int)std::min<size_t>(max_warps, (limit - tables) / per_warp);
    const size_t smem = tables + nwarps * per_warp;
    const void *fn = select_kernel(c->d, c->k, lut, qg);
    if (!fn) return cudaSuccess;
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
        P.slots[s] = n * s;
        if (n > 0) max_split = s;
    }
    if (!max_split) return cudaSuccess;
    P.qg = qg;
    P.lut = lut;
    P.nwarps = nwarps;
    P.smem = smem;
    P.max_split = max_split;
    return cudaSuccess;
}

// Minimise waves x (tokens per CTA + fixed per-CTA cost in token units).
int choose_split(const fq_ctx *c, const AttendPlan &P, int64_t units, int64_t T) {
    const int64_t n_tiles = (T + 31) / 32;
    const int nb = c->d / c->k;
    const double fixed = 64.0 + (P.lut ? (double)P.qg * c->N * (nb >= 32 ? nb : 32) / nb / 2 : 0.0);
    int best = 1;
    double best_cost = 0;
    for (int s = 1; s <= P.max_split && s <= n_tiles; ++s) {
        const int64_t slots = P.slots[s];
        if (slots <= 0) continue;
        const int64_t ctas = units * s;
        const double waves = (double)((ctas + slots - 1) / slots);
        const double cost = waves * ((double)T / s + fixed);
        if (best_cost == 0 || cost < best_cost * 0.98) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

}  // namespace

cudaError_t prepare_attend(fq_ctx *c) {
    for (int pi = 0; pi < 2; ++pi) {
        cudaError_t e = make_plan(c, pi);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool attend_supported(const fq_ctx *c) { return c->attend[0].nwarps > 0; }

cudaError_t launch_attend(const fq_ctx *c, const float *nu, const uint32_t *codes, const __half *q,
                          int64_t n_queries, int64_t q_per_group, int64_t T, int64_t k_row0, int64_t v_row0,
                          int64_t stride, float scale, float *out, cudaStream_t s) {
    // Queries of one group served together when the group has a multiple of four.
    const bool grouped = q_per_group % 4 == 0 && c->attend[1].nwarps > 0;
    const AttendPlan &P = c->attend[grouped ? 1 : 0];
    const int64_t units = n_queries / P.qg;
    const int split = choose_split(c, P, units, T);
    attend_detail::AttendArgs a;
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
    const void *fn = select_kernel(c->d, c->k, P.lut, P.qg);
    if (!fn) return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * split));
    cfg.blockDim = dim3(32 * P.nwarps);
    cfg.dynamicSmemBytes = P.smem;
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
