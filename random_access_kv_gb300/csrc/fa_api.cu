// C ABI of the iterated-map archive (include/fractal.h): argument checks, context set-up (the vertex
// table in double precision on the host), kernel dispatch. The kernels are in fa_archive.cu.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <new>
#include <vector>

#include "fa_internal.h"

namespace {

using fa::kMaxSegment;
using fa::kThreads;
constexpr int kMaxN = 4096;
constexpr double kMinMargin = 2e-5;     // the fp32 cell search needs this much room

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) {
            err = cudaSetDevice(dev);
            changed = err == cudaSuccess;
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

double cell_margin(int N, double r) { return (1.0 - r) * sin(M_PI / N) - r; }

void free_ctx(fa_ctx *c) {
    if (!c) return;
    cudaFree(c->V);
    cudaFree(c->Cf);
    cudaFree(c->flags);
    delete c;
}

}  // namespace

extern "C" {

double fa_ratio_limit(int N) {
    if (N < 2) return 0.0;
    const double s = sin(M_PI / N);
    return s / (1.0 + s);
}

int fa_max_segment(int N, double r) {
    if (N < 2 || !(r > 0.0) || !(r < fa_ratio_limit(N))) return 0;
    const double u = ldexp(1.0, -53);
    const double half_margin = 0.5 * cell_margin(N, r);
    const double delta = 1.01 * u * (1.0 + 4.0 * r);     // forward step, per coordinate
    const double eta = 8.0 * u;                           // backward step, per coordinate
    // error bound of the rebuilt point after j backward steps: sqrt(2) (delta + r eta) r^-j / (1 - r)
    double err = sqrt(2.0) * (delta + r * eta) / (1.0 - r);
    if (!(err <= half_margin)) return 0;
    int L = 1;                                            // decisions j = 0 .. L-1 all fit
    while (L < kMaxSegment && err / r <= half_margin) {
        err /= r;
        ++L;
    }
    return L;
}

int fa_create(fa_ctx **out, int N, double r, int L, int device) {
    if (!out) return FQ_EINVAL;
    *out = nullptr;
    if (N < 2 || N > kMaxN || !isfinite(r) || !(r > 0.0) || !(r < fa_ratio_limit(N))) return FQ_EINVAL;
    if (cell_margin(N, r) < kMinMargin || L < 1 || L > fa_max_segment(N, r)) return FQ_EINVAL;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return FQ_ENODEV;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return FQ_ENODEV;
    if (prop.major != 10 || prop.minor != 3) return FQ_ENODEV;
    DeviceGuard g(device);
    if (g.err != cudaSuccess) return FQ_ECUDA;

    fa_ctx *c = new (std::nothrow) fa_ctx();
    if (!c) return FQ_ENOMEM;
    c->device = device;
    c->num_sms = prop.multiProcessorCount;
    c->N = N;
    c->L = L;
    c->r = r;
    c->rinv = 1.0 / r;
    c->scaleN = (float)(N / (2.0 * M_PI));
    const double lim = r + 0.75 * cell_margin(N, r);
    c->lim2 = (float)(lim * lim);
    // Host tables in std::vector: an allocation failure there must not cross the C ABI.
    std::vector<double2> V;
    std::vector<float2> Cf;
    try {
        V.resize(N);
        Cf.resize(N);
    } catch (...) {
        free_ctx(c);
        return FQ_ENOMEM;
    }
    for (int k = 0; k < N; ++k) {
        const double a = 2.0 * M_PI * k / N;
        V[k] = make_double2(cos(a), sin(a));
        Cf[k] = make_float2((float)((1.0 - r) * V[k].x), (float)((1.0 - r) * V[k].y));
    }
    cudaError_t e = cudaMalloc((void **)&c->V, sizeof(double2) * N);
    if (e == cudaSuccess) e = cudaMalloc((void **)&c->Cf, sizeof(float2) * N);
    if (e == cudaSuccess) e = cudaMalloc((void **)&c->flags, 2 * sizeof(uint32_t));   // sticky word, taken copy
    if (e != cudaSuccess) {
        free_ctx(c);
        return e == cudaErrorMemoryAllocation ? FQ_ENOMEM : FQ_ECUDA;
    }
    e = cudaMemcpy(c->V, V.data(), sizeof(double2) * N, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(c->Cf, Cf.data(), sizeof(float2) * N, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(c->flags, 0, 2 * sizeof(uint32_t));
    if (e != cudaSuccess) {
        free_ctx(c);
        return FQ_ECUDA;
    }
    *out = c;
    return FQ_OK;
}

int fa_params(const fa_ctx *ctx, int *N, double *r, int *L) {
    if (!ctx) return FQ_EINVAL;
    if (N) *N = ctx->N;
    if (r) *r = ctx->r;
    if (L) *L = ctx->L;
    return FQ_OK;
}

int fa_vertex_table(const fa_ctx *ctx, double *V_host) {
    if (!ctx || !V_host) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    return cudaMemcpy(V_host, ctx->V, sizeof(double2) * ctx->N, cudaMemcpyDeviceToHost) == cudaSuccess ? FQ_OK
                                                                                                         : FQ_ECUDA;
}

int64_t fa_segments(const fa_ctx *ctx, int64_t T_cap) {
    if (!ctx || T_cap < 1 || T_cap > INT64_MAX - kMaxSegment) return -1;
    return (T_cap + ctx->L - 1) / ctx->L;
}

int fa_encode(fa_ctx *ctx, const uint16_t *sym, int64_t n_streams, int64_t n_new, int64_t T_cap, int64_t T_old,
              double *anchors, void *stream) {
    if (!ctx || n_streams < 0 || n_new < 0 || T_cap < 1 || T_old < 0 || T_old > T_cap - n_new) return FQ_EINVAL;
    if (n_streams == 0 || n_new == 0) return FQ_OK;
    if (!sym || !anchors) return FQ_EINVAL;
    if (!aligned(sym, 2) || !aligned(anchors, 16)) return FQ_EALIGN;
    const int64_t S_cap = fa_segments(ctx, T_cap);
    if (S_cap < 1) return FQ_EINVAL;
    const int64_t s0 = T_old / ctx->L, n_seg = (T_old + n_new - 1) / ctx->L - s0 + 1;
    if (n_streams > INT64_MAX / S_cap || n_streams > INT64_MAX / n_new) return FQ_EINVAL;
    const int64_t threads = n_streams * n_seg;
    if ((threads + kThreads - 1) / kThreads > INT32_MAX) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    return fa::launch_encode(ctx, sym, n_streams, n_new, S_cap, T_old, s0, n_seg, anchors, (cudaStream_t)stream) ==
                   cudaSuccess
               ? FQ_OK
               : FQ_ECUDA;
}

int fa_decode(fa_ctx *ctx, const double *anchors, int64_t n_streams, int64_t T_cap, int64_t T, uint16_t *out,
              void *stream) {
    if (!ctx || n_streams < 0 || T_cap < 1 || T < 0 || T > T_cap) return FQ_EINVAL;
    if (n_streams == 0 || T == 0) return FQ_OK;
    if (!anchors || !out) return FQ_EINVAL;
    if (!aligned(anchors, 16) || !aligned(out, 2)) return FQ_EALIGN;
    const int64_t S_cap = fa_segments(ctx, T_cap), S = (T + ctx->L - 1) / ctx->L;
    if (S_cap < 1) return FQ_EINVAL;
    if (n_streams > INT64_MAX / S_cap || n_streams > INT64_MAX / T) return FQ_EINVAL;
    const int64_t threads = n_streams * S;
    if ((threads + kThreads - 1) / kThreads > INT32_MAX) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    return fa::launch_decode(ctx, anchors, n_streams, S_cap, T, S, out, (cudaStream_t)stream) == cudaSuccess
               ? FQ_OK
               : FQ_ECUDA;
}

int fa_access(fa_ctx *ctx, const double *anchors, int64_t n_streams, int64_t T_cap, int64_t T, const int64_t *pos,
              int64_t n, uint16_t *out, void *stream) {
    if (!ctx || n_streams < 0 || T_cap < 1 || T < 0 || T > T_cap || n < 0) return FQ_EINVAL;
    if (n == 0) return FQ_OK;
    if (!pos || !out || (!anchors && n_streams > 0 && T > 0)) return FQ_EINVAL;
    if (!aligned(anchors, 16) || !aligned(pos, 8) || !aligned(out, 2)) return FQ_EALIGN;
    const int64_t S_cap = fa_segments(ctx, T_cap);
    if (S_cap < 1) return FQ_EINVAL;
    if (n_streams > INT64_MAX / T_cap || n_streams > INT64_MAX / S_cap) return FQ_EINVAL;
    if ((n + kThreads - 1) / kThreads > INT32_MAX) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    return fa::launch_access(ctx, anchors, n_streams, T_cap, S_cap, T, pos, n, out, (cudaStream_t)stream) ==
                   cudaSuccess
               ? FQ_OK
               : FQ_ECUDA;
}

int fa_status(fa_ctx *ctx, void *stream, uint32_t *flags) {
    if (!ctx || !flags) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t h = 0;
    // One atomic read-and-clear on the device (see fq_status).
    cudaError_t e = fq::launch_take_flags(ctx->flags, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, ctx->flags + 1, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return FQ_ECUDA;
    *flags = h;
    return FQ_OK;
}

void fa_destroy(fa_ctx *ctx) {
    if (!ctx) return;
    DeviceGuard g(ctx->device);
    cudaDeviceSynchronize();
    free_ctx(ctx);
}

}  // extern "C"
