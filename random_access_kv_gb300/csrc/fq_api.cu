// C ABI of libfq.so: argument validation, context set-up (derived tables built on the host in
// double precision), kernel dispatch. Declarations and contracts are in include/fq.h.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "fq_internal.h"

namespace {

// Restores the calling thread's current device on scope exit.
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

int log2_exact(int N) {
    if (N < 2 || (N & (N - 1))) return -1;
    int b = 0;
    while ((1 << b) < N) ++b;
    return b;
}

void free_ctx(fq_ctx *c) {
    if (!c) return;
    cudaFree(c->C);
    cudaFree(c->cc);
    cudaFree(c->Pi);
    cudaFree(c->Crot);
    cudaFree(c->flags);
    cudaFree(c->pi_split);
    cudaFree(c->grid2);
    cudaFree(c->pit_split);
    cudaFree(c->cb_split);
    cudaFree(c->cb_lanes);
    cudaFree(c->crot_split);
    cudaFree(c->cb_ops);
    cudaFree(c->k4_cells);
    cudaFree(c->k4_pool);
    cudaFree(c->k4_axis);
    cudaFree(c->k4_ncb);
    free(c);
}

// FQ_TEST_FAIL_ALLOC set in the environment: device allocations of fq_codebook_load fail, to test
// the out-of-memory path (the context is released and FQ_ENOMEM returned).
bool fail_alloc() { return getenv("FQ_TEST_FAIL_ALLOC") != nullptr; }

template <typename T>
cudaError_t upload(T **dst, const std::vector<T> &src) {
    if (fail_alloc()) return cudaErrorMemoryAllocation;
    cudaError_t e = cudaMalloc((void **)dst, src.size() * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
}

bool is_full(const fq_ctx *c) { return c->k == c->d; }

// Derived tables of a context, built on the host in double precision and copied to the device;
// the kernels' function attributes and launch plans.
cudaError_t build_tables(fq_ctx *c, const float *C_host, const float *Pi_host) {
    const int N = c->N, k = c->k, d = c->d;
    std::vector<float> C(C_host, C_host + (size_t)N * k);
    std::vector<float> P(Pi_host, Pi_host + (size_t)d * d);
    std::vector<float> cc(N);
    for (int n = 0; n < N; ++n) {
        double s = 0;
        for (int t = 0; t < k; ++t) s += (double)C[(size_t)n * k + t] * C[(size_t)n * k + t];
        cc[n] = (float)s;
    }
    cudaError_t e = upload(&c->C, C);
    if (e == cudaSuccess) e = upload(&c->cc, cc);
    if (e == cudaSuccess) e = upload(&c->Pi, P);
    if (e == cudaSuccess && is_full(c)) {
        // Crot[n][i] = sum_j C[n][j] Pi[j][i]  (row n = Pi^T c_n), accumulated in double.
        std::vector<float> R((size_t)N * d);
        std::vector<double> acc(d);
        for (int n = 0; n < N; ++n) {
            for (int i = 0; i < d; ++i) acc[i] = 0.0;
            for (int j = 0; j < d; ++j) {
                const double cj = C[(size_t)n * d + j];
                const float *prow = &P[(size_t)j * d];
                for (int i = 0; i < d; ++i) acc[i] += cj * (double)prow[i];
            }
            for (int i = 0; i < d; ++i) R[(size_t)n * d + i] = (float)acc[i];
        }
        e = upload(&c->Crot, R);
    }
    // flags[0]: the sticky word the kernels set; flags[1]: where fq_status takes it to.
    if (e == cudaSuccess) e = cudaMalloc((void **)&c->flags, 2 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(c->flags, 0, 2 * sizeof(uint32_t));
    if (e == cudaSuccess) e = is_full(c) ? fq::prepare_full(c) : fq::prepare_encode_blocks(c);
    if (e == cudaSuccess && !is_full(c)) e = fq::prepare_decode_blocks(c);
    if (e == cudaSuccess && fq::k2_tc_supported(c)) e = fq::prepare_k2_tc(c);
    if (e == cudaSuccess && !is_full(c) && fq::decode_tc_supported(c)) e = fq::prepare_decode_tc(c);
    if (e == cudaSuccess && is_full(c) && fq::full_tc_supported(c)) e = fq::prepare_full_tc(c);
    if (e == cudaSuccess && fq::k4_grid_supported(c)) e = fq::prepare_k4_grid(c);
    if (e == cudaSuccess && !is_full(c) && !c->grid2 && !c->k4_cells && fq::kq_tc_supported(c)) e = fq::prepare_kq_tc(c);
    if (e == cudaSuccess) e = fq::prepare_attend(c);
    return e;
}

}  // namespace

extern "C" {

const char *fq_strerror(int err) {
    switch (err) {
        case FQ_OK: return "ok";
        case FQ_EINVAL: return "invalid argument";
        case FQ_ENOMEM: return "out of memory";
        case FQ_ECUDA: return "CUDA error";
        case FQ_EALIGN: return "misaligned buffer";
        case FQ_ENODEV: return "no usable sm_103 device";
        default: return "unknown error";
    }
}

int fq_codebook_load(fq_ctx **out, const float *C_host, int N, int k, const float *Pi_host, int d,
                     int device) {
    if (!out) return FQ_EINVAL;
    *out = nullptr;
    if (!C_host || !Pi_host) return FQ_EINVAL;
    const int B = log2_exact(N);
    if (B < 0 || N > 65536) return FQ_EINVAL;
    // Block codes: d = 64 and 128 (all paths), d = 96 (CUDA-core kernels; k = 3 lives here).
    const bool blocks_ok = (d == 64 || d == 96 || d == 128) && (k == 1 || k == 2 || k == 3 || k == 4 || k == 8) &&
                           d % k == 0 && (size_t)N * k <= 32768;
    const bool full_ok = (d == 64 && k == 64 && N >= 64);
    if (!blocks_ok && !full_ok) return FQ_EINVAL;
    for (size_t i = 0; i < (size_t)N * k; ++i)
        if (!isfinite(C_host[i])) return FQ_EINVAL;
    for (size_t i = 0; i < (size_t)d * d; ++i)
        if (!isfinite(Pi_host[i])) return FQ_EINVAL;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return FQ_ENODEV;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return FQ_ENODEV;
    if (prop.major != 10 || prop.minor != 3) return FQ_ENODEV;
    DeviceGuard g(device);
    if (g.err != cudaSuccess) return FQ_ECUDA;

    fq_ctx *c = (fq_ctx *)calloc(1, sizeof(fq_ctx));
    if (!c) return FQ_ENOMEM;
    c->device = device;
    c->d = d;
    c->k = k;
    c->N = N;
    c->B = B;
    c->nb = d / k;
    c->R = c->nb * B;
    c->num_sms = prop.multiProcessorCount;
    c->smem_optin = (int)prop.sharedMemPerBlockOptin;

    // Host tables are built in std::vector: an allocation failure there must not cross the C ABI.
    cudaError_t e;
    try {
        e = build_tables(c, C_host, Pi_host);
    } catch (const std::bad_alloc &) {
        e = cudaErrorMemoryAllocation;
    } catch (...) {
        e = cudaErrorUnknown;
    }
    if (e != cudaSuccess) {
        const int rc = (e == cudaErrorMemoryAllocation) ? FQ_ENOMEM : FQ_ECUDA;
        free_ctx(c);
        return rc;
    }
    *out = c;
    return FQ_OK;
}

int64_t fq_code_words(const fq_ctx *ctx, int64_t M) {
    if (!ctx || M < 0 || M > (INT64_MAX - 31) / ctx->R) return -1;
    return (M * ctx->R + 31) / 32;
}

int fq_record_bits(const fq_ctx *ctx) { return ctx ? ctx->R : -1; }

int fq_shape(const fq_ctx *ctx, int *d, int *k, int *N) {
    if (!ctx) return FQ_EINVAL;
    if (d) *d = ctx->d;
    if (k) *k = ctx->k;
    if (N) *N = ctx->N;
    return FQ_OK;
}

static int encode_common(fq_ctx *ctx, const void *x, int64_t M, fq::RowMap map, int64_t rows_total,
                         float *nu, uint32_t *codes, void *stream) {
    if (!ctx || M < 0 || M > INT32_MAX) return FQ_EINVAL;
    if (M == 0) return FQ_OK;
    if (!x || !nu || !codes) return FQ_EINVAL;
    if (!aligned(x, 16) || !aligned(nu, 4) || !aligned(codes, 4)) return FQ_EALIGN;
    if (rows_total < 0 || fq_code_words(ctx, rows_total) < 0) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (is_full(ctx) && ctx->crot_split)
        e = fq::launch_encode_full_tc(ctx, (const __half *)x, M, map, nu, codes, s);
    else if (is_full(ctx))
        e = fq::launch_encode_full(ctx, (const __half *)x, M, map, nu, codes, s);
    else if (ctx->grid2)
        e = fq::launch_encode_k2_tc(ctx, (const __half *)x, M, map, nu, codes, s);
    else if (ctx->k4_cells)
        e = fq::launch_encode_k4_grid(ctx, (const __half *)x, M, map, nu, codes, s);
    else if (ctx->cb_ops)
        e = fq::launch_encode_kq_tc(ctx, (const __half *)x, M, map, nu, codes, s);
    else
        e = fq::launch_encode_blocks(ctx, (const __half *)x, M, map, nu, codes, s);
    return e == cudaSuccess ? FQ_OK : FQ_ECUDA;
}

int fq_encode(fq_ctx *ctx, const void *x, int64_t M, float *nu, uint32_t *codes, int64_t row0,
              void *stream) {
    if (row0 < 0 || M > INT64_MAX - row0) return FQ_EINVAL;
    fq::RowMap map{M > 0 ? M : 1, 0, row0};
    return encode_common(ctx, x, M, map, row0 + M, nu, codes, stream);
}

int fq_encode_append(fq_ctx *ctx, const void *x, int64_t n_seq, int64_t n_new, int64_t seq_capacity,
                     int64_t t0, float *nu, uint32_t *codes, void *stream) {
    if (n_seq < 0 || n_new < 0 || t0 < 0 || seq_capacity < 0) return FQ_EINVAL;
    if (n_new > seq_capacity || t0 > seq_capacity - n_new) return FQ_EINVAL;
    if (n_seq > 0 && seq_capacity > INT64_MAX / n_seq) return FQ_EINVAL;
    if (n_seq > 0 && n_new > INT64_MAX / n_seq) return FQ_EINVAL;
    const int64_t M = n_seq * n_new;
    fq::RowMap map{n_new > 0 ? n_new : 1, seq_capacity, t0};
    return encode_common(ctx, x, M, map, n_seq * seq_capacity, nu, codes, stream);
}

static int decode_common(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                         const int64_t *idx, int64_t n, void *out, bool out_f32, void *stream) {
    if (!ctx || M < 0 || n < 0 || n > INT32_MAX) return FQ_EINVAL;
    if (n == 0) return FQ_OK;
    if (!out || (!idx && n > M)) return FQ_EINVAL;
    if (M > 0 && (!nu || !codes)) return FQ_EINVAL;
    if (fq_code_words(ctx, M) < 0) return FQ_EINVAL;
    if (!aligned(out, 16) || !aligned(nu, 4) || !aligned(codes, 4) || !aligned(idx, 8)) return FQ_EALIGN;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (is_full(ctx))
        e = fq::launch_decode_full(ctx, nu, codes, M, idx, n, out, out_f32, s);
    else if (ctx->pit_split)
        e = fq::launch_decode_tc(ctx, nu, codes, M, idx, n, out, out_f32, s);
    else
        e = fq::launch_decode_blocks(ctx, nu, codes, M, idx, n, out, out_f32, s);
    return e == cudaSuccess ? FQ_OK : FQ_ECUDA;
}

int fq_decode(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M, void *out, void *stream) {
    return decode_common(ctx, nu, codes, M, nullptr, M, out, false, stream);
}

int fq_decode_gather(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M, const int64_t *idx,
                     int64_t n, void *out, void *stream) {
    if (n > 0 && !idx) return FQ_EINVAL;
    return decode_common(ctx, nu, codes, M, idx, n, out, false, stream);
}

int fq_decode_gather_f32(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M,
                         const int64_t *idx, int64_t n, float *out, void *stream) {
    if (n > 0 && !idx) return FQ_EINVAL;
    return decode_common(ctx, nu, codes, M, idx, n, out, true, stream);
}

int fq_attend(fq_ctx *ctx, const float *nu, const uint32_t *codes, int64_t M, const void *q,
              int64_t n_queries, int64_t q_per_group, int64_t T, int64_t k_row0, int64_t v_row0,
              int64_t stride, float scale, float *out, void *stream) {
    if (!ctx || M < 0 || n_queries < 0 || q_per_group < 1 || T < 1) return FQ_EINVAL;
    if (k_row0 < 0 || v_row0 < 0 || stride < 0 || !isfinite(scale)) return FQ_EINVAL;
    if (n_queries % q_per_group || n_queries > INT32_MAX / 8) return FQ_EINVAL;
    if (n_queries == 0) return FQ_OK;
    if (!nu || !codes || !q || !out) return FQ_EINVAL;
    if (fq_code_words(ctx, M) < 0) return FQ_EINVAL;
    // Every cached row of every group lies in [0, M).
    const int64_t groups = n_queries / q_per_group;
    for (int64_t r0 : {k_row0, v_row0}) {
        if (T > M || r0 > M - T) return FQ_EINVAL;
        if (groups > 1 && stride > (M - T - r0) / (groups - 1)) return FQ_EINVAL;
    }
    if (!aligned(nu, 4) || !aligned(codes, 4) || !aligned(q, 2) || !aligned(out, 4)) return FQ_EALIGN;
    if (!fq::attend_supported(ctx)) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    cudaError_t e = fq::launch_attend(ctx, nu, codes, (const __half *)q, n_queries, q_per_group, T, k_row0,
                                      v_row0, stride, scale, out, (cudaStream_t)stream);
    return e == cudaSuccess ? FQ_OK : FQ_ECUDA;
}

int fq_centroid_sums(fq_ctx *ctx, const void *x, int64_t M, const float *nu, const uint32_t *codes,
                     double *sums, double *counts, void *stream) {
    if (!ctx || M < 0 || M > INT32_MAX) return FQ_EINVAL;
    if (M == 0) return FQ_OK;
    if (!x || !nu || !codes || !sums || !counts) return FQ_EINVAL;
    if (fq_code_words(ctx, M) < 0) return FQ_EINVAL;
    if (!aligned(x, 16) || !aligned(nu, 4) || !aligned(codes, 4) || !aligned(sums, 8) || !aligned(counts, 8))
        return FQ_EALIGN;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    cudaError_t e = fq::launch_centroid_sums(ctx, (const __half *)x, M, nu, codes, sums, counts, (cudaStream_t)stream);
    return e == cudaSuccess ? FQ_OK : FQ_ECUDA;
}

int fq_selftest_wait(fq_ctx *ctx, uint64_t limit_ns, void *stream) {
    if (!ctx || limit_ns > 1000000000ull) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    return fq::launch_wait_selftest(ctx, limit_ns, (cudaStream_t)stream) == cudaSuccess ? FQ_OK : FQ_ECUDA;
}

int fq_status(fq_ctx *ctx, void *stream, uint32_t *flags) {
    if (!ctx || !flags) return FQ_EINVAL;
    DeviceGuard g(ctx->device);
    if (g.err != cudaSuccess) return FQ_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t h = 0;
    // Read and clear in one atomic step on the device, so that a flag another stream's kernel
    // raises meanwhile is kept for the next call rather than cleared unread.
    cudaError_t e = fq::launch_take_flags(ctx->flags, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, ctx->flags + 1, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return FQ_ECUDA;
    *flags = h;
    return FQ_OK;
}

void fq_destroy(fq_ctx *ctx) {
    if (!ctx) return;
    DeviceGuard g(ctx->device);
    cudaDeviceSynchronize();
    free_ctx(ctx);
}

}  // extern "C"
