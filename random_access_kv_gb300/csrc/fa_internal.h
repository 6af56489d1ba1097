// Internal declarations of the iterated-map archive, shared by its kernels (fa_archive.cu) and its
// C ABI (fa_api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fractal.h"

struct fa_ctx {
    int device = 0;
    int N = 0;
    int L = 0;
    double r = 0.0;
    double rinv = 0.0;
    float scaleN = 0.f;     // N / (2 pi): angle to vertex index
    float lim2 = 0.f;       // (r + 3/4 margin)^2: largest squared distance to a cell centre
    int num_sms = 0;
    double2 *V = nullptr;   // [N] vertices
    float2 *Cf = nullptr;   // [N] cell centres (1 - r) V(c), fp32
    uint32_t *flags = nullptr;   // [0] sticky FA_FLAG_* word, [1] the copy fa_status takes
};

namespace fq {
// flags[1] = atomic exchange of flags[0] with 0, by one device thread (defined in fq_selftest.cu).
cudaError_t launch_take_flags(uint32_t *flags, cudaStream_t s);
}  // namespace fq

namespace fa {

constexpr int kThreads = 256;
constexpr int kMaxSegment = 64;       // longest segment fa_max_segment returns

// Kernel launches on stream s; arguments already validated by the caller.
cudaError_t launch_encode(const fa_ctx *c, const uint16_t *sym, int64_t n_streams, int64_t n_new, int64_t S_cap,
                          int64_t T_old, int64_t s0, int64_t n_seg, double *anchors, cudaStream_t s);
cudaError_t launch_decode(const fa_ctx *c, const double *anchors, int64_t n_streams, int64_t S_cap, int64_t T,
                          int64_t S, uint16_t *out, cudaStream_t s);
cudaError_t launch_access(const fa_ctx *c, const double *anchors, int64_t n_streams, int64_t T_cap, int64_t S_cap,
                          int64_t T, const int64_t *pos, int64_t n, uint16_t *out, cudaStream_t s);

}  // namespace fa
