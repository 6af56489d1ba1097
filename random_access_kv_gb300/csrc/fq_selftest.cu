// Self-test of the failure path of the bounded waits: one CTA waits on an mbarrier that nothing
// completes. The wait must give up after the limit and report FQ_FLAG_TIMEOUT through the
// context's status word; the context stays usable. Nothing traps.
// Also the device half of fq_status / fa_status: the atomic read-and-clear of a status word.
#include "fq_internal.h"
#include "fq_sm100.cuh"

namespace fq {
namespace {

using namespace sm100;

__global__ void wait_selftest(uint32_t *flags, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, limit_ns);   // no arrival: gives up after limit_ns
    if (!ok && threadIdx.x == 0) atomicOr(flags, (uint32_t)FQ_FLAG_TIMEOUT);
}

__global__ void take_flags(uint32_t *flags) { flags[1] = atomicExch(flags, 0u); }

}  // namespace

cudaError_t launch_take_flags(uint32_t *flags, cudaStream_t s) {
    take_flags<<<1, 1, 0, s>>>(flags);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const fq_ctx *ctx, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest<<<1, 32, 0, s>>>(ctx->flags, limit_ns);
    return cudaGetLastError();
}

}  // namespace fq
