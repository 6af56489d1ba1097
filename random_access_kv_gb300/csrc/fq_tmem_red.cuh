// Tensor-memory loads with a per-lane reduction (tcgen05.ld.red, sm_103a): besides the loaded
// columns, the instruction returns the minimum over them for each lane (TMEM row), so a score
// tile folds to one value per 16 columns without a tree of minima on the CUDA cores.
// Written from the PTX ISA's description of tcgen05.ld; checked on the device (each lane's
// result equals the minimum of the columns it loaded, ties and negative values included).
#pragma once

#include <stdint.h>

namespace fq {
namespace sm100 {

// Minimum over 16 consecutive fp32 columns of this warp's 32 TMEM lanes, starting at taddr.
// Like tcgen05.ld, the result is valid only after tcgen05.wait::ld. The 16 loaded values are
// returned too (in v); they are written asynchronously as well, so v must stay unused (and its
// registers untouched) until the wait: `keep16` after the wait marks them as read there.
__device__ __forceinline__ float tmem_ldred16_min(uint32_t taddr, uint32_t (&v)[16]) {
    float m;
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x16.min.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15}, %16, [%17];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=f"(m)
        : "r"(taddr)
        : "memory");
    return m;
}

// Minimum over 8 consecutive fp32 columns (as tmem_ldred16_min).
__device__ __forceinline__ float tmem_ldred8_min(uint32_t taddr, uint32_t (&v)[8]) {
    float m;
    asm volatile("tcgen05.ld.red.sync.aligned.32x32b.x8.min.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, %8, [%9];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=f"(m)
                 : "r"(taddr)
                 : "memory");
    return m;
}

__device__ __forceinline__ void keep8(const uint32_t (&v)[8]) {
    asm volatile("" ::"r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
}

// Marks 16 registers as read here (no instruction): keeps a load's destination registers
// reserved until after tcgen05.wait::ld.
__device__ __forceinline__ void keep16(const uint32_t (&v)[16]) {
    asm volatile("" ::"r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                 "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}

}  // namespace sm100
}  // namespace fq
