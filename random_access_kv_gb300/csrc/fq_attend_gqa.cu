// Instantiations of the fused attention kernel that serve four queries of one cached group per
// cluster (grouped-query attention); a separate translation unit so that it compiles in parallel.
#include "fq_attend_kernel.cuh"

namespace fq {

const void *attend_kernel_gqa(int d, int k, bool lut) { return attend_detail::select_kernel_q<4>(d, k, lut); }

}  // namespace fq
