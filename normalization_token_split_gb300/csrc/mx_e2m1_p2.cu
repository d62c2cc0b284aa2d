// mx_e2m1_p2.cu -- instantiates the fused normalization + MX cast kernels
// (mx_kernel.cuh) for E2M1 elements and the MXNorm, p = 2 statistic, every
// block size and blocks-per-thread count; a unit of its own so that the
// kernel families compile in parallel.
#include "mx_kernel.cuh"

namespace nts {

NTS_MX_UNIT(mx_e2m1_p2, NTS_FMT_E2M1, kStatMxP2)

}  // namespace nts
