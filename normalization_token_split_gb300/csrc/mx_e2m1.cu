// mx_e2m1.cu -- instantiates the fused normalization + MX cast kernels
// (mx_kernel.cuh) for E2M1 elements; a unit of its own so that the
// two element formats compile in parallel.
#include "mx_kernel.cuh"

namespace nts {

MxKernel pick_mx_e2m1(int stat, int B, int bpt) { return pick_mx_format<NTS_FMT_E2M1>(stat, B, bpt); }

int read_and_clear_mx_e2m1_status(unsigned* out) { return read_and_clear_local_mx_status(out); }

}  // namespace nts
