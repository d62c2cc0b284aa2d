// mx_nvfp4.cu -- instantiates the fused normalization + block cast kernels
// (mx_kernel.cuh) for NVFP4: E2M1 elements in 16-value blocks with E4M3
// scales.  Only B = 16 exists for this format.
#include "mx_kernel.cuh"

namespace nts {

MxKernel pick_mx_nvfp4(int stat, int B, int bpt, bool gamma) {
  if (B != 16) return nullptr;
  switch (stat) {
    case kStatRms: return pick_mx_bpt<NTS_FMT_NVFP4, kStatRms, 2>(bpt, gamma);
    case kStatMxP1: return pick_mx_bpt<NTS_FMT_NVFP4, kStatMxP1, 2>(bpt, gamma);
    case kStatMxP2: return pick_mx_bpt<NTS_FMT_NVFP4, kStatMxP2, 2>(bpt, gamma);
    default: return nullptr;
  }
}

int read_and_clear_mx_nvfp4_status(unsigned* out) { return read_and_clear_local_mx_status(out); }

}  // namespace nts
