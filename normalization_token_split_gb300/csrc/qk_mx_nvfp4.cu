// qk_mx_nvfp4.cu -- instantiates the split-H QK-RMSNorm kernels
// (qk_kernel.cuh) with the block-cast epilogue: the normalized rows leave as
// NVFP4: E2M1 codes in 16-value blocks with E4M3 scales.
#include "qk_kernel.cuh"

namespace nts {

QkKernel pick_qk_mx_nvfp4(int N, int vpt, int G, int bv, int nt) {
  return pick_qk_input<kInBf16, kQkRms, kOutNvfp4>(N, vpt, G, bv, nt);
}

int read_and_clear_qk_mx_nvfp4_status(unsigned* out) { return read_and_clear_local_qk_status(out); }

}  // namespace nts
