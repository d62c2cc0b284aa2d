// qk_mx_e4m3.cu -- instantiates the split-H QK-RMSNorm kernels
// (qk_kernel.cuh) with the block-cast epilogue: the normalized rows leave as
// MX E4M3 codes with E8M0 scales (MXFP8).
#include "qk_kernel.cuh"

namespace nts {

QkKernel pick_qk_mx_e4m3(int N, int vpt, int G, int bv, int nt) {
  return pick_qk_input<kInBf16, kQkRms, kOutE4M3>(N, vpt, G, bv, nt);
}

int read_and_clear_qk_mx_e4m3_status(unsigned* out) { return read_and_clear_local_qk_status(out); }

}  // namespace nts
