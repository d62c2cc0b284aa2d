// qk_mx_e2m1.cu -- instantiates the split-H QK-RMSNorm kernels
// (qk_kernel.cuh) with the block-cast epilogue: the normalized rows leave as
// MX E2M1 codes with E8M0 scales (MXFP4).
#include "qk_kernel.cuh"

namespace nts {

QkKernel pick_qk_mx_e2m1(int N, int vpt, int G, int bv, int nt) {
  return pick_qk_input<kInBf16, kQkRms, kOutE2M1>(N, vpt, G, bv, nt);
}

int read_and_clear_qk_mx_e2m1_status(unsigned* out) { return read_and_clear_local_qk_status(out); }

}  // namespace nts
