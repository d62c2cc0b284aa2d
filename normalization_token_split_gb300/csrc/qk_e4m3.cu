// qk_e4m3.cu -- instantiates the split-H QK-RMSNorm kernels (qk_kernel.cuh)
// for FP8-E4M3 activations; a unit of its own so the input types compile
// in parallel.
#include "qk_kernel.cuh"

namespace nts {

QkKernel pick_qk_e4m3(int N, int vpt, int G, int bv, int nt) {
  return pick_qk_input<kInE4M3, kQkRms>(N, vpt, G, bv, nt);
}

int read_and_clear_qk_e4m3_status(unsigned* out) { return read_and_clear_local_qk_status(out); }

}  // namespace nts
