// qk_ln.cu -- instantiates the split-H kernels (qk_kernel.cuh) with the
// LayerNorm statistic (sum and sum of squares per shard) for bfloat16
// activations; a unit of its own so it compiles in parallel.
#include "qk_kernel.cuh"

namespace nts {

QkKernel pick_qk_ln(int N, int vpt, int G, int bv, int nt) {
  return pick_qk_input<kInBf16, kQkLn>(N, vpt, G, bv, nt);
}

int read_and_clear_qk_ln_status(unsigned* out) { return read_and_clear_local_qk_status(out); }

}  // namespace nts
