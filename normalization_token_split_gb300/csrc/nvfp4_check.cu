// nvfp4_check.cu -- self-checks of the block-scale arithmetic over every
// non-negative fp32 absmax: nts_debug_check_nvfp4_scale compares the NVFP4
// scale of the kernels (division by 6 without a divide instruction, scale
// reciprocals from a table) with the same scale taken through the IEEE
// quotient and the IEEE reciprocal; nts_debug_check_e8m0 compares the E8M0
// exponent (one add and one shift) with its field-by-field definition.
#include <cuda_runtime.h>

#include <cstdint>

#include "nts_debug.h"
#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

namespace {

// [0]: absmaxes whose (code, reciprocal) differ from the IEEE route;
// [1]: absmaxes with a normal quotient where div6_rn differs from it;
// [2]: absmaxes whose E8M0 exponent (emax 8 or 2) differs from the definition.
__device__ unsigned long long g_check_counts[3];

// every pattern 0 .. 0x7F800000 (+0 up to +inf; no NaN)
constexpr uint64_t kPatterns = 0x7F800001ull;

__global__ void __launch_bounds__(256) nvfp4_scale_check_kernel() {
  __shared__ float rcp[128];
  fill_e4m3_reciprocals(rcp, threadIdx.x, blockDim.x);
  __syncthreads();
  unsigned long long bad_code = 0, bad_quot = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < kPatterns; u += stride) {
    const float ay = __uint_as_float((uint32_t)u);
    float inv;
    const uint32_t sc = nvfp4_scale(ay, rcp, &inv);
    const float quot = __fdiv_rn(ay, 6.0f);
    const uint32_t ref = cvt_e4m3x2(quot, 0.f) & 0xFFu;
    const float ref_inv = ref != 0 ? __frcp_rn(f2_lo(e4m3x2_to_f2((uint16_t)ref))) : 0.f;
    if (sc != ref || __float_as_uint(inv) != __float_as_uint(ref_inv)) ++bad_code;
    if (quot >= 0x1p-126f && ay < __uint_as_float(0x7F800000u) &&
        __float_as_uint(div6_rn(ay)) != __float_as_uint(quot))
      ++bad_quot;
  }
  if (bad_code != 0) atomicAdd(&g_check_counts[0], bad_code);
  if (bad_quot != 0) atomicAdd(&g_check_counts[1], bad_quot);
}

__global__ void __launch_bounds__(256) e8m0_check_kernel() {
  unsigned long long bad = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < kPatterns; u += stride) {
    const float ay = __uint_as_float((uint32_t)u);
    if (e8m0_exponent(ay, 8) != e8m0_exponent_by_fields(ay, 8)) ++bad;
    if (e8m0_exponent(ay, 2) != e8m0_exponent_by_fields(ay, 2)) ++bad;
  }
  if (bad != 0) atomicAdd(&g_check_counts[2], bad);
}

// Clears the counters, runs `kern` over every pattern, reads the counters.
int run_check(void (*kern)(), unsigned long long* got) {
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");
  const unsigned long long zero[3] = {0, 0, 0};
  cudaError_t e = cudaMemcpyToSymbol(g_check_counts, zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clearing the check counters");
  kern<<<(unsigned)dev.sm_count * 8, 256>>>();
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "launching a self-check");
  e = cudaMemcpyFromSymbol(got, g_check_counts, 3 * sizeof(unsigned long long));  // waits
  if (e != cudaSuccess) return fail_cuda(e, "reading the check counters");
  return NTS_OK;
}

}  // namespace

}  // namespace nts

using namespace nts;

extern "C" int nts_debug_check_nvfp4_scale(uint64_t* code_mismatches,
                                           uint64_t* quotient_mismatches) {
  if (code_mismatches == nullptr || quotient_mismatches == nullptr)
    return fail(NTS_ERR_INVALID_ARG, "both output pointers must be non-NULL");
  unsigned long long got[3];
  const int rc = run_check(nvfp4_scale_check_kernel, got);
  if (rc != NTS_OK) return rc;
  *code_mismatches = got[0];
  *quotient_mismatches = got[1];
  return NTS_OK;
}

extern "C" int nts_debug_check_e8m0(uint64_t* mismatches) {
  if (mismatches == nullptr) return fail(NTS_ERR_INVALID_ARG, "mismatches must be non-NULL");
  unsigned long long got[3];
  const int rc = run_check(e8m0_check_kernel, got);
  if (rc != NTS_OK) return rc;
  *mismatches = got[2];
  return NTS_OK;
}
