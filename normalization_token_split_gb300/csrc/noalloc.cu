// noalloc.cu -- nts_mxnorm_cast_host_noalloc: the host-buffer MXNorm entry
// point with its device staging in a fixed array of the library instead of
// caller-allocated device buffers.
//
// Who needs it: callers that cannot allocate device memory when they call:
// processes whose device memory another framework's pool has already
// reserved (a cudaMalloc of staging buffers would fail), latency-bound loops
// that must not call the allocator after start-up (cudaFree synchronizes the
// device, cudaMalloc may), and host-only callers with no device allocator of
// their own.
//
// The staging lives in one file-scope array per device.  Every call on a
// device shares it, so calls that overlap in time (different streams, or
// host threads without ordering between their calls) race and corrupt each
// other's data: serialize them.  No part of the array has to start at zero:
// each call copies in everything the kernel reads before the kernel runs.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "nts.h"
#include "nts_internal.h"

namespace nts {

namespace {

// Modest, fixed capacity: X (2 B per element), gamma, codes and scales of
// one call, each section 256-byte aligned; e.g. 1024 tokens x 4096 values of
// MXFP8 take 12.6 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_addr_mu;
void* g_addr[kMaxDevices];  // the array's device address, once per device

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// The array's address on the current device: looked up once per device
// (with that device current) and kept.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "querying the current device");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(NTS_ERR_UNSUPPORTED, "device %d beyond the %d the static scratch serves", dev,
                kMaxDevices);
  std::lock_guard<std::mutex> lk(g_addr_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "locating the static scratch");
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return NTS_OK;
}

}  // namespace

}  // namespace nts

using namespace nts;

extern "C" {

int nts_mxnorm_cast_host_noalloc(const void* X_host, const float* gamma_host,
                                 uint8_t* codes_host, uint8_t* scales_host, int64_t T, int64_t D,
                                 float eps, int B, int fmt, int p, void* stream) {
  // Every argument is checked before anything is enqueued or the array is
  // touched.  First the scalars (this bounds D by 32768)...
  int rc = validate_mx_scalars(T, D, eps, B, fmt, p, true);
  if (rc != NTS_OK) return rc;
  if (T > 0 && (X_host == nullptr || codes_host == nullptr || scales_host == nullptr))
    return fail(NTS_ERR_INVALID_ARG, "X_host, codes_host and scales_host must be non-NULL");
  // ... then the capacity: X alone takes 2*T*D bytes, so a T above
  // capacity / (2*D) is refused before any product of T is formed (no
  // product below can then wrap around).
  const size_t xrow = (size_t)D * 2;
  if ((uint64_t)T > kNoAllocScratchBytes / xrow)
    return fail(NTS_ERR_UNSUPPORTED,
                "T=%lld, D=%lld: X alone exceeds the %zu-byte static scratch "
                "(use nts_mxnorm_cast_host with caller-owned buffers)",
                (long long)T, (long long)D, kNoAllocScratchBytes);
  const size_t xb = round256((size_t)T * xrow);
  const size_t gb = gamma_host != nullptr ? round256((size_t)D * 4) : 0;
  const size_t cb = round256((size_t)T * (size_t)(fmt == NTS_FMT_E4M3 ? D : D / 2));
  const size_t sb = round256((size_t)T * (size_t)(D / B));
  const size_t need = xb + gb + cb + sb;
  if (need > kNoAllocScratchBytes)
    return fail(NTS_ERR_UNSUPPORTED,
                "T=%lld, D=%lld needs %zu bytes of device scratch; the static scratch holds %zu "
                "(use nts_mxnorm_cast_host with caller-owned buffers)",
                (long long)T, (long long)D, need, kNoAllocScratchBytes);
  if (T == 0) return NTS_OK;

  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc != NTS_OK) return rc;
  unsigned char* at = static_cast<unsigned char*>(base);
  void* X_dev = at;
  float* gamma_dev = gamma_host != nullptr ? reinterpret_cast<float*>(at + xb) : nullptr;
  uint8_t* codes_dev = at + xb + gb;
  uint8_t* scales_dev = at + xb + gb + cb;

  if (gamma_host != nullptr) {
    const cudaError_t e = cudaMemcpyAsync(gamma_dev, gamma_host, (size_t)D * 4,
                                          cudaMemcpyHostToDevice,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "copying gamma to the device");
  }
  // copy in, kernel and copy back, all on the caller's stream
  return mxnorm_cast_host_one_stream(X_host, gamma_dev, codes_host, scales_host, X_dev, codes_dev,
                                     scales_dev, T, D, eps, B, fmt, p, stream);
}

}  // extern "C"
