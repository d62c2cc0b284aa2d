// sched.cu -- tile counters for the persistent kernels' dynamic scheduling.
//
// A persistent grid whose CTAs take tiles in a fixed round-robin order ends
// when its slowest CTA does; on GB300 the CTAs of one launch finish up to
// ~25 % apart (measured with a per-CTA timeline), so the kernels instead take
// each next tile from a counter (one atomicAdd per tile).  Every launch needs
// a counter pair that starts at zero: [0] the next tile, [1] CTAs finished.
// The last CTA of a launch to finish puts both back to zero, so a pair is
// ready again for the next launch on the same stream without any host work.
//
// The pairs live in a fixed device array (no allocation).  Each CUDA stream
// gets its own pair on first use, so launches on different streams, which
// may overlap, never share one.  A launch recorded into a CUDA graph gets a
// pair of its own, kept for the life of the process: a graph may be replayed
// on any stream, alongside direct launches, but the launches of one
// instantiated graph are ordered behind each other, so that launch never
// runs twice at once -- as long as the graph is not instantiated twice with
// both instances running at the same time, the one case that needs the
// round-robin order (nts_debug_set_schedule(0)) around its capture.  The
// round-robin order (a null pointer) is also kept for the per-thread
// default stream (one handle for every host thread's stream) and once the
// pool is used up.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "nts_internal.h"

namespace nts {

namespace {

constexpr int kSchedSlots = 1 << 16;   // 512 KB of device memory

__device__ __align__(256) unsigned int g_sched_pool[kSchedSlots][2];

}  // namespace

unsigned int* sched_counters(cudaStream_t stream) {
  if (stream == cudaStreamPerThread) return nullptr;
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capturing) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (capturing == cudaStreamCaptureStatusInvalidated) return nullptr;
  static std::mutex mu;
  static std::map<int, unsigned int*> base;                  // device -> pool address
  static std::map<std::pair<int, cudaStream_t>, int> slot;   // (device, stream) -> pair
  static std::map<int, int> used;                            // device -> pairs handed out
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  auto b = base.find(dev);
  if (b == base.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sched_pool) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    b = base.emplace(dev, static_cast<unsigned int*>(p)).first;
  }
  int& n = used[dev];
  if (capturing == cudaStreamCaptureStatusActive) {
    // a recorded launch: a pair for it alone
    if (n >= kSchedSlots) return nullptr;
    return b->second + 2 * n++;
  }
  const auto key = std::make_pair(dev, stream);
  auto it = slot.find(key);
  if (it == slot.end()) {
    if (n >= kSchedSlots) return nullptr;
    it = slot.emplace(key, n++).first;
  }
  return b->second + 2 * it->second;
}

}  // namespace nts
