// nts_internal.h -- declarations shared by the library's own translation
// units (host API and kernel launchers).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "nts.h"

namespace nts {

// A CTA has up to 480 consumer threads (the threads that own data) plus one
// producer warp that only issues the TMA copies.  512 threads leave up to
// 128 registers per thread.
constexpr int kMaxConsumers = 480;
constexpr int kMaxThreads = kMaxConsumers + 32;

// Per-call launch settings: automatic unless a debug override is set.
struct LaunchTuning {
  int force_vpt = 0;         // QK: 16-byte vectors per thread; MX: blocks per thread; 0 = auto
  int force_rows = 0;        // rows per tile, 0 = automatic
  int force_stages = 0;      // ring stages, 0 = automatic
  int64_t force_grid = 0;    // CTAs (MX) or clusters (QK), 0 = automatic
  int smem_budget = 102400;  // bytes of shared memory a CTA aims to stay under
  uint64_t wait_limit_ns = 1000000000ull;  // bounded mbarrier waits
  uint32_t missing_tx = 0;   // test hook, see nts_debug.h
  int dynamic = 1;           // take tiles from a counter (0: round-robin order)
  int direct = 1;            // decode-sized QK launches use the single-tile kernel
  int pdl = 1;               // launch with programmatic stream serialization
};

// The launch attribute that lets a grid be scheduled while the grid before
// it in the stream finishes (programmatic dependent launch).  Every kernel
// of the library waits (griddepcontrol.wait) before its first global-memory
// access, so this changes timing only.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// The launch attribute that lets the hardware balance the CTAs of a cluster
// over the SMs of its GPC as it sees fit.  With the default placement, a
// grid of the occupancy query's maximum cluster count, placed while the
// previous grid drains, sometimes left a cluster without room until other
// clusters had finished (per-CTA timelines on GB300: a split-H launch after
// an MX launch started one cluster ~48 us late, in half of the launches);
// with this policy every cluster started at once, and the occupancy query,
// which sees the attribute, admits one or two more clusters.
inline cudaLaunchAttribute cluster_policy_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  a.val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
  return a;
}

LaunchTuning current_tuning();

// Test hook (nts_debug_inject_failure): while injections remain, the next
// launch returns the injected status (with last-error text saying so)
// instead of touching the device; otherwise NTS_OK.
int take_injected_failure();

// The zeroed counter pair of `stream` for a dynamically scheduled launch
// (sched.cu), or nullptr: schedule round-robin.
unsigned int* sched_counters(cudaStream_t stream);

struct DeviceInfo {
  bool ok = false;
  int device = 0;
  int sm_count = 0;
  int max_smem_optin = 0;
};
const DeviceInfo& device_info();

// How the G threads of a row split its nvec 16-byte vectors: thread g owns
// vectors g, g+G, ..., g+(vpt-1)G.  G is a multiple of 32 (whole warps);
// G == 0 means the row is too wide.
struct RowShape {
  int vpt = 0;
  int G = 0;
};
RowShape choose_row_shape(int nvec, int force_vpt);

// Raise the kernel's dynamic shared memory limit (once per kernel/device).
int prepare_kernel(const void* kernel, size_t smem);
// Registers per thread of a kernel (cached per device).
int kernel_registers(const void* kernel, int* regs);
// Co-resident clusters of `cluster` CTAs for this launch configuration.
int max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg, int cluster,
                        int64_t* out);

// Record a failure for nts_last_error() and return `status`.
int fail(int status, const char* fmt, ...);
int fail_cuda(cudaError_t e, const char* what);
void log_launch(const char* name, const char* fmt, ...);

struct MxRequest {
  const void* X;
  const float* gamma;
  uint8_t* codes;
  uint8_t* scales;
  float* rinv;
  float* amax;
  int64_t T;
  int64_t D;
  float eps;
  int B;
  int fmt;
  int p;        // 0 = RMSNorm statistic, 1 or 2 = MXNorm
  double corr;  // c(B, p) for MXNorm
  int post;     // MXNorm from E8M0-rounded absmaxes (post-round)
};

struct QkRequest {
  const void* X;
  const float* gamma;
  void* Y;
  float* rinv;
  int64_t T;
  int64_t H;
  const float* beta = nullptr;  // LayerNorm only (nullable)
  float* mean = nullptr;        // LayerNorm only (nullable)
  uint8_t* codes = nullptr;     // block-cast output (replaces Y)
  uint8_t* scales = nullptr;
};

// What a QK launch reads, computes and writes beyond the common case (bf16
// in, RMSNorm, bf16 out).
struct QkOptions {
  int in_e4m3 = 0;      // activations are E4M3 codes, value = code * x_scale
  float x_scale = 1.f;
  int layernorm = 0;    // LayerNorm statistic (bf16 input only)
  int out_fmt = -1;     // >= 0: block-cast output in this nts_elem_fmt (RMSNorm only)
  int B = 0;            // ... with blocks of B elements
};

// One launch normalizing 1 or 2 tensors (Q and K) with the same N.
int launch_qknorm(const QkRequest* rq, int ntensors, float eps, int N, const QkOptions& opt,
                  cudaStream_t stream, const LaunchTuning& tune);
int launch_mx(const MxRequest& rq, cudaStream_t stream, const LaunchTuning& tune);

// Headwise QK-Norm with every head inside one CTA (heads_kernel.cu): for
// N == 1, head_dim in {8, 16, ..., 256} and H <= 30720.
bool heads_whole_path(int64_t H, int64_t head_dim, int N);
int launch_heads(const void* X, const float* gamma, void* Y, float* rinv, int64_t T, int64_t H,
                 int64_t head_dim, float eps, cudaStream_t stream, const LaunchTuning& tune);
int read_and_clear_heads_status(unsigned* out);

// The checks of an MX call (RMSNorm+MXCast or MXNorm) that involve no
// pointer: T, D, eps, B, fmt and p.
int validate_mx_scalars(int64_t T, int64_t D, float eps, int B, int fmt, int p, bool mxnorm);
// nts_mxnorm_cast_host with its copies and kernel all on `stream`, never
// chunked (so it creates no copy streams or events).
int mxnorm_cast_host_one_stream(const void* X_host, const float* gamma_dev, uint8_t* codes_host,
                                uint8_t* scales_host, void* X_dev, uint8_t* codes_dev,
                                uint8_t* scales_dev, int64_t T, int64_t D, float eps, int B,
                                int fmt, int p, void* stream);

int read_and_clear_qk_status(unsigned* out);
int read_and_clear_mx_status(unsigned* out);

}  // namespace nts
