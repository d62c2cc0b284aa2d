// mx_launch.cu -- launch-shape selection and launch of the fused
// normalization + MX cast kernels (mx_kernel.cuh).
#include <cuda_runtime.h>

#include <algorithm>

#include "mx_kernel.cuh"
#include "nts_debug.h"

namespace nts {

namespace {

struct MxShape {
  int bpt = 0;  // units (blocks, or halves of 64-value blocks) per consumer thread
  int G = 0;    // consumer threads per row
};

// Threads for a row of K blocks, bpt each: 16 (half a warp, two rows per
// warp) when that covers it, else whole warps.
int threads_for(int K, int bpt) {
  const int n = (K + bpt - 1) / bpt;
  return n <= 16 ? 16 : (n + 31) / 32 * 32;
}

// Threads per row: the fewest (16, or whole warps) that cover the row's K
// units of VB vectors with at most 16 vectors per thread (8 blocks of 16
// values, 4 of 32, 4 halves of 64-value blocks); then units per thread: the
// fewest that still cover the row with those threads, so the units spread
// over all of them.  Measured on GB300 over
// D = 1024..16384 and B = 16..64: more than 16 vectors per thread, or more
// warps per row than needed, cost up to 40 %; at D = 5120 this picks 3
// blocks of 32 on 64 threads (6690 GB/s, against 6470 for 4 blocks and
// 6390 for 5 blocks on 32 threads).
MxShape choose_mx_shape(int K, int VB, int force_bpt) {
  MxShape sh;
  if (force_bpt > 0) {
    sh.bpt = force_bpt;
  } else {
    const int cap = std::max(1, std::min(8, 16 / VB));
    const int G = threads_for(K, cap);
    sh.bpt = std::max(1, std::min(cap, (K + G - 1) / G));
  }
  sh.G = threads_for(K, sh.bpt);
  if (sh.G > kMaxConsumers) sh.G = 0;
  return sh;
}

// The kernel for element format fmt, statistic stat, block size B, bpt
// blocks per thread and a gain or none (nullptr if none is built).
MxKernel pick_mx(int fmt, int stat, int B, int bpt, bool gamma) {
  if (fmt == NTS_FMT_NVFP4) return pick_mx_nvfp4(stat, B, bpt, gamma);
  if (stat < kStatRms || stat > kStatMxP2 || (fmt != NTS_FMT_E4M3 && fmt != NTS_FMT_E2M1))
    return nullptr;
  MxKernel (*const table[2][3])(int, int, bool) = {
      {pick_mx_e4m3_rms, pick_mx_e4m3_p1, pick_mx_e4m3_p2},
      {pick_mx_e2m1_rms, pick_mx_e2m1_p1, pick_mx_e2m1_p2}};
  return table[fmt == NTS_FMT_E2M1 ? 1 : 0][stat](B, bpt, gamma);
}

}  // namespace

// The launch shape of an MX request, without touching the device: units
// per thread, threads per row, rows per tile, ring stages, shared memory
// and the kernel, from the request's sizes, the device's SM count and
// opt-in shared memory per CTA, and the tuning overrides.
struct MxLaunchShape {
  int bpt = 0, G = 0, R = 0, S = 0;
  size_t smem = 0;
  MxKernel kern = nullptr;
};

// CTAs of `threads` threads with `smem` bytes of dynamic shared memory and
// `regs` registers per thread that fit on one SM (0 registers: not limited
// by them): the shared memory of an SM is the opt-in maximum per CTA plus
// the 1 KB each CTA reserves, registers are allocated per warp in units of
// 8 per thread from 64 K, and an SM holds at most 2048 threads.
int mx_ctas_per_sm(int threads, size_t smem, int regs, int max_smem_optin) {
  const size_t kReserved = 1024;
  const size_t smem_sm = (size_t)max_smem_optin + kReserved;
  const int warps = (threads + 31) / 32;
  int n = (int)(smem_sm / (smem + kReserved));
  if (regs > 0) n = std::min(n, 65536 / (((regs + 7) / 8 * 8) * 32 * warps));
  n = std::min(n, 2048 / (warps * 32));
  return std::min(n, 32);
}

int mx_launch_shape(int64_t T, int D, int B, int fmt, int p, bool gamma, int sm_count,
                    int max_smem_optin, int regs, const LaunchTuning& tune,
                    MxLaunchShape* out) {
  const int K = D / B;
  // tune.force_vpt selects the units per thread for this kernel family; a
  // unit is a block, or half a block of 64 values (the kernel splits those
  // between two lanes, each with the 32-value layout)
  const bool split = B == 64;
  const MxShape sh = split ? choose_mx_shape(2 * K, 4, tune.force_vpt)
                           : choose_mx_shape(K, B / 8, tune.force_vpt);
  if (sh.G == 0) return fail(NTS_ERR_UNSUPPORTED, "row too wide: D = %d", D);

  // Rows per tile: about four consumer warps and at least 8 KB per stage;
  // fewer rows when T is small so that the tiles spread over the GPU.
  int R = std::max(1, 128 / sh.G);
  R = std::max(R, (8192 + 2 * D - 1) / (2 * D));
  R = std::min(R, std::max(1, kMaxConsumers / sh.G));
  while (R > 1 && (T + R - 1) / R < (int64_t)2 * sm_count) R /= 2;
  if (sh.G < 32) R = (R + 1) / 2 * 2;   // whole warps: an even number of 16-thread rows
  if (tune.force_rows > 0) R = tune.force_rows;
  if (R * sh.G > kMaxConsumers) return fail(NTS_ERR_UNSUPPORTED, "tile of %d rows too large", R);
  if ((R * sh.G) % 32 != 0)
    return fail(NTS_ERR_UNSUPPORTED, "%d rows of %d threads are not whole warps", R, sh.G);

  // Ring depth: the deepest ring of at most four stages that keeps as many
  // CTAs per SM as two stages allow (registers `regs` per thread, when
  // known).  Measured on GB300 over the MXNorm grid: resident CTAs first,
  // ring depth second -- D = 5120, 16-value E2M1 blocks, two rows of
  // 10 KB per tile: two stages (four CTAs per SM) 126.0 us, three (three
  // CTAs) 140.6 us; D = 1024 with 16 KB stages: three stages 31.1 us, two
  // 32.1 us at the same four CTAs.
  const bool nvfp4 = fmt == NTS_FMT_NVFP4;
  const int nthreads = R * sh.G + 32;
  auto ctas = [&](int s) {
    return mx_ctas_per_sm(nthreads, mx_layout(s, R, D, sh.G, nvfp4).total, regs, max_smem_optin);
  };
  const int most = ctas(2);
  int S = 4;
  while (S > 2 && (ctas(S) < most ||
                   mx_layout(S, R, D, sh.G, nvfp4).total > (uint32_t)tune.smem_budget))
    --S;
  while (S > 1 && mx_layout(S, R, D, sh.G, nvfp4).total > (uint32_t)max_smem_optin) --S;
  if (tune.force_stages > 0) S = tune.force_stages;
  const size_t smem = mx_layout(S, R, D, sh.G, nvfp4).total;
  if (smem > (size_t)max_smem_optin)
    return fail(NTS_ERR_UNSUPPORTED, "row too wide for shared memory: D = %d", D);

  const int stat = p == 0 ? kStatRms : (p == 1 ? kStatMxP1 : kStatMxP2);
  MxKernel kern = pick_mx(fmt, stat, B, sh.bpt, gamma);
  if (kern == nullptr) return fail(NTS_ERR_UNSUPPORTED, "no kernel for B=%d bpt=%d", B, sh.bpt);
  out->bpt = sh.bpt;
  out->G = sh.G;
  out->R = R;
  out->S = S;
  out->smem = smem;
  out->kern = kern;
  return NTS_OK;
}

int launch_mx(const MxRequest& rq, cudaStream_t stream, const LaunchTuning& tune) {
  if (const int injected = take_injected_failure()) return injected;
  const int D = (int)rq.D;
  const int K = D / rq.B;
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");
  // the kernel does not depend on the ring depth or the rows per tile: its
  // register count enters the choice of both
  MxLaunchShape ls;
  int rc = mx_launch_shape(rq.T, D, rq.B, rq.fmt, rq.p, rq.gamma != nullptr, dev.sm_count,
                           dev.max_smem_optin, 0, tune, &ls);
  if (rc != NTS_OK) return rc;
  int regs = 0;
  rc = kernel_registers((const void*)ls.kern, &regs);
  if (rc != NTS_OK) return rc;
  rc = mx_launch_shape(rq.T, D, rq.B, rq.fmt, rq.p, rq.gamma != nullptr, dev.sm_count,
                       dev.max_smem_optin, regs, tune, &ls);
  if (rc != NTS_OK) return rc;
  const MxShape sh{ls.bpt, ls.G};
  const int R = ls.R, S = ls.S;
  const size_t smem = ls.smem;
  MxKernel kern = ls.kern;

  MxParams prm;
  prm.X = static_cast<const __nv_bfloat16*>(rq.X);
  prm.gamma = rq.gamma;
  prm.codes = rq.codes;
  prm.scales = rq.scales;
  prm.rinv_out = rq.rinv;
  prm.amax_out = rq.amax;
  prm.T = rq.T;
  prm.ntiles = (rq.T + R - 1) / R;
  prm.D = D;
  prm.K = K;
  prm.G = sh.G;
  prm.R = R;
  prm.S = S;
  prm.eps = rq.eps;
  prm.corr = 0.f;
  if (rq.p == 1) prm.corr = (float)rq.corr;
  if (rq.p == 2) prm.corr = (float)(rq.corr * rq.corr);
  prm.post = rq.post;
  // every codes row starts 32-byte aligned when the base does and a row is
  // a whole number of 32-byte pieces
  const size_t crow_bytes = rq.fmt == NTS_FMT_E4M3 ? (size_t)D : (size_t)D / 2;
  prm.wide = (reinterpret_cast<uintptr_t>(rq.codes) % 32 == 0 && crow_bytes % 32 == 0) ? 1 : 0;
  prm.wait_limit_ns = tune.wait_limit_ns;
  prm.missing_tx = tune.missing_tx;
  prm.sched = tune.dynamic ? sched_counters(stream) : nullptr;

  rc = prepare_kernel((const void*)kern, smem);
  if (rc != NTS_OK) return rc;

  const int nthreads = R * sh.G + 32;  // consumers + producer warp
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nthreads, smem);
  if (e != cudaSuccess) return fail_cuda(e, "occupancy query for the MX kernel");
  if (per_sm < 1) return fail(NTS_ERR_UNSUPPORTED, "MX kernel does not fit on an SM");
  int64_t grid = std::min<int64_t>(prm.ntiles, (int64_t)per_sm * dev.sm_count);
  if (tune.force_grid > 0) grid = std::min<int64_t>(prm.ntiles, tune.force_grid);

  log_launch(rq.p == 0 ? "rmsnorm_mxcast" : (rq.post ? "mxnorm_postround_cast" : "mxnorm_cast"),
             "T=%lld D=%d B=%d fmt=%d p=%d bpt=%d G=%d R=%d S=%d smem=%zu grid=%lld (%d/SM)",
             (long long)rq.T, D, rq.B, rq.fmt, rq.p, sh.bpt, sh.G, R, S, smem, (long long)grid,
             per_sm);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = tune.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return fail_cuda(e, "launching the MX kernel");
  return NTS_OK;
}

int read_and_clear_mx_status(unsigned* out) {
  int (*const readers[])(unsigned*) = {
      read_and_clear_mx_e4m3_rms_status, read_and_clear_mx_e4m3_p1_status,
      read_and_clear_mx_e4m3_p2_status,  read_and_clear_mx_e2m1_rms_status,
      read_and_clear_mx_e2m1_p1_status,  read_and_clear_mx_e2m1_p2_status,
      read_and_clear_mx_nvfp4_status};
  unsigned all = 0;
  for (auto read : readers) {
    unsigned v = 0;
    const int rc = read(&v);
    if (rc != NTS_OK) return rc;
    all |= v;
  }
  *out = all;
  return NTS_OK;
}

}  // namespace nts

extern "C" int nts_debug_mx_launch_shape(int64_t T, int64_t D, int B, int fmt, int p,
                                         int sm_count, int max_smem_optin, int regs,
                                         int32_t* shape) {
  using namespace nts;
  if (shape == nullptr || T < 0 || D <= 0 || D > (1 << 30) || sm_count <= 0 ||
      max_smem_optin <= 0 || regs < 0 || regs > 255 || (B != 16 && B != 32 && B != 64) ||
      D % B != 0 || p < 0 || p > 2 ||
      (fmt != NTS_FMT_E4M3 && fmt != NTS_FMT_E2M1 && fmt != NTS_FMT_NVFP4) ||
      (fmt == NTS_FMT_NVFP4 && B != 16))
    return fail(NTS_ERR_INVALID_ARG, "bad shape query");
  MxLaunchShape ls;
  const int rc = mx_launch_shape(T, (int)D, B, fmt, p, false, sm_count, max_smem_optin, regs,
                                 current_tuning(), &ls);
  if (rc != NTS_OK) return rc;
  shape[0] = ls.bpt;
  shape[1] = ls.G;
  shape[2] = ls.R;
  shape[3] = ls.S;
  shape[4] = (int32_t)ls.smem;
  return NTS_OK;
}
