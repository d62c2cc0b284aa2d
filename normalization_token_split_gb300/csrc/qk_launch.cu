// qk_launch.cu -- launch-shape selection and launch of the split-H
// QK-RMSNorm and LayerNorm kernels (qk_kernel.cuh).
#include <cuda_runtime.h>

#include <algorithm>

#include "qk_kernel.cuh"

namespace nts {

int launch_qknorm(const QkRequest* rq, int ntensors, float eps, int N, const QkOptions& opt,
                  cudaStream_t stream, const LaunchTuning& tune) {
  if (const int injected = take_injected_failure()) return injected;
  const int layernorm = opt.layernorm;
  const int ES = opt.in_e4m3 ? 1 : 2;
  const int NS = layernorm ? 2 : 1;
  const bool mx_out = opt.out_fmt >= 0;
  if (layernorm && opt.in_e4m3) return fail(NTS_ERR_UNSUPPORTED, "LayerNorm of E4M3 input");
  if (mx_out && (layernorm || opt.in_e4m3))
    return fail(NTS_ERR_UNSUPPORTED, "block-cast output of LayerNorm or E4M3 input");
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");
  // psum: fp32 parameters staged per CTA (gamma, and beta when given)
  int Wmax = 0, psum = 0;
  int64_t Tsum = 0;
  for (int k = 0; k < ntensors; ++k) {
    const int W = (int)(rq[k].H / N);
    Wmax = std::max(Wmax, W);
    psum += W * ((layernorm && rq[k].beta != nullptr) ? 2 : 1);
    Tsum += rq[k].T;
  }

  // The row shape (vectors per thread, threads per row) fits the widest
  // shard; narrower shards leave the extra slots idle.
  const RowShape rs = choose_row_shape(Wmax / 8, tune.force_vpt);
  if (rs.G == 0) return fail(NTS_ERR_UNSUPPORTED, "shard row too wide: H/N = %d", Wmax);

  // Rows per tile: up to four (at most 256 consumer threads: the kernel
  // keeps about 120 registers per thread, so larger CTAs cost residency),
  // fewer when there are few tokens so that the tiles spread over the GPU.
  int R = std::max(1, std::min(4, 256 / rs.G));
  while (R > 1 && (Tsum + R - 1) / R < (int64_t)2 * dev.sm_count / N) R /= 2;
  if (tune.force_rows > 0) R = tune.force_rows;
  if (R * rs.G > kMaxConsumers) return fail(NTS_ERR_UNSUPPORTED, "tile of %d rows too large", R);

  // Ring depth: up to 4 stages within the shared-memory budget; the widest
  // shards (whose staged gamma alone is up to 120 KB) fall back to fewer.
  // The variants bound by their per-row work rather than by DRAM take
  // fewer (measured on GB300 at [8192, 5120], N = 4, back-to-back launches):
  // the block-cast output of one tensor two (4-5 % faster than four),
  // of Q and K in one launch three (3 % faster than two), LayerNorm three
  // (1.5 % faster than two, which was 7-8 % faster than four), E4M3 input
  // three (3 % faster than four, 8 % faster than two).
  // gamma is split into the conflict-free layout when both copies fit.
  int gsplit = 1;
  int S = layernorm ? 3 : mx_out ? (ntensors > 1 ? 3 : 2) : (opt.in_e4m3 ? 3 : 4);
  const bool nvfp4 = mx_out && opt.out_fmt == NTS_FMT_NVFP4;
  auto layout = [&](int s, int split) {
    return qk_layout(N, s, R, Wmax, psum, rs.G, split, ES, NS, nvfp4);
  };
  while (S > 2 && layout(S, 1).total > (uint32_t)tune.smem_budget) --S;
  if (layout(S, 1).total > (uint32_t)dev.max_smem_optin) gsplit = 0;
  while (S > 1 && layout(S, gsplit).total > (uint32_t)dev.max_smem_optin) --S;
  if (tune.force_stages > 0) S = tune.force_stages;
  const QkLayout L = layout(S, gsplit);
  const size_t smem = L.total;
  if (smem > (size_t)dev.max_smem_optin)
    return fail(NTS_ERR_UNSUPPORTED, "shard row too wide for shared memory: H/N = %d", Wmax);

  const int bv = mx_out ? opt.B / 8 : 1;   // block-cast output: vectors per block
  // the kernels with G fixed at compile time serve one-warp shard rows that
  // fill all their vector slots, in every tensor of the launch, with gamma
  // in the split layout
  bool full = rs.G == 32 && gsplit == 1;
  for (int k = 0; k < ntensors; ++k) full = full && rq[k].H / N / 8 == (int64_t)rs.vpt * rs.G;
  const int gsel = full ? 32 : 0;
  QkKernel kern;
  if (mx_out)
    kern = opt.out_fmt == NTS_FMT_E4M3   ? pick_qk_mx_e4m3(N, rs.vpt, gsel, bv, ntensors)
           : opt.out_fmt == NTS_FMT_E2M1 ? pick_qk_mx_e2m1(N, rs.vpt, gsel, bv, ntensors)
                                         : pick_qk_mx_nvfp4(N, rs.vpt, gsel, bv, ntensors);
  else
    kern = layernorm    ? pick_qk_ln(N, rs.vpt, gsel, bv, ntensors)
           : opt.in_e4m3 ? pick_qk_e4m3(N, rs.vpt, gsel, bv, ntensors)
                         : pick_qk_bf16(N, rs.vpt, gsel, bv, ntensors);
  if (kern == nullptr) return fail(NTS_ERR_UNSUPPORTED, "no kernel for N=%d vpt=%d", N, rs.vpt);

  QkParams prm = {};
  uint32_t gam = L.gam;
  int64_t ntiles = 0;
  for (int k = 0; k < ntensors; ++k) {
    QkTensor& tn = prm.ten[k];
    tn.X = rq[k].X;
    tn.gamma = rq[k].gamma;
    tn.beta = layernorm ? rq[k].beta : nullptr;
    tn.mean_out = layernorm ? rq[k].mean : nullptr;
    tn.Y = static_cast<__nv_bfloat16*>(rq[k].Y);
    tn.codes = rq[k].codes;
    tn.scales = rq[k].scales;
    tn.rinv_out = rq[k].rinv;
    tn.T = rq[k].T;
    tn.ntiles = (rq[k].T + R - 1) / R;
    tn.H = (int)rq[k].H;
    tn.inv_H = (float)(1.0 / (double)rq[k].H);
    tn.W = (int)(rq[k].H / N);
    tn.nvec = tn.W / 8;
    tn.gam = gam;
    gam += (uint32_t)tn.W * 4;
    if (tn.beta != nullptr) {
      tn.bet = gam;
      gam += (uint32_t)tn.W * 4;
    }
    ntiles += tn.ntiles;
  }
  prm.ntensors = ntensors;
  prm.ntiles = ntiles;
  prm.Wmax = Wmax;
  prm.G = rs.G;
  prm.R = R;
  prm.S = S;
  prm.gsplit = gsplit;
  prm.psum = psum;
  prm.bv = mx_out ? opt.B / 8 : 1;
  prm.bshift = 0;
  while (mx_out && (1 << prm.bshift) < opt.B) ++prm.bshift;   // B = 2^bshift
  prm.eps = eps;
  prm.x_scale = opt.x_scale;
  prm.wait_limit_ns = tune.wait_limit_ns;
  prm.missing_tx = tune.missing_tx;
  prm.sched = tune.dynamic ? sched_counters(stream) : nullptr;
  if (ntiles == 0) return NTS_OK;

  // Decode-sized launches (every tile in one wave of single-tile clusters):
  // the kernel without producer, ring or mbarriers (qk_direct.cu).  It has
  // no waits, so the missing-bytes test hook keeps the persistent kernel.
  if (tune.direct && !mx_out && rs.vpt <= 5 && tune.force_rows == 0 &&
      tune.force_stages == 0 && tune.force_grid == 0 && tune.missing_tx == 0) {
    QkKernel dk = pick_qk_direct(N, rs.vpt, opt.in_e4m3, layernorm);
    const size_t dsmem = (size_t)R * N * (rs.G / 32) * 4 * NS;
    cudaLaunchConfig_t dc = {};
    cudaLaunchAttribute da[3];
    da[0].id = cudaLaunchAttributeClusterDimension;
    da[0].val.clusterDim.x = N;
    da[0].val.clusterDim.y = 1;
    da[0].val.clusterDim.z = 1;
    da[1] = cluster_policy_attribute();
    dc.blockDim = dim3(R * rs.G);
    dc.dynamicSmemBytes = dsmem;
    dc.stream = stream;
    dc.attrs = da;
    dc.numAttrs = 2;
    int64_t dmax = 0;
    int rc = dk != nullptr ? max_active_clusters((const void*)dk, dc, N, &dmax) : NTS_OK;
    if (rc != NTS_OK) return rc;
    if (dk != nullptr && ntiles <= dmax) {
      dc.gridDim = dim3((unsigned)(ntiles * N));
      da[2] = pdl_attribute();
      dc.numAttrs = tune.pdl ? 3 : 2;
      log_launch(layernorm ? "layernorm_split" : "qknorm_rms", "direct: tensors=%d T=%lld H=%d N=%d vpt=%d G=%d R=%d clusters=%lld",
                 ntensors, (long long)rq[0].T, (int)rq[0].H, N, rs.vpt, rs.G, R,
                 (long long)ntiles);
      const cudaError_t e = cudaLaunchKernelEx(&dc, dk, prm);
      if (e != cudaSuccess) return fail_cuda(e, "launching qknorm_rms");
      return NTS_OK;
    }
  }

  const int nthreads = R * rs.G + 32;  // consumers + producer warp
  int rc = prepare_kernel((const void*)kern, smem);
  if (rc != NTS_OK) return rc;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = N;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = cluster_policy_attribute();
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;

  int64_t max_clusters = 0;
  rc = max_active_clusters((const void*)kern, cfg, N, &max_clusters);
  if (rc != NTS_OK) return rc;
  int64_t ncl = std::min<int64_t>(ntiles, max_clusters);
  if (tune.force_grid > 0) ncl = std::min<int64_t>(ntiles, tune.force_grid);
  cfg.gridDim = dim3((unsigned)(ncl * N));
  attr[2] = pdl_attribute();
  cfg.numAttrs = tune.pdl ? 3 : 2;

  log_launch(layernorm ? "layernorm_split" : (mx_out ? "qknorm_rms_mxcast" : "qknorm_rms"),
             "tensors=%d T=%lld H=%d N=%d vpt=%d G=%d R=%d S=%d gsplit=%d "
             "smem=%zu clusters=%lld/%lld", ntensors, (long long)rq[0].T, (int)rq[0].H, N, rs.vpt,
             rs.G, R, S, gsplit, smem, (long long)ncl, (long long)max_clusters);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return fail_cuda(e, layernorm ? "launching layernorm_split" : "launching qknorm_rms");
  return NTS_OK;
}

int read_and_clear_qk_status(unsigned* out) {
  int (*const readers[])(unsigned*) = {
      read_and_clear_qk_bf16_status,    read_and_clear_qk_e4m3_status,
      read_and_clear_qk_ln_status,      read_and_clear_qk_mx_e4m3_status,
      read_and_clear_qk_mx_e2m1_status, read_and_clear_qk_mx_nvfp4_status,
      read_and_clear_heads_status};
  unsigned all = 0;
  for (auto* read : readers) {
    unsigned v = 0;
    const int rc = read(&v);
    if (rc != NTS_OK) return rc;
    all |= v;
  }
  *out = all;
  return NTS_OK;
}

}  // namespace nts
