// qknorm_cluster.cu -- layerwise QK-RMSNorm with split-H scalar partial sums
// on one GB300: the N shards of a row are the N CTAs of a thread-block
// cluster, and the per-shard sums of squares are exchanged through
// distributed shared memory.
//
// Method (SwiftQK, Eq. (1) and Algorithm 1, Sec. III.A-D):
//   Phase A  each shard forms its local sum of squares in fp32;
//   Phase B  the partial sums are exchanged and combined while the weight
//            product x*gamma, which does not depend on them, is formed;
//   Phase C  y = (x*gamma) * 1/sqrt(S/H_total + eps), written once.
//
// GB300 mapping (what differs from the pages' multi-GPU kernel):
//  * shard k of every row is handled by CTA k of a cluster of N CTAs, so the
//    "remote write + spin on a peer flag" of Algorithm 1 becomes N stores to
//    the peers' shared memory (st.shared::cluster) followed by a split
//    hardware cluster barrier (arrive.release ... wait.acquire);
//  * the overlap of Phase B is between the two halves of that split barrier:
//    every warp issues x*gamma after arriving and only then waits;
//  * the block-level token pipeline of Sec. III.D is a persistent loop over
//    tiles of R rows, fed by a ring of S shared-memory stages that one thread
//    fills with bulk TMA copies (cp.async.bulk) S-1 tiles ahead;
//  * deadlock safety (Sec. III.D) needs no bounded grid here: the hardware
//    co-schedules a cluster's CTAs and no CTA waits on another cluster.  The
//    grid is still sized from the cluster occupancy query, for throughput.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

__device__ unsigned int g_qk_status;  // kStatusTimeout bits, read by nts_check_status

struct QkParams {
  const __nv_bfloat16* X;
  const float* gamma;
  __nv_bfloat16* Y;
  float* rinv_out;
  int64_t T;
  int64_t ntiles;
  int H;        // full row width H_total
  int W;        // H / N, the columns of one shard
  int nvec;     // W / 8 16-byte vectors per shard row
  int G;        // threads per row (multiple of 32)
  int R;        // rows per tile
  int S;        // ring stages
  float eps;
  uint64_t wait_limit_ns;
  uint32_t missing_tx;  // test hook: bytes expected on the first stage but never sent
};

// Shared memory: ring[S][R][W] bf16 | full[S] mbarriers | part[2][R][N][WPR] f32.
template <int N>
__host__ __device__ inline size_t qk_smem_bytes(int S, int R, int W, int G) {
  size_t ring = (size_t)S * R * W * 2;
  size_t bars = (size_t)S * 8;
  size_t part = (size_t)2 * R * N * (G / 32) * 4;
  return ring + bars + part;
}

template <int N, int VPT>
__global__ void __launch_bounds__(kMaxThreads, 1) qknorm_cluster_kernel(const QkParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t rank = (N > 1) ? cluster_ctarank() : 0u;
  const int64_t cid = cluster_id_x();
  const int64_t ncl = num_clusters_x();
  const int tid = threadIdx.x;
  const int row = tid / p.G;
  const int g = tid - row * p.G;
  const int wpr = p.G >> 5;
  const int wir = g >> 5;
  const int lane = tid & 31;

  const uint32_t stage_bytes = (uint32_t)p.R * p.W * 2;
  const uint32_t ring = smem_addr(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.S * stage_bytes);
  float* part = reinterpret_cast<float*>(full + p.S);

  const int64_t my_tiles = cid < p.ntiles ? (p.ntiles - 1 - cid) / ncl + 1 : 0;
  const __nv_bfloat16* Xs = p.X + (size_t)rank * p.W;  // this shard's column origin

  if (tid == 0) {
    for (int s = 0; s < p.S; ++s) mbar_init(smem_addr(&full[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Peers must be running before anyone stores into their shared memory:
  // this arrive is matched by a wait just before the first exchange.
  if (N > 1) cluster_arrive_relaxed();

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int64_t j) {
    const int64_t t0 = (cid + j * ncl) * p.R;
    const int nrows = (int)min64(p.R, p.T - t0);
    const int s = (int)(j % p.S);
    const uint32_t bar = smem_addr(&full[s]);
    const uint32_t row_bytes = (uint32_t)p.W * 2;
    mbar_arrive_expect_tx(bar, nrows * row_bytes + (j == 0 ? p.missing_tx : 0u));
    const uint32_t dst = ring + (uint32_t)s * stage_bytes;
    for (int r = 0; r < nrows; ++r)
      bulk_g2s(dst + r * row_bytes, Xs + (size_t)(t0 + r) * p.H, row_bytes, bar, policy);
  };

  if (tid == 0) {
    const int64_t pre = min64(p.S, my_tiles);
    for (int64_t j = 0; j < pre; ++j) issue(j);
  }

  bool aborted = false;
  bool first = true;
  for (int64_t j = 0; j < my_tiles; ++j) {
    const int s = (int)(j % p.S);
    const uint32_t parity = (uint32_t)((j / p.S) & 1);
    const int64_t t = (cid + j * ncl) * p.R + row;
    const bool valid = t < p.T;

    if (!mbar_wait_bounded(smem_addr(&full[s]), parity, aborted ? 0 : p.wait_limit_ns)) {
      if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
      aborted = true;
    }

    // ---- Phase A: local sum of squares of this shard (fp32).
    uint4 xr[VPT];
    float ss = 0.f;
    const uint32_t srow = ring + (uint32_t)s * stage_bytes + (uint32_t)row * p.W * 2;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = i * p.G + g;
      if (valid && v < p.nvec) {
        xr[i] = ld_shared_v4(srow + v * 16);
        float f[8];
        bf16x8_to_f32(xr[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
      } else {
        xr[i] = make_uint4(0, 0, 0, 0);
      }
    }
    ss = warp_sum(ss);

    // ---- Exchange: every warp publishes its partial into slot
    // part[j&1][row][rank][wir] of every CTA of the cluster.
    if (N > 1 && first) cluster_wait_acquire();
    first = false;
    if (lane == 0) {
      float* slot = part + ((((size_t)(j & 1) * p.R + row) * N + rank) * wpr + wir);
      const uint32_t local = smem_addr(slot);
#pragma unroll
      for (int k = 0; k < N; ++k) st_cluster_f32(map_to_rank(local, k), ss);
    }
    cluster_arrive_release();

    // ---- Phase B (overlapped with the exchange): w = x * gamma.
    float w[VPT][8];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = i * p.G + g;
      float f[8];
      bf16x8_to_f32(xr[i], f);
      if (valid && v < p.nvec) {
        const float4* gp = reinterpret_cast<const float4*>(p.gamma + (size_t)rank * p.W + v * 8);
        const float4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
        w[i][0] = f[0] * g0.x; w[i][1] = f[1] * g0.y; w[i][2] = f[2] * g0.z; w[i][3] = f[3] * g0.w;
        w[i][4] = f[4] * g1.x; w[i][5] = f[5] * g1.y; w[i][6] = f[6] * g1.z; w[i][7] = f[7] * g1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[i][e] = 0.f;
      }
    }
    cluster_wait_acquire();

    // Every thread of this CTA has finished Phase A of tile j: stage s is
    // free for tile j + S.
    if (tid == 0 && !aborted && j + p.S < my_tiles) issue(j + p.S);

    // ---- Phase C: combine in rank order, scale, store the shard.
    if (valid) {
      const float* sl = part + (((size_t)(j & 1) * p.R + row) * N) * wpr;
      float S = 0.f;
      for (int k = 0; k < N * wpr; ++k) S += sl[k];
      const float rinv = 1.0f / sqrtf(S / (float)p.H + p.eps);
      __nv_bfloat16* yrow = p.Y + (size_t)t * p.H + (size_t)rank * p.W;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = i * p.G + g;
        if (v < p.nvec) {
          uint4 o;
          o.x = pack_bf16x2_rn(w[i][0] * rinv, w[i][1] * rinv);
          o.y = pack_bf16x2_rn(w[i][2] * rinv, w[i][3] * rinv);
          o.z = pack_bf16x2_rn(w[i][4] * rinv, w[i][5] * rinv);
          o.w = pack_bf16x2_rn(w[i][6] * rinv, w[i][7] * rinv);
          st_global_v4_stream(yrow + v * 8, o);
        }
      }
      if (p.rinv_out != nullptr && rank == 0 && g == 0) p.rinv_out[t] = rinv;
    }
  }
  // A CTA with no tiles still matches its start-up arrive.
  if (N > 1 && first) cluster_wait_acquire();

  // After a timeout, let copies still in flight land before the CTA's shared
  // memory is released (bounded again).
  if (aborted && tid == 0) {
    for (int64_t j = max64(0, my_tiles - p.S); j < my_tiles; ++j)
      (void)mbar_wait_bounded(smem_addr(&full[j % p.S]), (uint32_t)((j / p.S) & 1),
                              p.wait_limit_ns);
  }
}

// ------------------------------------------------------------------ launch

namespace {

using QkKernel = void (*)(QkParams);

template <int N>
QkKernel pick_qk_kernel(int vpt) {
  switch (vpt) {
    case 1: return qknorm_cluster_kernel<N, 1>;
    case 2: return qknorm_cluster_kernel<N, 2>;
    case 3: return qknorm_cluster_kernel<N, 3>;
    case 4: return qknorm_cluster_kernel<N, 4>;
    case 5: return qknorm_cluster_kernel<N, 5>;
    case 6: return qknorm_cluster_kernel<N, 6>;
    case 8: return qknorm_cluster_kernel<N, 8>;
    default: return nullptr;
  }
}

QkKernel pick_qk(int N, int vpt) {
  switch (N) {
    case 1: return pick_qk_kernel<1>(vpt);
    case 2: return pick_qk_kernel<2>(vpt);
    case 4: return pick_qk_kernel<4>(vpt);
    case 8: return pick_qk_kernel<8>(vpt);
    default: return nullptr;
  }
}

size_t qk_smem(int N, int S, int R, int W, int G) {
  switch (N) {
    case 1: return qk_smem_bytes<1>(S, R, W, G);
    case 2: return qk_smem_bytes<2>(S, R, W, G);
    case 4: return qk_smem_bytes<4>(S, R, W, G);
    default: return qk_smem_bytes<8>(S, R, W, G);
  }
}

}  // namespace

int launch_qknorm(const void* X, const float* gamma, void* Y, float* rinv, int64_t T, int H,
                  float eps, int N, cudaStream_t stream, const LaunchTuning& tune) {
  const int W = H / N;
  const int nvec = W / 8;
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");

  RowShape rs = choose_row_shape(nvec, tune.force_vpt);
  if (rs.G == 0) return fail(NTS_ERR_UNSUPPORTED, "shard row too wide: H/N = %d", W);

  // Rows per tile: about 256 threads per CTA, fewer when T is small so that
  // the tiles spread over the GPU.
  int R = std::max(1, 256 / rs.G);
  R = std::min(R, 16);
  while (R > 1 && (T + R - 1) / R < (int64_t)2 * dev.sm_count / N) R /= 2;
  if (tune.force_rows > 0) R = tune.force_rows;
  if (R * rs.G > kMaxThreads) return fail(NTS_ERR_UNSUPPORTED, "tile of %d rows too large", R);

  // Ring depth: as many stages (up to 4) as fit in ~100 KB, at least 2 when
  // one row-tile allows it.
  const size_t stage = (size_t)R * W * 2;
  int S = 4;
  while (S > 1 && qk_smem(N, S, R, W, rs.G) > (size_t)tune.smem_budget) --S;
  if (tune.force_stages > 0) S = tune.force_stages;
  const size_t smem = qk_smem(N, S, R, W, rs.G);
  if (smem > (size_t)dev.max_smem_optin || stage == 0)
    return fail(NTS_ERR_UNSUPPORTED, "shard row too wide for shared memory: H/N = %d", W);

  QkKernel kern = pick_qk(N, rs.vpt);
  if (kern == nullptr) return fail(NTS_ERR_UNSUPPORTED, "no kernel for N=%d vpt=%d", N, rs.vpt);

  QkParams prm;
  prm.X = static_cast<const __nv_bfloat16*>(X);
  prm.gamma = gamma;
  prm.Y = static_cast<__nv_bfloat16*>(Y);
  prm.rinv_out = rinv;
  prm.T = T;
  prm.ntiles = (T + R - 1) / R;
  prm.H = H;
  prm.W = W;
  prm.nvec = nvec;
  prm.G = rs.G;
  prm.R = R;
  prm.S = S;
  prm.eps = eps;
  prm.wait_limit_ns = tune.wait_limit_ns;
  prm.missing_tx = tune.missing_tx;

  const int nthreads = R * rs.G;
  int rc = prepare_kernel((const void*)kern, smem);
  if (rc != NTS_OK) return rc;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = N;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  int64_t max_clusters = 0;
  rc = max_active_clusters((const void*)kern, cfg, N, &max_clusters);
  if (rc != NTS_OK) return rc;
  int64_t ncl = std::min<int64_t>(prm.ntiles, max_clusters);
  if (tune.force_grid > 0) ncl = std::min<int64_t>(prm.ntiles, tune.force_grid);
  cfg.gridDim = dim3((unsigned)(ncl * N));

  log_launch("qknorm_rms", "T=%lld H=%d N=%d vpt=%d G=%d R=%d S=%d smem=%zu clusters=%lld/%lld",
             (long long)T, H, N, rs.vpt, rs.G, R, S, smem, (long long)ncl,
             (long long)max_clusters);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return fail_cuda(e, "launching qknorm_rms");
  return NTS_OK;
}

int read_and_clear_qk_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qk_status, sizeof(v));
  if (e != cudaSuccess) return fail_cuda(e, "reading the qknorm status word");
  e = cudaMemcpyToSymbol(g_qk_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clearing the qknorm status word");
  *out = v;
  return NTS_OK;
}

}  // namespace nts
