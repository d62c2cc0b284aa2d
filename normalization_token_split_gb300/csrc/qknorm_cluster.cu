// qknorm_cluster.cu -- layerwise QK-RMSNorm with split-H scalar partial sums
// on one GB300: the N shards of a row are the N CTAs of a thread-block
// cluster, and the per-shard sums of squares travel through distributed
// shared memory.
//
// Method (SwiftQK, Eq. (1) and Algorithm 1, Sec. III.A-D):
//   Phase A  each shard forms its local sum of squares in fp32;
//   Phase B  the partial sums are exchanged and combined while the weight
//            product x*gamma, which does not depend on them, is formed;
//   Phase C  y = (x*gamma) * 1/sqrt(S/H_total + eps), written once.
//
// GB300 mapping (what differs from the pages' multi-GPU kernel):
//  * shard k of every row is handled by CTA k of a cluster of N CTAs.  The
//    "remote write + spin on a peer flag" of Algorithm 1 becomes, per warp,
//    N st.async stores of its fp32 partial into the peers' shared memory,
//    each completing 4 transaction bytes on the receiving row's mbarrier.
//    A receiver waits on its own mbarrier only: no cluster barrier and no
//    memory fence sits in the token loop, so nothing waits for the previous
//    tile's global stores;
//  * Phase B is the window between those sends and the wait: every warp
//    multiplies its registers by gamma (one bulk copy into shared memory per
//    CTA, split once into a bank-conflict-free layout) with packed f32x2
//    instructions, then waits;
//  * start-up stays off the critical path: the producer issues gamma and the
//    first tiles at once, and consumers defer the cluster start-up wait to
//    their first exchange (a timeline probe showed a blocking prologue cost
//    ~4 us of a 60 us launch);
//  * the block-level token pipeline of Sec. III.D is a persistent loop over
//    tiles of R rows.  A producer warp keeps a ring of S shared-memory stages
//    filled with bulk TMA copies; consumer warps release a stage (an
//    "empty" mbarrier) as soon as its data is in registers;
//  * deadlock safety (Sec. III.D) needs no bounded grid: the hardware
//    co-schedules a cluster's CTAs and no CTA waits on another cluster.  The
//    grid is still sized from the cluster occupancy query, for throughput.
//    Every wait in the kernel is bounded in time (an expired wait sets the
//    status word and the kernel finishes with undefined outputs).
#include <cuda_runtime.h>

#include <algorithm>

#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

__device__ unsigned int g_qk_status;  // kStatusTimeout bits, read by nts_check_status

// One tensor normalized by a launch (a launch covers one or two: Q and K).
struct QkTensor {
  const __nv_bfloat16* X;
  const float* gamma;
  __nv_bfloat16* Y;
  float* rinv_out;
  int64_t T;
  int64_t ntiles;  // ceil(T / R)
  int H;           // full row width H_total
  int W;           // H / N, the columns of one shard
  int nvec;        // W / 8 16-byte vectors per shard row
  uint32_t gam;    // shared-memory offset of this tensor's staged gamma
};

struct QkParams {
  QkTensor ten[2];
  int ntensors;
  int64_t ntiles;  // tiles of all tensors; tensor 0's come first
  int Wmax;        // widest shard of the tensors
  int G;           // consumer threads per row (multiple of 32)
  int R;           // rows per tile
  int S;           // ring stages
  int gsplit;      // 1: gamma re-laid out into split halves; 0: read as copied
  float eps;
  uint64_t wait_limit_ns;
  uint32_t missing_tx;  // test hook: bytes expected on the first stage but never sent
};

// Shared memory layout (bytes, in order):
//   ring  [S][R][Wmax] bf16       the staged shard rows
//   gstg  per tensor [W] f32      gamma of this shard as copied (one bulk
//                                 copy); absent when gsplit == 0
//   gam   per tensor [2][nvec] float4: the same, split into the low and high
//         halves of each 8-value vector (conflict-free reads); when the
//         shards are too wide for both copies, gam holds gamma as copied
//   full  [S], empty [S]          ring mbarriers
//   gbar                          gamma-arrival mbarrier
//   xbar  [2][R]                  exchange mbarriers (double-buffered by tile)
//   part  [2][R][N][WPR] f32      partial sums received from every warp of
//                                 every shard of a row
struct QkLayout {
  uint32_t ring, gstg, gam, full, empty, gbar, xbar, part, total;
};

__host__ __device__ inline QkLayout qk_layout(int N, int S, int R, int Wmax, int Wsum, int G,
                                              int gsplit) {
  QkLayout L;
  L.ring = 0;
  L.gstg = L.ring + (uint32_t)S * R * Wmax * 2;
  L.gam = L.gstg + (gsplit ? (uint32_t)Wsum * 4 : 0u);
  L.full = L.gam + (uint32_t)Wsum * 4;
  L.empty = L.full + (uint32_t)S * 8;
  L.gbar = L.empty + (uint32_t)S * 8;
  L.xbar = L.gbar + 8;
  L.part = L.xbar + (uint32_t)2 * R * 8;
  L.total = L.part + (uint32_t)2 * R * N * (G / 32) * 4;
  return L;
}

// Tensor and first row of the tile with global index `tile`.
__device__ __forceinline__ int qk_tile(const QkParams& p, int64_t tile, int64_t* t0) {
  const int k = (p.ntensors > 1 && tile >= p.ten[0].ntiles) ? 1 : 0;
  *t0 = (tile - (k ? p.ten[0].ntiles : 0)) * p.R;
  return k;
}

template <int N, int VPT>
__global__ void __launch_bounds__(kMaxThreads, 1) qknorm_cluster_kernel(const QkParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t rank = (N > 1) ? cluster_ctarank() : 0u;
  const int64_t cid = cluster_id_x();
  const int64_t ncl = num_clusters_x();
  const int tid = threadIdx.x;
  const int nconsumer = p.R * p.G;
  const int lane = tid & 31;
  const int wpr = p.G >> 5;
  const int Wsum = p.ten[0].W + (p.ntensors > 1 ? p.ten[1].W : 0);
  const QkLayout L = qk_layout(N, p.S, p.R, p.Wmax, Wsum, p.G, p.gsplit);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t stage_bytes = (uint32_t)p.R * p.Wmax * 2;
  const int64_t my_tiles = cid < p.ntiles ? (p.ntiles - 1 - cid) / ncl + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < p.S; ++s) {
      mbar_init(sbase + L.full + 8 * s, 1);
      mbar_init(sbase + L.empty + 8 * s, nconsumer / 32);
    }
    for (int b = 0; b < 2 * p.R; ++b) mbar_init(sbase + L.xbar + 8 * b, 1);
    mbar_init(sbase + L.gbar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (tid >= nconsumer) {
    // ------------------------------------------------------ producer warp
    // It touches only this CTA's shared memory, so it starts the ring at
    // once; its half of the cluster start-up barrier is completed later.
    if (N > 1) cluster_arrive_relaxed();
    if (lane == 0) {
      bool aborted = false;
      // this shard's gamma first (every CTA re-reads it, so no evict hint)
      mbar_arrive_expect_tx(sbase + L.gbar, (uint32_t)Wsum * 4);
      for (int k = 0; k < p.ntensors; ++k)
        bulk_g2s_plain(sbase + p.ten[k].gam - L.gam + L.gstg,
                       p.ten[k].gamma + (size_t)rank * p.ten[k].W, (uint32_t)p.ten[k].W * 4,
                       sbase + L.gbar);
      const uint64_t policy = l2_policy_evict_first();
      for (int64_t j = 0; j < my_tiles; ++j) {
        const int s = (int)(j % p.S);
        if (j >= p.S &&
            !mbar_wait_bounded(sbase + L.empty + 8 * s, (uint32_t)((j / p.S - 1) & 1),
                               p.wait_limit_ns)) {
          atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
          break;
        }
        int64_t t0;
        const QkTensor& tn = p.ten[qk_tile(p, cid + j * ncl, &t0)];
        const int nrows = (int)min64(p.R, tn.T - t0);
        const uint32_t row_bytes = (uint32_t)tn.W * 2;
        const uint32_t bar = sbase + L.full + 8 * s;
        const uint32_t dst = sbase + L.ring + (uint32_t)s * stage_bytes;
        const __nv_bfloat16* src = tn.X + (size_t)t0 * tn.H + (size_t)rank * tn.W;
        mbar_arrive_expect_tx(bar, nrows * row_bytes + (j == 0 ? p.missing_tx : 0u));
        if (N == 1) {
          bulk_g2s(dst, src, nrows * row_bytes, bar, policy);
        } else {
          for (int r = 0; r < nrows; ++r)
            bulk_g2s(dst + r * row_bytes, src + (size_t)r * tn.H, row_bytes, bar, policy);
        }
      }
      // let the last copies land before this CTA can retire
      for (int64_t j = max64(0, my_tiles - p.S); j < my_tiles && !aborted; ++j)
        (void)mbar_wait_bounded(sbase + L.full + 8 * (int)(j % p.S), (uint32_t)((j / p.S) & 1),
                                p.wait_limit_ns);
      (void)mbar_wait_bounded(sbase + L.gbar, 0, p.wait_limit_ns);
    }
    __syncwarp();
    if (N > 1) cluster_wait_acquire();
  } else {
    // ------------------------------------------------------- consumer warps
    // Every CTA of the cluster must be running, with its barriers
    // initialised, before anyone stores into a peer's shared memory: arrive
    // now, wait just before the first exchange (the first tile's loads and
    // Phase A overlap the start-up).
    if (N > 1) cluster_arrive_release();
    bool started = (N == 1);
    bool have_gamma = false;

    const int row = tid / p.G;
    const int g = tid - row * p.G;
    const int wir = g >> 5;
    const bool exchange = (N > 1) || (wpr > 1);
    bool aborted = false;
    for (int64_t j = 0; j < my_tiles; ++j) {
      const int s = (int)(j % p.S);
      int64_t t0;
      const QkTensor& tn = p.ten[qk_tile(p, cid + j * ncl, &t0)];
      const int64_t t = t0 + row;
      const bool valid = t < tn.T;
      const int nvec = tn.nvec;

      if (!mbar_wait_bounded(sbase + L.full + 8 * s, (uint32_t)((j / p.S) & 1),
                             aborted ? 0 : p.wait_limit_ns)) {
        if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
        aborted = true;
      }

      // ---- Phase A: this shard's sum of squares (fp32, packed pairs).  The
      // values are converted once and kept as fp32 pairs in w; four
      // independent accumulators keep the FMA chains short.
      uint64_t w[VPT][4];
      uint64_t acc[4] = {0, 0, 0, 0};  // {0.f, 0.f} each
      const uint32_t srow = sbase + L.ring + (uint32_t)s * stage_bytes + (uint32_t)row * tn.W * 2;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = i * p.G + g;
        uint4 xr = make_uint4(0, 0, 0, 0);
        if (valid && v < nvec) xr = ld_shared_v4(srow + v * 16);
        w[i][0] = bf16x2_to_f2(xr.x);
        w[i][1] = bf16x2_to_f2(xr.y);
        w[i][2] = bf16x2_to_f2(xr.z);
        w[i][3] = bf16x2_to_f2(xr.w);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = f2_fma(w[i][q], w[i][q], acc[q]);
      }
      // the stage's data is in registers: hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(sbase + L.empty + 8 * s);
      const uint64_t a01 = f2_add(acc[0], acc[1]), a23 = f2_add(acc[2], acc[3]);
      const uint64_t a = f2_add(a01, a23);
      const float ss = warp_sum(f2_lo(a) + f2_hi(a));

      // ---- exchange: send this warp's partial to every shard of the row
      const int b = (int)(j & 1);
      const uint32_t xbar = sbase + L.xbar + 8 * (b * p.R + row);
      const uint32_t slot0 = sbase + L.part + 4 * (uint32_t)((b * p.R + row) * N * wpr);
      if (!started) {
        cluster_wait_acquire();
        started = true;
      }
      if (exchange) {
        if (g == 0) mbar_arrive_expect_tx(xbar, (uint32_t)(N * wpr * 4));
        if (lane == 0) {
          const uint32_t slot = slot0 + 4 * (rank * wpr + wir);
#pragma unroll
          for (int k = 0; k < N; ++k)
            st_async_f32(map_to_rank(slot, k), ss, map_to_rank(xbar, k));
        }
      }

      // ---- Phase B (overlapping the exchange): w = x * gamma, in place
      if (!have_gamma) {
        // once: wait for the copied gamma and split it into the layout the
        // loop reads (consecutive lanes, consecutive 16 bytes)
        if (!mbar_wait_bounded(sbase + L.gbar, 0, aborted ? 0 : p.wait_limit_ns)) {
          if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
        }
        for (int k = 0; k < p.ntensors && p.gsplit; ++k) {
          const QkTensor& tk = p.ten[k];
          const float4* src = reinterpret_cast<const float4*>(smem + tk.gam - L.gam + L.gstg);
          float4* dst = reinterpret_cast<float4*>(smem + tk.gam);
          for (int q = tid; q < tk.nvec; q += nconsumer) {
            dst[q] = src[2 * q];
            dst[tk.nvec + q] = src[2 * q + 1];
          }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nconsumer) : "memory");
        have_gamma = true;
      }
      // split layout: halves nvec*16 bytes apart, vectors 16 apart; as
      // copied: halves 16 apart, vectors 32 apart
      const uint32_t gam_lo = sbase + tn.gam;
      const uint32_t gam_hi = gam_lo + (p.gsplit ? (uint32_t)nvec * 16 : 16u);
      const uint32_t gstride = p.gsplit ? 16u : 32u;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = min(i * p.G + g, nvec - 1);
        const uint4 glo = ld_shared_v4(gam_lo + v * gstride);
        const uint4 ghi = ld_shared_v4(gam_hi + v * gstride);
        w[i][0] = f2_mul(w[i][0], f2(__uint_as_float(glo.x), __uint_as_float(glo.y)));
        w[i][1] = f2_mul(w[i][1], f2(__uint_as_float(glo.z), __uint_as_float(glo.w)));
        w[i][2] = f2_mul(w[i][2], f2(__uint_as_float(ghi.x), __uint_as_float(ghi.y)));
        w[i][3] = f2_mul(w[i][3], f2(__uint_as_float(ghi.z), __uint_as_float(ghi.w)));
      }

      // ---- combine in rank order (then warp order within a shard)
      float S = ss;
      if (exchange) {
        if (!mbar_wait_bounded(xbar, (uint32_t)((j >> 1) & 1), aborted ? 0 : p.wait_limit_ns)) {
          if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
        }
        const float* sl = reinterpret_cast<const float*>(smem + (slot0 - sbase));
        S = 0.f;
        for (int k = 0; k < N * wpr; ++k) S += sl[k];
      }

      // ---- Phase C: scale and store the shard
      if (valid) {
        const float rinv = 1.0f / sqrtf(S / (float)tn.H + p.eps);
        const uint64_t rr = f2(rinv, rinv);
        __nv_bfloat16* yrow = tn.Y + (size_t)t * tn.H + (size_t)rank * tn.W;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = i * p.G + g;
          if (v < nvec) {
            uint4 o;
            const uint64_t y0 = f2_mul(w[i][0], rr), y1 = f2_mul(w[i][1], rr);
            const uint64_t y2 = f2_mul(w[i][2], rr), y3 = f2_mul(w[i][3], rr);
            o.x = pack_bf16x2_rn(f2_lo(y0), f2_hi(y0));
            o.y = pack_bf16x2_rn(f2_lo(y1), f2_hi(y1));
            o.z = pack_bf16x2_rn(f2_lo(y2), f2_hi(y2));
            o.w = pack_bf16x2_rn(f2_lo(y3), f2_hi(y3));
            st_global_v4_stream(yrow + v * 8, o);
          }
        }
        if (tn.rinv_out != nullptr && rank == 0 && g == 0) tn.rinv_out[t] = rinv;
      }
    }
    if (!started) cluster_wait_acquire();  // a CTA without tiles
  }

  // No CTA leaves while a peer may still store into its shared memory.
  if (N > 1) {
    cluster_arrive_release();
    cluster_wait_acquire();
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

}  // namespace

int launch_qknorm(const QkRequest* rq, int ntensors, float eps, int N, cudaStream_t stream,
                  const LaunchTuning& tune) {
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");
  int Wmax = 0, Wsum = 0;
  int64_t Tsum = 0;
  for (int k = 0; k < ntensors; ++k) {
    Wmax = std::max(Wmax, (int)(rq[k].H / N));
    Wsum += (int)(rq[k].H / N);
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
  // gamma is split into the conflict-free layout when both copies fit.
  int gsplit = 1;
  int S = 4;
  while (S > 2 && qk_layout(N, S, R, Wmax, Wsum, rs.G, 1).total > (uint32_t)tune.smem_budget) --S;
  if (qk_layout(N, S, R, Wmax, Wsum, rs.G, 1).total > (uint32_t)dev.max_smem_optin) gsplit = 0;
  while (S > 1 && qk_layout(N, S, R, Wmax, Wsum, rs.G, gsplit).total > (uint32_t)dev.max_smem_optin)
    --S;
  if (tune.force_stages > 0) S = tune.force_stages;
  const QkLayout L = qk_layout(N, S, R, Wmax, Wsum, rs.G, gsplit);
  const size_t smem = L.total;
  if (smem > (size_t)dev.max_smem_optin)
    return fail(NTS_ERR_UNSUPPORTED, "shard row too wide for shared memory: H/N = %d", Wmax);

  QkKernel kern = pick_qk(N, rs.vpt);
  if (kern == nullptr) return fail(NTS_ERR_UNSUPPORTED, "no kernel for N=%d vpt=%d", N, rs.vpt);

  QkParams prm = {};
  uint32_t gam = L.gam;
  int64_t ntiles = 0;
  for (int k = 0; k < ntensors; ++k) {
    QkTensor& tn = prm.ten[k];
    tn.X = static_cast<const __nv_bfloat16*>(rq[k].X);
    tn.gamma = rq[k].gamma;
    tn.Y = static_cast<__nv_bfloat16*>(rq[k].Y);
    tn.rinv_out = rq[k].rinv;
    tn.T = rq[k].T;
    tn.ntiles = (rq[k].T + R - 1) / R;
    tn.H = (int)rq[k].H;
    tn.W = (int)(rq[k].H / N);
    tn.nvec = tn.W / 8;
    tn.gam = gam;
    gam += (uint32_t)tn.W * 4;
    ntiles += tn.ntiles;
  }
  prm.ntensors = ntensors;
  prm.ntiles = ntiles;
  prm.Wmax = Wmax;
  prm.G = rs.G;
  prm.R = R;
  prm.S = S;
  prm.gsplit = gsplit;
  prm.eps = eps;
  prm.wait_limit_ns = tune.wait_limit_ns;
  prm.missing_tx = tune.missing_tx;
  if (ntiles == 0) return NTS_OK;

  const int nthreads = R * rs.G + 32;  // consumers + producer warp
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
  int64_t ncl = std::min<int64_t>(ntiles, max_clusters);
  if (tune.force_grid > 0) ncl = std::min<int64_t>(ntiles, tune.force_grid);
  cfg.gridDim = dim3((unsigned)(ncl * N));

  log_launch("qknorm_rms", "tensors=%d T=%lld H=%d N=%d vpt=%d G=%d R=%d S=%d gsplit=%d "
             "smem=%zu clusters=%lld/%lld", ntensors, (long long)rq[0].T, (int)rq[0].H, N, rs.vpt,
             rs.G, R, S, gsplit, smem, (long long)ncl, (long long)max_clusters);
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
