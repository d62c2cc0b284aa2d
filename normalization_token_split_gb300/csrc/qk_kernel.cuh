// qk_kernel.cuh -- layerwise QK-RMSNorm with split-H scalar partial sums
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
#pragma once

#include <cuda_runtime.h>

#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

// kStatusTimeout bits of the QK kernels of the including translation unit;
// every unit has its own word (no relocatable device code).
static __device__ unsigned int g_qk_status;

// Element type of the activations read by a launch.
enum { kInBf16 = 0, kInE4M3 = 1 };
// Statistic: RMSNorm (one sum of squares) or LayerNorm (sum and sum of
// squares, the SwiftQK notes' two additive scalars, Sec. 5e).
enum { kQkRms = 0, kQkLn = 1 };
// Output: bf16 rows, or the block cast of the normalized rows (MX E4M3 or
// E2M1 codes with E8M0 scales, or NVFP4) written in place of them.
enum { kOutBf16 = 0, kOutE4M3 = 1, kOutE2M1 = 2, kOutNvfp4 = 3 };

// One tensor normalized by a launch (a launch covers one or two: Q and K).
struct QkTensor {
  const void* X;   // bf16 or E4M3 codes [T, H]
  const float* gamma;
  const float* beta;     // LayerNorm shift (nullable)
  __nv_bfloat16* Y;
  uint8_t* codes;        // block-cast output: element codes [T, H] or [T, H/2]
  uint8_t* scales;       // ... and block scales [T, H/B]
  float* rinv_out;       // RMSNorm: 1/rms; LayerNorm: 1/sqrt(var + eps)
  float* mean_out;       // LayerNorm mean (nullable)
  int64_t T;
  int64_t ntiles;  // ceil(T / R)
  int H;           // full row width H_total
  float inv_H;     // fp32(1 / H)
  int W;           // H / N, the columns of one shard
  int nvec;        // W / 8 16-byte vectors per shard row
  uint32_t gam;    // shared-memory offset of this tensor's staged gamma
  uint32_t bet;    // ... and of its staged beta (0 when beta is NULL)
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
  int psum;        // fp32 parameters staged per CTA (gamma, and beta, of every tensor)
  int bv;          // block-cast output: 16-byte vectors per block (B / 8)
  int bshift;      // ... and log2(B)
  float eps;
  float x_scale;   // E4M3 input: value = code * x_scale
  uint64_t wait_limit_ns;
  uint32_t missing_tx;  // test hook: bytes expected on the first stage but never sent
  unsigned int* sched;  // zeroed counter pair (next tile, clusters done), or
                        // nullptr: every tile in round-robin order
};

// Shared memory layout (bytes, in order):
//   ring  [S][R][Wmax] elements   the staged shard rows (2 or 1 bytes each)
//   gstg  per tensor [W] f32      gamma (and beta) of this shard as copied
//                                 (bulk copies); absent when gsplit == 0
//   gam   per tensor [2][nvec] float4: the same, split into the low and high
//         halves of each 8-value vector (conflict-free reads); when the
//         shards are too wide for both copies, gam holds them as copied
//   full  [S], empty [S]          ring mbarriers
//   gbar                          gamma-arrival mbarrier
//   gsync                         consumers' mbarrier after the gamma relayout
//   xbar  [2][R]                  exchange mbarriers (double-buffered by tile)
//   tbar  [S+1]                   tile-number mbarriers (dynamic order, N > 1)
//   tile  [S+1] i64               tile numbers sent by the cluster's rank 0
//   tloc  [S] i64                 tile in stage s for the consumers (-1: done)
//   part  [2][R][N][WPR][NS] f32  partial sums received from every warp of
//                                 every shard of a row (NS = 1 RMS, 2 LN)
struct QkLayout {
  uint32_t ring, gstg, gam, full, empty, gbar, xbar, tbar, tile, tloc, part, rcp, total;
};

// rcp: the NVFP4 scale reciprocals (128 floats), or for LayerNorm the
// {n, 1/n} pairs of every warp of a shard row of each tensor ([2][16]
// float2); empty otherwise.
__host__ __device__ inline QkLayout qk_layout(int N, int S, int R, int Wmax, int Wsum, int G,
                                              int gsplit, int esize, int ns, bool nvfp4) {
  QkLayout L;
  L.ring = 0;
  L.gstg = L.ring + (uint32_t)S * R * Wmax * esize;
  L.gam = L.gstg + (gsplit ? (uint32_t)Wsum * 4 : 0u);
  L.full = L.gam + (uint32_t)Wsum * 4;
  L.empty = L.full + (uint32_t)S * 8;
  L.gbar = L.empty + (uint32_t)S * 8;
  L.xbar = L.gbar + 16;   // gbar, then gsync
  L.tbar = L.xbar + (uint32_t)2 * R * 8;
  L.tile = L.tbar + (uint32_t)(S + 1) * 8;
  L.tloc = L.tile + (uint32_t)(S + 1) * 8;
  L.part = L.tloc + (uint32_t)S * 8;
  L.rcp = L.part + (uint32_t)2 * R * N * (G / 32) * 4 * ns;
  L.total = L.rcp + (nvfp4 ? 128u * 4u : (ns == 2 ? 2u * 16u * 8u : 0u));
  return L;
}

// Tensor and first row of the tile with global index `tile`.
__device__ __forceinline__ int qk_tile(const QkParams& p, int64_t tile, int64_t* t0) {
  const int k = (p.ntensors > 1 && tile >= p.ten[0].ntiles) ? 1 : 0;
  *t0 = (tile - (k ? p.ten[0].ntiles : 0)) * p.R;
  return k;
}

// Eight activations of vector v of a staged row as four fp32 pairs; zeros
// when !inb (the load is predicated, the conversion is not).
template <int IN>
__device__ __forceinline__ void load_vector(const unsigned char* srow, int v, bool inb,
                                            float x_scale, uint64_t (&w)[4]) {
  if (IN == kInBf16) {
    uint4 x = make_uint4(0, 0, 0, 0);
    if (inb) x = lds128(srow + v * 16);
    w[0] = bf16x2_to_f2(x.x);
    w[1] = bf16x2_to_f2(x.y);
    w[2] = bf16x2_to_f2(x.z);
    w[3] = bf16x2_to_f2(x.w);
  } else {
    uint2 x = make_uint2(0, 0);
    if (inb) x = lds64(srow + v * 8);
    const uint64_t sc = f2(x_scale, x_scale);
    w[0] = f2_mul(e4m3x2_to_f2((uint16_t)(x.x & 0xFFFFu)), sc);
    w[1] = f2_mul(e4m3x2_to_f2((uint16_t)(x.x >> 16)), sc);
    w[2] = f2_mul(e4m3x2_to_f2((uint16_t)(x.y & 0xFFFFu)), sc);
    w[3] = f2_mul(e4m3x2_to_f2((uint16_t)(x.y >> 16)), sc);
  }
}

// ---- LayerNorm statistics that combine exactly across shards and warps
//
// The SwiftQK notes (Sec. 5e) reduce LayerNorm to two scalars per shard that
// add up across shards.  Sending (sum x, sum x^2) and forming
// var = sum x^2 / H - mu^2 loses var to cancellation when |mu| >> sigma, so
// each warp sends instead its sum s1 and M2 = sum (x - m)^2 about its own
// mean m = s1 * fp32(1/n) (n: its number of values).  With mu the row mean,
//   sum (x - mu)^2 = sum_k [ M2_k + n_k (m_k - mu)^2 ]
// (the parallel-axis identity, exact for means used consistently; Chan,
// Golub and LeVeque's pairwise update), still two scalars per warp.

// Values of the row shard held by warp `wir`: vectors i*G + 32*wir + lane
// below nvec, 8 values each.
template <int VPT>
__device__ __forceinline__ int ln_warp_count(int nvec, int G, int wir) {
  int n = 0;
#pragma unroll
  for (int i = 0; i < VPT; ++i) n += min(max(nvec - i * G - 32 * wir, 0), 32);
  return 8 * n;
}

// {n, fp32(1/n)} of a warp's count n (1/n = 0 for an empty warp): the mean a
// warp's M2 is taken about is s1 * fp32(1/n), the same expression on the
// sending and on the receiving side.
__device__ __forceinline__ float2 ln_count_pair(int n) {
  return make_float2((float)n, n > 0 ? 1.0f / (float)n : 0.f);
}

// s1 and M2 of this warp's values w (vectors beyond nvec hold zeros and are
// left out of M2; FULL: there are none); `c` = ln_count_pair of the warp's
// count; whole warp.
template <int VPT, bool FULL>
__device__ __forceinline__ void ln_warp_stats(const uint64_t (&w)[VPT][4], int G, int g, int nvec,
                                              float2 c, float* s1_out, float* m2_out) {
  uint64_t c0 = 0, c1 = 0;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    c0 = f2_add(c0, f2_add(w[i][0], w[i][1]));
    c1 = f2_add(c1, f2_add(w[i][2], w[i][3]));
  }
  const uint64_t cs = f2_add(c0, c1);
  const float s1 = warp_sum(f2_lo(cs) + f2_hi(cs));
  const float m = s1 * c.y;
  const uint64_t nm = f2(-m, -m);
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (FULL || i * G + g < nvec) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t d = f2_add(w[i][q], nm);
        acc[q] = f2_fma(d, d, acc[q]);
      }
    }
  }
  const uint64_t a = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  *s1_out = s1;
  *m2_out = warp_sum(f2_lo(a) + f2_hi(a));
}

// Row mean and variance from the (s1, M2) pairs of the row's N shards x
// wpr warps (`parts`, rank order then warp order, pairs 8 bytes apart),
// every shard's warps laid out alike; cnt(w) = ln_count_pair of warp w.
template <typename Cnt>
__device__ __forceinline__ void ln_combine(const float* parts, int N, int wpr, Cnt cnt,
                                           float inv_H, float* mu_out, float* var_out) {
  float s1 = 0.f;
  for (int k = 0; k < N * wpr; ++k) s1 += parts[2 * k];
  const float mu = s1 * inv_H;
  float m2 = 0.f;
  for (int w = 0; w < wpr; ++w) {
    const float2 c = cnt(w);
    for (int r = 0; r < N; ++r) {
      const float* pk = parts + 2 * (r * wpr + w);
      const float d = pk[0] * c.y - mu;
      m2 = fmaf(c.x * d, d, m2 + pk[1]);
    }
  }
  *mu_out = mu;
  *var_out = m2 * inv_H;
}

// Registers: 96 per thread (4 CTAs of 160 threads per SM) beat 128 (3 CTAs)
// by 5-12 % on GB300, and 112 or 72-80 by 5-15 %, for every variant (the
// LayerNorm kernel takes 92 at 96 with no spills, 2-6 % faster than at 104,
// where it took 102 and 3 CTAs).  At 8 vectors per thread LayerNorm keeps
// 104 and the block-cast output 128, so as not to spill.
// GC: the consumer threads per row when known at compile time (32, the
// common shape: slot offsets then fold into the instructions' immediates),
// or 0: p.G.  GC > 0 also promises that every shard row of every tensor
// fills all VPT x GC vector slots, so the slots need no range checks, and
// that gamma (and beta) are staged in the split layout.  BV:
// the E8M0 block-cast output's vectors per block when known at compile time
// (2, 4 or 8), or 0: p.bv.  NT: 1 when the launch has exactly one tensor
// (its parameters then need no indexing by the tile), or 0: p.ntensors.
template <int N, int VPT, int IN, int STAT, int OUT, int GC, int BV, int NT>
__global__ void __maxnreg__(STAT == kQkLn ? (VPT == 8 ? 104 : 96) : ((OUT != kOutBf16 && VPT == 8) ? 128 : 96))
    qknorm_cluster_kernel(const QkParams p) {
  constexpr int ES = (IN == kInBf16) ? 2 : 1;  // bytes per activation
  const int G = GC > 0 ? GC : p.G;
  constexpr bool kFull = GC > 0;   // nvec == VPT * G for every tensor
  constexpr int NS = (STAT == kQkLn) ? 2 : 1;  // scalars exchanged per warp
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t rank = (N > 1) ? cluster_ctarank() : 0u;
  const int64_t cid = cluster_id_x();
  const int64_t ncl = num_clusters_x();
  const int tid = threadIdx.x;
  const int nconsumer = p.R * G;
  const int lane = tid & 31;
  const int wpr = G >> 5;
  // block-cast output: vectors per block and log2 of the block size (NVFP4
  // blocks are 16 values: fixed at compile time)
  const int kBv = OUT == kOutNvfp4 ? 2 : (BV > 0 ? BV : p.bv);
  const int kBshift = OUT == kOutNvfp4 ? 4 : (BV == 2 ? 4 : BV == 4 ? 5 : BV == 8 ? 6 : p.bshift);
  const QkLayout L = qk_layout(N, p.S, p.R, p.Wmax, p.psum, G, p.gsplit, ES, NS,
                               OUT == kOutNvfp4);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t stage_bytes = (uint32_t)p.R * p.Wmax * ES;
  int64_t* tloc = reinterpret_cast<int64_t*>(smem + L.tloc);
  // Tile order: the first S tiles of every cluster are fixed (cid + n * ncl,
  // no start-up latency); later ones come from the launch's counter, taken
  // by the cluster's rank 0 and sent to every CTA of the cluster through a
  // ring of S + 1 slots.  Rank 0 writes the number of tile q only after its
  // consumers have finished tile q - S - 1 (they released the stage of
  // tile q - S, which they start only after tile q - S - 1's combine), and
  // that combine needed every peer's partial sums of the tile, so every peer
  // has read the number that the slot held.
  const bool dyn = p.sched != nullptr;

  if (tid == 0) {
    for (int s = 0; s < p.S; ++s) {
      mbar_init(sbase + L.full + 8 * s, 1);
      mbar_init(sbase + L.empty + 8 * s, nconsumer / 32);
      mbar_init(sbase + L.tbar + 8 * s, 1);
    }
    mbar_init(sbase + L.tbar + 8 * p.S, 1);
    for (int b = 0; b < 2 * p.R; ++b) mbar_init(sbase + L.xbar + 8 * b, 1);
    mbar_init(sbase + L.gbar, 1);
    mbar_init(sbase + L.gbar + 8, nconsumer / 32);   // gsync
    fence_mbar_init();
  }
  float* rcp = reinterpret_cast<float*>(smem + L.rcp);
  if (OUT == kOutNvfp4) fill_e4m3_reciprocals(rcp, tid, (int)blockDim.x);
  float2* lnc = reinterpret_cast<float2*>(smem + L.rcp);
  if (STAT == kQkLn) {
    for (int q = tid; q < 32; q += (int)blockDim.x) {
      const int k = q >> 4;
      lnc[q] = ln_count_pair(k < p.ntensors ? ln_warp_count<VPT>(p.ten[k].nvec, G, q & 15) : 0);
    }
  }
  __syncthreads();
  // everything above touched shared memory only
  grid_dependency_wait();
  allow_dependent_launch();

  if (tid >= nconsumer) {
    // ------------------------------------------------------ producer warp
    // It touches only this CTA's shared memory, so it starts the ring at
    // once; its half of the cluster start-up barrier is completed later.
    if (N > 1) cluster_arrive_relaxed();
    if (lane == 0) {
      bool aborted = false;
      // this shard's gamma (and beta) first (every CTA re-reads them, so no
      // evict hint)
      mbar_arrive_expect_tx(sbase + L.gbar, (uint32_t)p.psum * 4);
      for (int k = 0; k < p.ntensors; ++k) {
        const QkTensor& tk = p.ten[k];
        bulk_g2s_plain(sbase + tk.gam - L.gam + L.gstg, tk.gamma + (size_t)rank * tk.W,
                       (uint32_t)tk.W * 4, sbase + L.gbar);
        if (STAT == kQkLn && tk.beta != nullptr)
          bulk_g2s_plain(sbase + tk.bet - L.gam + L.gstg, tk.beta + (size_t)rank * tk.W,
                         (uint32_t)tk.W * 4, sbase + L.gbar);
      }
      const uint64_t policy = l2_policy_evict_first();
      // ring stage s of tile j and the parity of its pass, (j / S) & 1, kept
      // incrementally (no 64-bit division in the loop)
      int s = 0;
      uint32_t ph = 0;
      int64_t n = 0;      // tiles issued
      int kd = 0;         // tile-number slot of the next dynamic tile
      uint32_t pd = 0;    // its pass parity over the S + 1 slots
      while (true) {
        if (n >= p.S && !mbar_wait_bounded(sbase + L.empty + 8 * s, ph ^ 1u, p.wait_limit_ns)) {
          atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
          break;
        }
        int64_t tile;
        if (n < p.S || !dyn) {
          tile = cid + n * ncl;
        } else if (N == 1) {
          tile = ncl * p.S + (int64_t)atomicAdd(p.sched, 1u);
        } else {
          const uint32_t tb = sbase + L.tbar + 8 * kd;
          if (rank == 0) {
            // Every CTA of the cluster runs, its barriers initialised: this
            // is pass S or later, so the consumers released stage 0, which
            // they do only after the cluster start-up wait.
            const int64_t tk = ncl * p.S + (int64_t)atomicAdd(p.sched, 1u);
            const int64_t v = tk < p.ntiles ? tk : -1;
            const uint32_t slot = sbase + L.tile + 8 * kd;
#pragma unroll
            for (int k = 0; k < N; ++k)
              st_async_u64(map_to_rank(slot, k), (uint64_t)v, map_to_rank(tb, k));
          }
          mbar_arrive_expect_tx(tb, 8);
          if (!mbar_wait_bounded(tb, pd, p.wait_limit_ns)) {
            atomicOr(&g_qk_status, kStatusTimeout);
            aborted = true;
            break;
          }
          tile = *reinterpret_cast<volatile int64_t*>(smem + L.tile + 8 * kd);
          if (++kd == p.S + 1) {
            kd = 0;
            pd ^= 1u;
          }
        }
        const uint32_t bar = sbase + L.full + 8 * s;
        if (tile < 0 || tile >= p.ntiles) {
          tloc[s] = -1;   // published by the arrive (release) below
          mbar_arrive(bar);
          break;
        }
        tloc[s] = tile;
        int64_t t0;
        const QkTensor& tn = p.ten[NT == 1 ? 0 : qk_tile(p, tile, &t0)];
        if (NT == 1) t0 = tile * p.R;
        const int nrows = (int)min64(p.R, tn.T - t0);
        const uint32_t row_bytes = (uint32_t)tn.W * ES;
        const uint32_t dst = sbase + L.ring + (uint32_t)s * stage_bytes;
        const char* src = static_cast<const char*>(tn.X) +
                          ((size_t)t0 * tn.H + (size_t)rank * tn.W) * ES;
        mbar_arrive_expect_tx(bar, nrows * row_bytes + (n == 0 ? p.missing_tx : 0u));
        if (N == 1) {
          bulk_g2s(dst, src, nrows * row_bytes, bar, policy);
        } else {
          for (int r = 0; r < nrows; ++r)
            bulk_g2s(dst + r * row_bytes, src + (size_t)r * tn.H * ES, row_bytes, bar, policy);
        }
        ++n;
        if (++s == p.S) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Normally the consumers have waited for every copy before the CTA can
      // retire; after an expired wait, let the copies in flight land first.
      for (int64_t j = max64(0, n - p.S); j < n && aborted; ++j)
        (void)mbar_wait_bounded(sbase + L.full + 8 * (int)(j % p.S), (uint32_t)((j / p.S) & 1),
                                p.wait_limit_ns);
      (void)mbar_wait_bounded(sbase + L.gbar, 0, p.wait_limit_ns);
      // rank 0 counts its cluster out; the last re-arms the pair
      if (dyn && rank == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == (unsigned)(ncl - 1)) {
          atomicExch(p.sched, 0u);
          atomicExch(p.sched + 1, 0u);
        }
      }
    }
    __syncwarp();
    if (N > 1) cluster_wait_acquire();
  } else {
    // ------------------------------------------------------- consumer warps
    // Every CTA of the cluster must be running, with its barriers
    // initialised, before anyone stores into a peer's shared memory: arrive
    // now, wait after the first tile's Phase A (its loads and Phase A
    // overlap the start-up).
    if (N > 1) cluster_arrive_release();
    bool started = (N == 1);
    bool have_gamma = false;

    const int row = tid / G;
    const int g = tid - row * G;
    const int wir = g >> 5;
    const bool exchange = (N > 1) || (wpr > 1);
    bool aborted = false;
    int s = 0;          // ring stage of the j-th tile
    uint32_t ph = 0;    // (j / S) & 1
    for (int64_t j = 0;; ++j) {
      // a warp leaves together: an expired wait on one lane ends all 32 (the
      // shuffles and barriers below need the whole warp)
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(sbase + L.full + 8 * s, ph, p.wait_limit_ns))) {
        if (lane == 0) atomicOr(&g_qk_status, kStatusTimeout);
        break;
      }
      const int64_t tile = *reinterpret_cast<volatile int64_t*>(tloc + s);
      if (tile < 0 || tile >= p.ntiles) break;   // no more tiles
      int64_t t0;
      const int tk = NT == 1 ? 0 : qk_tile(p, tile, &t0);   // tensor of the tile
      if (NT == 1) t0 = tile * p.R;
      const QkTensor& tn = p.ten[NT == 1 ? 0 : tk];
      const int64_t t = t0 + row;
      const bool valid = t < tn.T;
      const int nvec = kFull ? VPT * GC : tn.nvec;

      // ---- Phase A: this shard's sum of squares (and, for LayerNorm, its
      // sum) in fp32 packed pairs.  The values are converted once and kept
      // as fp32 pairs in w; independent accumulators keep chains short.
      uint64_t w[VPT][4];
      uint64_t acc[4] = {0, 0, 0, 0};  // {0.f, 0.f} each
      const unsigned char* srow =
          smem + L.ring + (uint32_t)s * stage_bytes + (uint32_t)row * tn.W * ES;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = i * G + g;
        // a row beyond T (last tile) reads stale shared memory when full: its
        // partial sums only reach its own, unstored, combine
        load_vector<IN>(srow, v, kFull || (valid && v < nvec), p.x_scale, w[i]);
        if (STAT != kQkLn) {
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[q] = f2_fma(w[i][q], w[i][q], acc[q]);
        }
      }
      // The cluster start-up wait comes before the stage goes back: rank 0's
      // producer sends tile numbers into the peers' shared memory only once
      // stage 0 is back (pass S and later), so they are running by then.
      if (!started) {
        cluster_wait_acquire();
        started = true;
      }
      // the stage's data is in registers: hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(sbase + L.empty + 8 * s);
      // RMSNorm: ss = this warp's sum of squares.  LayerNorm: ss = its sum,
      // s1 = its M2 about its own mean (ln_warp_stats)
      float ss, s1 = 0.f;
      if (STAT == kQkLn) {
        ln_warp_stats<VPT, kFull>(w, G, g, nvec, lnc[16 * tk + wir], &ss, &s1);
      } else {
        const uint64_t a01 = f2_add(acc[0], acc[1]), a23 = f2_add(acc[2], acc[3]);
        const uint64_t a = f2_add(a01, a23);
        ss = warp_sum(f2_lo(a) + f2_hi(a));
      }

      // ---- exchange: send this warp's partial to every shard of the row
      const int b = (int)(j & 1);
      const uint32_t xbar = sbase + L.xbar + 8 * (b * p.R + row);
      const uint32_t slot0 = sbase + L.part + 4 * NS * (uint32_t)((b * p.R + row) * N * wpr);
      if (exchange) {
        if (g == 0) mbar_arrive_expect_tx(xbar, (uint32_t)(N * wpr * 4 * NS));
        // lane k sends to rank k: the N stores leave in one instruction
        if (lane < N) {
          const uint32_t slot = slot0 + 4 * NS * (rank * wpr + wir);
          if (STAT == kQkLn)
            st_async_f32x2(map_to_rank(slot, lane), ss, s1, map_to_rank(xbar, lane));
          else
            st_async_f32(map_to_rank(slot, lane), ss, map_to_rank(xbar, lane));
        }
      }

      // ---- Phase B (overlapping the exchange): w = x * gamma, in place
      // (RMSNorm; LayerNorm multiplies by gamma after centring, Phase C)
      if (!have_gamma) {
        // once: wait for the copied gamma and split it into the layout the
        // loop reads (consecutive lanes, consecutive 16 bytes)
        if (!mbar_wait_bounded(sbase + L.gbar, 0, aborted ? 0 : p.wait_limit_ns)) {
          if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
        }
        for (int k = 0; k < p.ntensors && p.gsplit; ++k) {
          const QkTensor& tk = p.ten[k];
          for (int par = 0; par < ((STAT == kQkLn && tk.beta != nullptr) ? 2 : 1); ++par) {
            const uint32_t off = par ? tk.bet : tk.gam;
            const float4* src = reinterpret_cast<const float4*>(smem + off - L.gam + L.gstg);
            float4* dst = reinterpret_cast<float4*>(smem + off);
            for (int q = tid; q < tk.nvec; q += nconsumer) {
              dst[q] = src[2 * q];
              dst[tk.nvec + q] = src[2 * q + 1];
            }
          }
        }
        // every consumer warp's share is written (a bounded wait, unlike a
        // named barrier: a warp that left on an expired wait cannot hang it)
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + L.gbar + 8);
        if (!mbar_wait_bounded(sbase + L.gbar + 8, 0, aborted ? 0 : p.wait_limit_ns)) {
          if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
        }
        have_gamma = true;
      }
      // split layout: halves nvec*16 bytes apart, vectors 16 apart; as
      // copied: halves 16 apart, vectors 32 apart
      // (the GC = 32 kernels always have the split layout)
      const bool gsplit = kFull || p.gsplit;
      const unsigned char* gam_lo = smem + tn.gam;
      const unsigned char* gam_hi = gam_lo + (gsplit ? (uint32_t)nvec * 16 : 16u);
      const uint32_t gstride = gsplit ? 16u : 32u;
#pragma unroll
      for (int i = 0; i < VPT && STAT != kQkLn; ++i) {
        const int v = kFull ? i * G + g : min(i * G + g, nvec - 1);
        const uint4 glo = lds128(gam_lo + v * gstride);
        const uint4 ghi = lds128(gam_hi + v * gstride);
        w[i][0] = f2_mul(w[i][0], f2(__uint_as_float(glo.x), __uint_as_float(glo.y)));
        w[i][1] = f2_mul(w[i][1], f2(__uint_as_float(glo.z), __uint_as_float(glo.w)));
        w[i][2] = f2_mul(w[i][2], f2(__uint_as_float(ghi.x), __uint_as_float(ghi.y)));
        w[i][3] = f2_mul(w[i][3], f2(__uint_as_float(ghi.z), __uint_as_float(ghi.w)));
      }
      // block-cast output: each block's absmax of x*gamma, still before the
      // combine (a block is bv consecutive vectors, i.e. bv adjacent lanes)
      float am[OUT != kOutBf16 ? VPT : 1];
      if (OUT != kOutBf16) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          float m = absmax8(0.f, w[i]);
          // bv = B/8 is 2, 4 or 8: at most three steps, unrolled and guarded
          // by the (warp-uniform) block size; NVFP4 blocks are always 16
#pragma unroll
          for (int o = 1; o < 8; o <<= 1)
            if (o < kBv) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
          am[i] = m;
        }
      }

      // ---- combine in rank order (then warp order within a shard)
      float S = ss, mu = 0.f, var = 0.f;
      if (exchange) {
        if (!mbar_wait_bounded(xbar, (uint32_t)((j >> 1) & 1), aborted ? 0 : p.wait_limit_ns)) {
          if (!aborted) atomicOr(&g_qk_status, kStatusTimeout);
          aborted = true;
        }
        const float* sl = reinterpret_cast<const float*>(smem + (slot0 - sbase));
        if (STAT == kQkLn) {
          ln_combine(sl, N, wpr, [&](int w) { return lnc[16 * tk + w]; }, tn.inv_H, &mu, &var);
        } else {
          S = 0.f;
          for (int k = 0; k < N * wpr; ++k) S += sl[k];
        }
      } else if (STAT == kQkLn) {
        const float own[2] = {ss, s1};
        ln_combine(own, 1, 1, [&](int w) { return lnc[16 * tk + w]; }, tn.inv_H, &mu, &var);
      }

      // ---- Phase C: scale (and for LayerNorm centre and shift), store
      if (valid) {
        float rinv;
        if (STAT == kQkLn) {
          rinv = rsqrtf(var + p.eps);
        } else {
          // the hardware reciprocal square root (a few 1e-8 relative error)
          rinv = rsqrtf(fmaf(S, tn.inv_H, p.eps));
        }
        const uint64_t rr = f2(rinv, rinv);
        const float nmr = -mu * rinv;
        __nv_bfloat16* yrow = tn.Y + (size_t)t * tn.H + (size_t)rank * tn.W;
        // block-cast output: this shard's codes and scales of row t
        uint8_t* crow = nullptr;
        uint8_t* srow_sc = nullptr;
        int vshift = 0;   // vector -> block: v >> vshift
        if (OUT != kOutBf16) {
          const size_t first = (size_t)t * tn.H + (size_t)rank * tn.W;  // element index
          crow = OUT == kOutE4M3 ? tn.codes + first : tn.codes + first / 2;
          srow_sc = tn.scales + (first >> kBshift);
          vshift = kBshift - 3;
        }
        // Block scales spread over the lanes of a block (B/8 adjacent lanes
        // hold a block's vectors and, after the shuffles above, its absmax):
        // lane r of the group forms the scales of the slots r, r + B/8, ...,
        // stores their scale bytes (one store per round serves 32 blocks)
        // and hands each slot's multiplier to the others by one shuffle.
        constexpr int kBvC = OUT == kOutNvfp4 ? 2 : (BV > 0 ? BV : 1);
        constexpr bool kDist = kFull && OUT != kOutBf16 && (OUT == kOutNvfp4 || BV > 0);
        constexpr int kRounds = kDist ? (VPT + kBvC - 1) / kBvC : 1;
        float isd[kRounds];
        if (kDist) {
          constexpr int kGroupShift = kBvC == 2 ? 1 : kBvC == 4 ? 2 : 3;
          const int r = g & (kBvC - 1);
          const int grp = g >> kGroupShift;
#pragma unroll
          for (int j = 0; j < kRounds; ++j) {
            float a = am[j * kBvC];
#pragma unroll
            for (int q = 1; q < kBvC; ++q)
              if (j * kBvC + q < VPT) a = r == q ? am[j * kBvC + q] : a;
            const int sl = j * kBvC + r;   // this lane's slot
            float is;
            uint32_t sbyte;
            if (OUT == kOutNvfp4) {
              sbyte = nvfp4_scale(a * rinv, rcp, &is);
            } else {
              sbyte = (uint32_t)(e8m0_exponent(a * rinv, OUT == kOutE4M3 ? 8 : 2) + 127);
              is = __uint_as_float((254u - sbyte) << 23);
            }
            if (sl < VPT) srow_sc[sl * (32 / kBvC) + grp] = (uint8_t)sbyte;
            isd[j] = is;
          }
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = i * G + g;
          if (OUT != kOutBf16) {
            if (kFull || v < nvec) {
              // scale of this vector's block, then its eight codes
              float is;
              uint32_t keep = ~0u, sbyte;
              if (kDist) {
                // the multiplier from the lane that formed it (NVFP4: a zero
                // scale has the multiplier 0)
                is = __shfl_sync(0xFFFFFFFFu, isd[i / kBvC], (lane & ~(kBvC - 1)) | (i % kBvC));
                if (OUT == kOutNvfp4) keep = is != 0.f ? ~0u : 0u;
              } else {
                if (OUT == kOutNvfp4) {
                  sbyte = nvfp4_scale(am[i] * rinv, rcp, &is);
                  keep = sbyte != 0 ? ~0u : 0u;
                } else {
                  sbyte = (uint32_t)(e8m0_exponent(am[i] * rinv, OUT == kOutE4M3 ? 8 : 2) + 127);
                  is = __uint_as_float((254u - sbyte) << 23);  // 2^-e, e = sbyte - 127
                }
                if ((g & (kBv - 1)) == 0) srow_sc[v >> vshift] = (uint8_t)sbyte;
              }
              // q = fp32(fp32(w * rinv) * s), s = 2^-e or fp32(1/scale): the
              // two products of the definition, with no per-vector choice
              // (measured on GB300: the one-product form's per-vector
              // bound check and branch cost more than the product it saves)
              uint64_t q[4];
              const uint64_t ss = f2(is, is);
#pragma unroll
              for (int h = 0; h < 4; ++h) q[h] = f2_mul(f2_mul(w[i][h], rr), ss);
              if (OUT == kOutE4M3) {
                const uint32_t lo = cvt_e4m3x4(f2_lo(q[0]), f2_hi(q[0]), f2_lo(q[1]), f2_hi(q[1]));
                const uint32_t hi = cvt_e4m3x4(f2_lo(q[2]), f2_hi(q[2]), f2_lo(q[3]), f2_hi(q[3]));
                st_global_v2(crow + 8 * v, lo, hi);
              } else {
                const uint32_t c = cvt_e2m1x8(f2_lo(q[0]), f2_hi(q[0]), f2_lo(q[1]), f2_hi(q[1]),
                                              f2_lo(q[2]), f2_hi(q[2]), f2_lo(q[3]), f2_hi(q[3]));
                st_global_u32(crow + 4 * v, c & keep);
              }
            }
            continue;
          }
          if (kFull || v < nvec) {
            uint4 o;
            uint64_t y0, y1, y2, y3;
            if (STAT == kQkLn) {
              // y = (x rinv - mu rinv) gamma + beta  (w still holds x)
              const uint4 glo = lds128(gam_lo + v * gstride);
              const uint4 ghi = lds128(gam_hi + v * gstride);
              uint4 blo = make_uint4(0, 0, 0, 0), bhi = make_uint4(0, 0, 0, 0);
              if (tn.beta != nullptr) {
                const unsigned char* bet_lo = smem + tn.bet;
                const unsigned char* bet_hi = bet_lo + (gsplit ? (uint32_t)nvec * 16 : 16u);
                blo = lds128(bet_lo + v * gstride);
                bhi = lds128(bet_hi + v * gstride);
              }
              const uint64_t m2 = f2(nmr, nmr);
              y0 = f2_fma(f2_fma(w[i][0], rr, m2), f2(__uint_as_float(glo.x), __uint_as_float(glo.y)),
                          f2(__uint_as_float(blo.x), __uint_as_float(blo.y)));
              y1 = f2_fma(f2_fma(w[i][1], rr, m2), f2(__uint_as_float(glo.z), __uint_as_float(glo.w)),
                          f2(__uint_as_float(blo.z), __uint_as_float(blo.w)));
              y2 = f2_fma(f2_fma(w[i][2], rr, m2), f2(__uint_as_float(ghi.x), __uint_as_float(ghi.y)),
                          f2(__uint_as_float(bhi.x), __uint_as_float(bhi.y)));
              y3 = f2_fma(f2_fma(w[i][3], rr, m2), f2(__uint_as_float(ghi.z), __uint_as_float(ghi.w)),
                          f2(__uint_as_float(bhi.z), __uint_as_float(bhi.w)));
            } else {
              y0 = f2_mul(w[i][0], rr);
              y1 = f2_mul(w[i][1], rr);
              y2 = f2_mul(w[i][2], rr);
              y3 = f2_mul(w[i][3], rr);
            }
            o.x = pack_bf16x2_rn(f2_lo(y0), f2_hi(y0));
            o.y = pack_bf16x2_rn(f2_lo(y1), f2_hi(y1));
            o.z = pack_bf16x2_rn(f2_lo(y2), f2_hi(y2));
            o.w = pack_bf16x2_rn(f2_lo(y3), f2_hi(y3));
            st_global_v4_stream(yrow + v * 8, o);
          }
        }
        if (tn.rinv_out != nullptr && rank == 0 && g == 0) tn.rinv_out[t] = rinv;
        if (STAT == kQkLn && tn.mean_out != nullptr && rank == 0 && g == 0) tn.mean_out[t] = mu;
      }
      if (aborted) break;
      if (++s == p.S) {
        s = 0;
        ph ^= 1u;
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

using QkKernel = void (*)(QkParams);

template <int N, int IN, int STAT, int OUT, int GC, int BV, int NT>
QkKernel pick_qk_vpt(int vpt) {
  switch (vpt) {
    case 1: return qknorm_cluster_kernel<N, 1, IN, STAT, OUT, GC, BV, NT>;
    case 2: return qknorm_cluster_kernel<N, 2, IN, STAT, OUT, GC, BV, NT>;
    case 3: return qknorm_cluster_kernel<N, 3, IN, STAT, OUT, GC, BV, NT>;
    case 4: return qknorm_cluster_kernel<N, 4, IN, STAT, OUT, GC, BV, NT>;
    case 5: return qknorm_cluster_kernel<N, 5, IN, STAT, OUT, GC, BV, NT>;
    case 6: return qknorm_cluster_kernel<N, 6, IN, STAT, OUT, GC, BV, NT>;
    case 8: return qknorm_cluster_kernel<N, 8, IN, STAT, OUT, GC, BV, NT>;
    default: return nullptr;
  }
}

// One-warp shard rows that fill their slots (G = 32: the launcher passes 32
// only then) take the kernels with G, and for the E8M0 block-cast outputs
// the block size, fixed at compile time; other shapes read both from the
// parameters.  Launches of one tensor (nt = 1) take the kernels without
// per-tile tensor indexing where that was measured to pay (block-cast
// outputs: 4 %; LayerNorm, E4M3 input: 2 %; bf16 output: none) -- the
// E8M0 outputs for 32-value blocks only, to bound the instantiations.
template <int N, int IN, int STAT, int OUT>
QkKernel pick_qk_rows(int vpt, int G, int bv, int nt) {
  if (G == 32) {
    if constexpr (OUT == kOutE4M3 || OUT == kOutE2M1) {
      switch (bv) {
        case 2: return pick_qk_vpt<N, IN, STAT, OUT, 32, 2, 0>(vpt);
        case 4: return nt == 1 ? pick_qk_vpt<N, IN, STAT, OUT, 32, 4, 1>(vpt)
                               : pick_qk_vpt<N, IN, STAT, OUT, 32, 4, 0>(vpt);
        case 8: return pick_qk_vpt<N, IN, STAT, OUT, 32, 8, 0>(vpt);
        default: return nullptr;
      }
    } else if constexpr (OUT == kOutNvfp4) {
      return nt == 1 ? pick_qk_vpt<N, IN, STAT, OUT, 32, 0, 1>(vpt)
                     : pick_qk_vpt<N, IN, STAT, OUT, 32, 0, 0>(vpt);
    } else if constexpr (STAT == kQkLn || IN != kInBf16) {
      // no entry point launches two such tensors at once
      if (nt == 1) return pick_qk_vpt<N, IN, STAT, OUT, 32, 0, 1>(vpt);
    } else {
      return pick_qk_vpt<N, IN, STAT, OUT, 32, 0, 0>(vpt);
    }
  }
  return pick_qk_vpt<N, IN, STAT, OUT, 0, 0, 0>(vpt);
}

// Instantiates every QK kernel for input type IN, statistic STAT and output
// OUT in the calling unit; G = consumer threads per row, bv = 16-byte
// vectors per block of the block-cast output, nt = tensors of the launch.
template <int IN, int STAT, int OUT = kOutBf16>
QkKernel pick_qk_input(int N, int vpt, int G, int bv, int nt) {
  switch (N) {
    case 1: return pick_qk_rows<1, IN, STAT, OUT>(vpt, G, bv, nt);
    case 2: return pick_qk_rows<2, IN, STAT, OUT>(vpt, G, bv, nt);
    case 4: return pick_qk_rows<4, IN, STAT, OUT>(vpt, G, bv, nt);
    case 8: return pick_qk_rows<8, IN, STAT, OUT>(vpt, G, bv, nt);
    default: return nullptr;
  }
}

static inline int read_and_clear_local_qk_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qk_status, sizeof(v));
  if (e != cudaSuccess) return fail_cuda(e, "reading a QK status word");
  e = cudaMemcpyToSymbol(g_qk_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clearing a QK status word");
  *out = v;
  return NTS_OK;
}

// The single-tile kernel for decode-sized launches (qk_direct.cu).
QkKernel pick_qk_direct(int N, int vpt, int in_e4m3, int layernorm);

// Defined by qk_bf16.cu, qk_e4m3.cu, qk_ln.cu and qk_mx_*.cu.
QkKernel pick_qk_bf16(int N, int vpt, int G, int bv, int nt);
QkKernel pick_qk_e4m3(int N, int vpt, int G, int bv, int nt);
QkKernel pick_qk_ln(int N, int vpt, int G, int bv, int nt);
QkKernel pick_qk_mx_e4m3(int N, int vpt, int G, int bv, int nt);
QkKernel pick_qk_mx_e2m1(int N, int vpt, int G, int bv, int nt);
QkKernel pick_qk_mx_nvfp4(int N, int vpt, int G, int bv, int nt);
int read_and_clear_qk_bf16_status(unsigned* out);
int read_and_clear_qk_e4m3_status(unsigned* out);
int read_and_clear_qk_ln_status(unsigned* out);
int read_and_clear_qk_mx_e4m3_status(unsigned* out);
int read_and_clear_qk_mx_e2m1_status(unsigned* out);
int read_and_clear_qk_mx_nvfp4_status(unsigned* out);

}  // namespace nts
