// qk_direct.cu -- the split-H QK-RMSNorm (bf16 or E4M3 activations) and
// LayerNorm for launches with at most one tile per cluster (decode-sized
// token counts), where latency, not bandwidth, sets the time.
//
// Same method and arithmetic as the persistent kernel (qk_kernel.cuh):
// Phase A sums squares per shard in fp32, the partial sums cross the
// cluster through distributed shared memory and are added in rank order,
// Phase C writes (x*gamma)*rinv once.  What it leaves out is everything a
// single tile does not need: no producer warp, no TMA ring, no mbarriers and
// no gamma staging.  Every thread issues the global loads of its x and gamma
// vectors at the very start (after the dependent-launch wait), so their
// latency overlaps the cluster start-up barrier; one more cluster barrier orders the partial sums.  The summation
// order is the persistent kernel's, so the results are identical bit for bit.
#include <cuda_runtime.h>

#include "nts_device.cuh"
#include "nts_internal.h"
#include "qk_kernel.cuh"

namespace nts {

namespace {

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One tile of R rows per cluster; blockDim = R * G; dynamic shared memory:
// part[R][N][WPR][NS] f32, the partial sums of every warp of every shard
// (NS = 1 for RMSNorm, 2 for LayerNorm: sum of squares and sum).
template <int N, int VPT, int IN, int STAT>
__global__ void __launch_bounds__(kMaxThreads, 1) qk_direct_kernel(const QkParams p) {
  constexpr int ES = (IN == kInBf16) ? 2 : 1;
  constexpr int NS = (STAT == kQkLn) ? 2 : 1;
  extern __shared__ __align__(16) float part[];
  const uint32_t rank = (N > 1) ? cluster_ctarank() : 0u;
  const int64_t tile = (N > 1) ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int wpr = p.G >> 5;
  const int row = tid / p.G;
  const int g = tid - row * p.G;
  const int wir = g >> 5;
  if (N > 1) cluster_arrive_relaxed();  // start-up: peers must run before DSMEM stores
  grid_dependency_wait();               // no global access before this
  allow_dependent_launch();

  int64_t t0;
  const QkTensor& tn = p.ten[qk_tile(p, tile, &t0)];
  const int64_t t = t0 + row;
  const bool valid = t < tn.T;
  const int nvec = tn.nvec;
  const unsigned char* xrow = static_cast<const unsigned char*>(tn.X) +
                              ((size_t)t * tn.H + (size_t)rank * tn.W) * ES;
  const float* grow = tn.gamma + (size_t)rank * tn.W;
  const float* brow = (STAT == kQkLn && tn.beta != nullptr) ? tn.beta + (size_t)rank * tn.W
                                                           : nullptr;

  // every load first
  uint4 xv[VPT];
  float4 g0[VPT], g1[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = i * p.G + g;
    xv[i] = make_uint4(0, 0, 0, 0);
    g0[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    g1[i] = g0[i];
    if (v < nvec) {
      if (valid) {
        if (IN == kInBf16) {
          xv[i] = ldg_nc_v4(xrow + v * 16);
        } else {
          const uint2 c = ldg_nc_v2(xrow + v * 8);
          xv[i].x = c.x;
          xv[i].y = c.y;
        }
      }
      g0[i] = __ldg(reinterpret_cast<const float4*>(grow + v * 8));
      g1[i] = __ldg(reinterpret_cast<const float4*>(grow + v * 8) + 1);
    }
  }

  // Phase A, in the persistent kernel's order
  uint64_t w[VPT][4];
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (IN == kInBf16) {
      w[i][0] = bf16x2_to_f2(xv[i].x);
      w[i][1] = bf16x2_to_f2(xv[i].y);
      w[i][2] = bf16x2_to_f2(xv[i].z);
      w[i][3] = bf16x2_to_f2(xv[i].w);
    } else {
      const uint64_t sc = f2(p.x_scale, p.x_scale);
      w[i][0] = f2_mul(e4m3x2_to_f2((uint16_t)(xv[i].x & 0xFFFFu)), sc);
      w[i][1] = f2_mul(e4m3x2_to_f2((uint16_t)(xv[i].x >> 16)), sc);
      w[i][2] = f2_mul(e4m3x2_to_f2((uint16_t)(xv[i].y & 0xFFFFu)), sc);
      w[i][3] = f2_mul(e4m3x2_to_f2((uint16_t)(xv[i].y >> 16)), sc);
    }
    if (STAT != kQkLn) {
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = f2_fma(w[i][q], w[i][q], acc[q]);
    }
  }
  // RMSNorm: ss = this warp's sum of squares.  LayerNorm: ss = its sum, s1 =
  // its M2 about its own mean
  float ss, s1 = 0.f;
  // LayerNorm counts: computed here as the persistent kernel tabulates them
  auto cnt = [&](int wi) { return ln_count_pair(ln_warp_count<VPT>(nvec, p.G, wi)); };
  if (STAT == kQkLn) {
    ln_warp_stats<VPT, false>(w, p.G, g, nvec, cnt(wir), &ss, &s1);
  } else {
    const uint64_t a = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
    ss = warp_sum(f2_lo(a) + f2_hi(a));
  }

  // Phase B: w = x * gamma (RMSNorm; LayerNorm multiplies after centring)
#pragma unroll
  for (int i = 0; i < VPT && STAT != kQkLn; ++i) {
    w[i][0] = f2_mul(w[i][0], f2(g0[i].x, g0[i].y));
    w[i][1] = f2_mul(w[i][1], f2(g0[i].z, g0[i].w));
    w[i][2] = f2_mul(w[i][2], f2(g1[i].x, g1[i].y));
    w[i][3] = f2_mul(w[i][3], f2(g1[i].z, g1[i].w));
  }

  // exchange: slot [row][rank][warp] of every CTA of the cluster
  float S = ss, mu = 0.f, var = 0.f;
  if (N > 1 || wpr > 1) {
    float* slots = part + (size_t)row * N * wpr * NS;
    if (N > 1) {
      cluster_wait_acquire();
      if (lane < N) {   // lane k stores into rank k
        const uint32_t slot = smem_addr(slots + NS * (rank * wpr + wir));
        st_cluster_f32(map_to_rank(slot, lane), ss);
        if (STAT == kQkLn) st_cluster_f32(map_to_rank(slot + 4, lane), s1);
      }
      __syncwarp();
      cluster_arrive_release();
      cluster_wait_acquire();
    } else {
      if (lane == 0) {
        slots[NS * wir] = ss;
        if (STAT == kQkLn) slots[NS * wir + 1] = s1;
      }
      __syncthreads();
    }
    if (STAT == kQkLn) {
      ln_combine(slots, N, wpr, cnt, tn.inv_H, &mu, &var);
    } else {
      S = 0.f;
      for (int k = 0; k < N * wpr; ++k) S += slots[k];
    }
  } else if (STAT == kQkLn) {
    const float own[2] = {ss, s1};
    ln_combine(own, 1, 1, cnt, tn.inv_H, &mu, &var);
  }

  // Phase C
  if (valid) {
    float rinv;
    if (STAT == kQkLn) {
      rinv = rsqrtf(var + p.eps);
    } else {
      rinv = rsqrtf(fmaf(S, tn.inv_H, p.eps));
    }
    const uint64_t rr = f2(rinv, rinv);
    const float nmr = -mu * rinv;
    __nv_bfloat16* yrow = tn.Y + (size_t)t * tn.H + (size_t)rank * tn.W;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = i * p.G + g;
      if (v < nvec) {
        uint64_t y0, y1, y2, y3;
        if (STAT == kQkLn) {
          float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
          if (brow != nullptr) {
            b0 = __ldg(reinterpret_cast<const float4*>(brow + v * 8));
            b1 = __ldg(reinterpret_cast<const float4*>(brow + v * 8) + 1);
          }
          // y = (x rinv - mu rinv) gamma + beta  (w still holds x)
          const uint64_t m2 = f2(nmr, nmr);
          y0 = f2_fma(f2_fma(w[i][0], rr, m2), f2(g0[i].x, g0[i].y), f2(b0.x, b0.y));
          y1 = f2_fma(f2_fma(w[i][1], rr, m2), f2(g0[i].z, g0[i].w), f2(b0.z, b0.w));
          y2 = f2_fma(f2_fma(w[i][2], rr, m2), f2(g1[i].x, g1[i].y), f2(b1.x, b1.y));
          y3 = f2_fma(f2_fma(w[i][3], rr, m2), f2(g1[i].z, g1[i].w), f2(b1.z, b1.w));
        } else {
          y0 = f2_mul(w[i][0], rr);
          y1 = f2_mul(w[i][1], rr);
          y2 = f2_mul(w[i][2], rr);
          y3 = f2_mul(w[i][3], rr);
        }
        uint4 o;
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
}

template <int N, int IN, int STAT>
QkKernel pick_direct_vpt(int vpt) {
  switch (vpt) {
    case 1: return qk_direct_kernel<N, 1, IN, STAT>;
    case 2: return qk_direct_kernel<N, 2, IN, STAT>;
    case 3: return qk_direct_kernel<N, 3, IN, STAT>;
    case 4: return qk_direct_kernel<N, 4, IN, STAT>;
    case 5: return qk_direct_kernel<N, 5, IN, STAT>;
    default: return nullptr;  // wider rows keep the persistent kernel (registers)
  }
}

template <int IN, int STAT>
QkKernel pick_direct_n(int N, int vpt) {
  switch (N) {
    case 1: return pick_direct_vpt<1, IN, STAT>(vpt);
    case 2: return pick_direct_vpt<2, IN, STAT>(vpt);
    case 4: return pick_direct_vpt<4, IN, STAT>(vpt);
    case 8: return pick_direct_vpt<8, IN, STAT>(vpt);
    default: return nullptr;
  }
}

}  // namespace

QkKernel pick_qk_direct(int N, int vpt, int in_e4m3, int layernorm) {
  if (layernorm) return in_e4m3 ? nullptr : pick_direct_n<kInBf16, kQkLn>(N, vpt);
  return in_e4m3 ? pick_direct_n<kInE4M3, kQkRms>(N, vpt) : pick_direct_n<kInBf16, kQkRms>(N, vpt);
}

}  // namespace nts
