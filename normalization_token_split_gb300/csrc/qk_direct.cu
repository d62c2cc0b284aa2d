// qk_direct.cu -- the split-H QK-RMSNorm for launches with at most one tile
// per cluster (decode-sized token counts), where latency, not bandwidth,
// sets the time.
//
// Same method and arithmetic as the persistent kernel (qk_kernel.cuh):
// Phase A sums squares per shard in fp32, the partial sums cross the
// cluster through distributed shared memory and are added in rank order,
// Phase C writes (x*gamma)*rinv once.  What it leaves out is everything a
// single tile does not need: no producer warp, no TMA ring, no mbarriers and
// no gamma staging.  Every thread issues the global loads of its x and gamma
// vectors at the very start, so their latency overlaps the cluster start-up
// barrier; one more cluster barrier orders the partial sums.  The summation
// order is the persistent kernel's, so the results are identical bit for bit.
#include <cuda_runtime.h>

#include "nts_device.cuh"
#include "nts_internal.h"
#include "qk_kernel.cuh"

namespace nts {

namespace {

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One tile of R rows per cluster; blockDim = R * G; dynamic shared memory:
// part[R][N][WPR] f32, the partial sums of every warp of every shard.
template <int N, int VPT>
__global__ void __launch_bounds__(kMaxThreads, 1) qk_direct_kernel(const QkParams p) {
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

  int64_t t0;
  const QkTensor& tn = p.ten[qk_tile(p, tile, &t0)];
  const int64_t t = t0 + row;
  const bool valid = t < tn.T;
  const int nvec = tn.nvec;
  const __nv_bfloat16* xrow =
      static_cast<const __nv_bfloat16*>(tn.X) + (size_t)t * tn.H + (size_t)rank * tn.W;
  const float* grow = tn.gamma + (size_t)rank * tn.W;

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
      if (valid) xv[i] = ldg_nc_v4(xrow + v * 8);
      g0[i] = __ldg(reinterpret_cast<const float4*>(grow + v * 8));
      g1[i] = __ldg(reinterpret_cast<const float4*>(grow + v * 8) + 1);
    }
  }

  // Phase A, in the persistent kernel's order
  uint64_t w[VPT][4];
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    w[i][0] = bf16x2_to_f2(xv[i].x);
    w[i][1] = bf16x2_to_f2(xv[i].y);
    w[i][2] = bf16x2_to_f2(xv[i].z);
    w[i][3] = bf16x2_to_f2(xv[i].w);
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = f2_fma(w[i][q], w[i][q], acc[q]);
  }
  const uint64_t a = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  const float ss = warp_sum(f2_lo(a) + f2_hi(a));

  // Phase B: w = x * gamma
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    w[i][0] = f2_mul(w[i][0], f2(g0[i].x, g0[i].y));
    w[i][1] = f2_mul(w[i][1], f2(g0[i].z, g0[i].w));
    w[i][2] = f2_mul(w[i][2], f2(g1[i].x, g1[i].y));
    w[i][3] = f2_mul(w[i][3], f2(g1[i].z, g1[i].w));
  }

  // exchange: slot [row][rank][warp] of every CTA of the cluster
  float S = ss;
  if (N > 1 || wpr > 1) {
    float* slots = part + (size_t)row * N * wpr;
    if (N > 1) {
      cluster_wait_acquire();
      if (lane == 0) {
        const uint32_t slot = smem_addr(slots + rank * wpr + wir);
#pragma unroll
        for (int k = 0; k < N; ++k) st_cluster_f32(map_to_rank(slot, k), ss);
      }
      __syncwarp();
      cluster_arrive_release();
      cluster_wait_acquire();
    } else {
      if (lane == 0) slots[wir] = ss;
      __syncthreads();
    }
    S = 0.f;
    for (int k = 0; k < N * wpr; ++k) S += slots[k];
  }

  // Phase C
  if (valid) {
    const float rinv = rsqrtf(fmaf(S, tn.inv_H, p.eps));
    const uint64_t rr = f2(rinv, rinv);
    __nv_bfloat16* yrow = tn.Y + (size_t)t * tn.H + (size_t)rank * tn.W;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = i * p.G + g;
      if (v < nvec) {
        const uint64_t y0 = f2_mul(w[i][0], rr), y1 = f2_mul(w[i][1], rr);
        const uint64_t y2 = f2_mul(w[i][2], rr), y3 = f2_mul(w[i][3], rr);
        uint4 o;
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

template <int N>
QkKernel pick_direct_vpt(int vpt) {
  switch (vpt) {
    case 1: return qk_direct_kernel<N, 1>;
    case 2: return qk_direct_kernel<N, 2>;
    case 3: return qk_direct_kernel<N, 3>;
    case 4: return qk_direct_kernel<N, 4>;
    case 5: return qk_direct_kernel<N, 5>;
    default: return nullptr;  // wider rows keep the persistent kernel (registers)
  }
}

}  // namespace

QkKernel pick_qk_direct(int N, int vpt) {
  switch (N) {
    case 1: return pick_direct_vpt<1>(vpt);
    case 2: return pick_direct_vpt<2>(vpt);
    case 4: return pick_direct_vpt<4>(vpt);
    case 8: return pick_direct_vpt<8>(vpt);
    default: return nullptr;
  }
}

}  // namespace nts
