// mx_norm_cast.cu -- fused per-token normalization + MX block cast on one
// GB300: RMSNorm + MXCast, and MXNorm + MXCast (p = 1 or 2).
//
// Method (MXNorm paper card, abstract, Fig. 1 caption and Fig. A.1):
//   a row of D values is cut into K = D/B blocks of B contiguous values; each
//   block is stored as B element codes (E4M3 or E2M1) sharing one E8M0 scale
//   2^round(log2(normalized absmax / 2^emax)).  RMSNorm + MXCast takes the
//   RMS from sum x^2 over the row; MXNorm estimates it from the block
//   absmaxes the cast computes anyway, rho~ = c(B,p) * M_p(absmax), a
//   reduction B times smaller.  Both are fused into one kernel (Fig. 8).
//
// GB300 mapping:
//  * a persistent grid of CTAs walks tiles of R whole rows; one thread keeps
//    a ring of S shared-memory stages filled with 1-D bulk TMA copies (rows
//    are contiguous, so one copy per tile), S-1 tiles ahead;
//  * G threads share a row (whole warps), each owning VPT 16-byte vectors of
//    8 values: a block of B values spans B/8 consecutive lanes, so its absmax
//    is a 1-3 step xor-shuffle and the element codes of a warp form one
//    coalesced 256- or 128-byte store;
//  * the row statistic is a warp shuffle reduction plus one CTA barrier;
//  * the E8M0 exponent is integer arithmetic on the fp32 absmax bits, and the
//    element cast is the hardware cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32.
#include <cuda_runtime.h>

#include <algorithm>

#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

__device__ unsigned int g_mx_status;  // kStatusTimeout bits, read by nts_check_status

struct MxParams {
  const __nv_bfloat16* X;
  const float* gamma;   // nullable
  uint8_t* codes;
  uint8_t* scales;
  float* rinv_out;      // nullable
  float* amax_out;      // nullable
  int64_t T;
  int64_t ntiles;
  int D;
  int nvec;             // D / 8
  int G;                // threads per row (multiple of 32)
  int R;                // rows per tile
  int S;                // ring stages
  int K;                // D / B blocks per row
  int gl;               // lanes per block, B / 8 (2, 4 or 8)
  float eps;
  float corr;           // MXNorm: c(B,1) for p = 1, c(B,2)^2 for p = 2
  uint64_t wait_limit_ns;
  uint32_t missing_tx;  // test hook: bytes expected on the first stage but never sent
};

enum { kStatRms = 0, kStatMxP1 = 1, kStatMxP2 = 2 };

// Shared memory: ring[S][R][D] bf16 | full[S] mbarriers | red[2][R][WPR] f32.
__host__ __device__ inline size_t mx_smem_bytes(int S, int R, int D, int G) {
  return (size_t)S * R * D * 2 + (size_t)S * 8 + (size_t)2 * R * (G / 32) * 4;
}

// E8M0 exponent of a block whose normalized absmax is `ay` (>= 0):
// round(log2 ay) - emax, where the log2 rounding goes up exactly when the
// fp32 significand is >= the first fp32 value above sqrt(2) (0x3504F4 in the
// mantissa field); zero and subnormal absmaxes give the smallest scale.
__device__ __forceinline__ int e8m0_exponent(float ay, int emax) {
  const uint32_t b = __float_as_uint(ay);
  const int field = (int)(b >> 23);
  if (field == 0) return -127;
  const int e = field - 127 + ((b & 0x7FFFFFu) >= 0x3504F4u ? 1 : 0) - emax;
  return max(-127, min(127, e));
}

template <int VPT, int FMT, int STAT>
__global__ void __launch_bounds__(kMaxThreads, 1) mx_norm_cast_kernel(const MxParams p) {
  constexpr int kEmax = (FMT == NTS_FMT_E4M3) ? 8 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int row = tid / p.G;
  const int g = tid - row * p.G;
  const int wpr = p.G >> 5;
  const int wir = g >> 5;
  const int lane = tid & 31;
  const bool leader = (g & (p.gl - 1)) == 0;

  const uint32_t stage_bytes = (uint32_t)p.R * p.D * 2;
  const uint32_t ring = smem_addr(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.S * stage_bytes);
  float* red = reinterpret_cast<float*>(full + p.S);

  const int64_t cta = blockIdx.x, ncta = gridDim.x;
  const int64_t my_tiles = cta < p.ntiles ? (p.ntiles - 1 - cta) / ncta + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < p.S; ++s) mbar_init(smem_addr(&full[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int64_t j) {
    const int64_t t0 = (cta + j * ncta) * p.R;
    const int nrows = (int)min64(p.R, p.T - t0);
    const int s = (int)(j % p.S);
    const uint32_t bar = smem_addr(&full[s]);
    const uint32_t bytes = (uint32_t)nrows * p.D * 2;
    mbar_arrive_expect_tx(bar, bytes + (j == 0 ? p.missing_tx : 0u));
    bulk_g2s(ring + (uint32_t)s * stage_bytes, p.X + (size_t)t0 * p.D, bytes, bar, policy);
  };
  if (tid == 0) {
    const int64_t pre = min64(p.S, my_tiles);
    for (int64_t j = 0; j < pre; ++j) issue(j);
  }

  bool aborted = false;
  for (int64_t j = 0; j < my_tiles; ++j) {
    const int s = (int)(j % p.S);
    const uint32_t parity = (uint32_t)((j / p.S) & 1);
    const int64_t t = (cta + j * ncta) * p.R + row;
    const bool valid = t < p.T;

    if (!mbar_wait_bounded(smem_addr(&full[s]), parity, aborted ? 0 : p.wait_limit_ns)) {
      if (!aborted) atomicOr(&g_mx_status, kStatusTimeout);
      aborted = true;
    }

    // ---- load, weight, block absmax, row statistic
    float w[VPT][8];
    float am[VPT];
    float acc = 0.f;
    const uint32_t srow = ring + (uint32_t)s * stage_bytes + (uint32_t)row * p.D * 2;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = i * p.G + g;
      const bool inb = valid && v < p.nvec;
      float m = 0.f;
      if (inb) {
        float f[8];
        bf16x8_to_f32(ld_shared_v4(srow + v * 16), f);
        if (STAT == kStatRms) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(f[e], f[e], acc);
        }
        if (p.gamma != nullptr) {
          const float4* gp = reinterpret_cast<const float4*>(p.gamma + v * 8);
          const float4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
          f[0] *= g0.x; f[1] *= g0.y; f[2] *= g0.z; f[3] *= g0.w;
          f[4] *= g1.x; f[5] *= g1.y; f[6] *= g1.z; f[7] *= g1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          w[i][e] = f[e];
          m = fmaxf(m, fabsf(f[e]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[i][e] = 0.f;
      }
      // block absmax across the B/8 lanes of the block
      for (int o = 1; o < p.gl; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      am[i] = m;
      if (STAT != kStatRms && inb && leader) acc += (STAT == kStatMxP1) ? m : m * m;
    }
    acc = warp_sum(acc);
    float* rbuf = red + (size_t)(j & 1) * p.R * wpr;
    if (lane == 0) rbuf[row * wpr + wir] = acc;
    __syncthreads();  // row partials visible; every read of stage s done

    if (tid == 0 && !aborted && j + p.S < my_tiles) issue(j + p.S);

    if (valid) {
      float tot = 0.f;
      for (int k = 0; k < wpr; ++k) tot += rbuf[row * wpr + k];
      float ms;
      if (STAT == kStatRms) {
        ms = tot / (float)p.D;
      } else if (STAT == kStatMxP1) {
        const float rho = p.corr * (tot / (float)p.K);
        ms = rho * rho;
      } else {
        ms = p.corr * (tot / (float)p.K);
      }
      const float rinv = 1.0f / sqrtf(ms + p.eps);
      if (p.rinv_out != nullptr && g == 0) p.rinv_out[t] = rinv;

#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = i * p.G + g;
        if (v < p.nvec) {
          const int e = e8m0_exponent(am[i] * rinv, kEmax);
          const float inv_scale = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
          if (leader) {
            const int k = v / p.gl;
            p.scales[(size_t)t * p.K + k] = (uint8_t)(e + 127);
            if (p.amax_out != nullptr) p.amax_out[(size_t)t * p.K + k] = am[i];
          }
          float q[8];
#pragma unroll
          for (int e2 = 0; e2 < 8; ++e2) q[e2] = (w[i][e2] * rinv) * inv_scale;
          if (FMT == NTS_FMT_E4M3) {
            const uint32_t lo = cvt_e4m3x2(q[0], q[1]) | (cvt_e4m3x2(q[2], q[3]) << 16);
            const uint32_t hi = cvt_e4m3x2(q[4], q[5]) | (cvt_e4m3x2(q[6], q[7]) << 16);
            st_global_v2_stream(p.codes + (size_t)t * p.D + (size_t)v * 8, lo, hi);
          } else {
            const uint32_t b = cvt_e2m1x2(q[0], q[1]) | (cvt_e2m1x2(q[2], q[3]) << 8) |
                               (cvt_e2m1x2(q[4], q[5]) << 16) | (cvt_e2m1x2(q[6], q[7]) << 24);
            st_global_u32_stream(p.codes + (size_t)t * (p.D / 2) + (size_t)v * 4, b);
          }
        }
      }
    }
  }

  if (aborted && tid == 0) {
    for (int64_t j = max64(0, my_tiles - p.S); j < my_tiles; ++j)
      (void)mbar_wait_bounded(smem_addr(&full[j % p.S]), (uint32_t)((j / p.S) & 1),
                              p.wait_limit_ns);
  }
}

// ------------------------------------------------------------------ launch

namespace {

using MxKernel = void (*)(MxParams);

template <int FMT, int STAT>
MxKernel pick_vpt(int vpt) {
  switch (vpt) {
    case 1: return mx_norm_cast_kernel<1, FMT, STAT>;
    case 2: return mx_norm_cast_kernel<2, FMT, STAT>;
    case 3: return mx_norm_cast_kernel<3, FMT, STAT>;
    case 4: return mx_norm_cast_kernel<4, FMT, STAT>;
    case 5: return mx_norm_cast_kernel<5, FMT, STAT>;
    case 6: return mx_norm_cast_kernel<6, FMT, STAT>;
    case 8: return mx_norm_cast_kernel<8, FMT, STAT>;
    default: return nullptr;
  }
}

template <int FMT>
MxKernel pick_stat(int stat, int vpt) {
  switch (stat) {
    case kStatRms: return pick_vpt<FMT, kStatRms>(vpt);
    case kStatMxP1: return pick_vpt<FMT, kStatMxP1>(vpt);
    case kStatMxP2: return pick_vpt<FMT, kStatMxP2>(vpt);
    default: return nullptr;
  }
}

MxKernel pick_mx(int fmt, int stat, int vpt) {
  return fmt == NTS_FMT_E4M3 ? pick_stat<NTS_FMT_E4M3>(stat, vpt)
                             : pick_stat<NTS_FMT_E2M1>(stat, vpt);
}

}  // namespace

int launch_mx(const MxRequest& rq, cudaStream_t stream, const LaunchTuning& tune) {
  const int D = (int)rq.D;
  const int nvec = D / 8;
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");

  RowShape rs = choose_row_shape(nvec, tune.force_vpt);
  if (rs.G == 0) return fail(NTS_ERR_UNSUPPORTED, "row too wide: D = %d", D);

  int R = std::max(1, 256 / rs.G);
  R = std::min(R, 16);
  while (R > 1 && (rq.T + R - 1) / R < (int64_t)2 * dev.sm_count) R /= 2;
  if (tune.force_rows > 0) R = tune.force_rows;
  if (R * rs.G > kMaxThreads) return fail(NTS_ERR_UNSUPPORTED, "tile of %d rows too large", R);

  int S = 4;
  while (S > 1 && mx_smem_bytes(S, R, D, rs.G) > (size_t)tune.smem_budget) --S;
  if (tune.force_stages > 0) S = tune.force_stages;
  const size_t smem = mx_smem_bytes(S, R, D, rs.G);
  if (smem > (size_t)dev.max_smem_optin)
    return fail(NTS_ERR_UNSUPPORTED, "row too wide for shared memory: D = %d", D);

  const int stat = rq.p == 0 ? kStatRms : (rq.p == 1 ? kStatMxP1 : kStatMxP2);
  MxKernel kern = pick_mx(rq.fmt, stat, rs.vpt);
  if (kern == nullptr) return fail(NTS_ERR_UNSUPPORTED, "no kernel for vpt=%d", rs.vpt);

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
  prm.nvec = nvec;
  prm.G = rs.G;
  prm.R = R;
  prm.S = S;
  prm.K = D / rq.B;
  prm.gl = rq.B / 8;
  prm.eps = rq.eps;
  prm.corr = 0.f;
  if (rq.p == 1) prm.corr = (float)rq.corr;
  if (rq.p == 2) prm.corr = (float)(rq.corr * rq.corr);
  prm.wait_limit_ns = tune.wait_limit_ns;
  prm.missing_tx = tune.missing_tx;

  int rc = prepare_kernel((const void*)kern, smem);
  if (rc != NTS_OK) return rc;

  const int nthreads = R * rs.G;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nthreads, smem);
  if (e != cudaSuccess) return fail_cuda(e, "occupancy query for the MX kernel");
  if (per_sm < 1) return fail(NTS_ERR_UNSUPPORTED, "MX kernel does not fit on an SM");
  int64_t grid = std::min<int64_t>(prm.ntiles, (int64_t)per_sm * dev.sm_count);
  if (tune.force_grid > 0) grid = std::min<int64_t>(prm.ntiles, tune.force_grid);

  log_launch(rq.p == 0 ? "rmsnorm_mxcast" : "mxnorm_cast",
             "T=%lld D=%d B=%d fmt=%d p=%d vpt=%d G=%d R=%d S=%d smem=%zu grid=%lld (%d/SM)",
             (long long)rq.T, D, rq.B, rq.fmt, rq.p, rs.vpt, rs.G, R, S, smem, (long long)grid,
             per_sm);
  kern<<<(unsigned)grid, nthreads, smem, stream>>>(prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "launching the MX kernel");
  return NTS_OK;
}

int read_and_clear_mx_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_mx_status, sizeof(v));
  if (e != cudaSuccess) return fail_cuda(e, "reading the MX status word");
  e = cudaMemcpyToSymbol(g_mx_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clearing the MX status word");
  *out = v;
  return NTS_OK;
}

}  // namespace nts
