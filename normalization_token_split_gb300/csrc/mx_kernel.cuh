// mx_kernel.cuh -- fused per-token normalization + MX block cast on one
// GB300: RMSNorm + MXCast, and MXNorm + MXCast (p = 1 or 2).
//
// Method (MXNorm paper card, abstract, Fig. 1 caption and Fig. A.1):
//   a row of D values is cut into K = D/B blocks of B contiguous values; each
//   block is stored as B element codes (E4M3 or E2M1) sharing one E8M0 scale
//   2^round(log2(normalized absmax / 2^emax)), or (NVFP4, Table 4's second
//   format) 16 E2M1 codes sharing one E4M3 scale, normalized absmax / 6.
//   RMSNorm + MXCast takes the RMS from sum x^2 over the row; MXNorm
//   estimates it from the block absmaxes the cast computes anyway,
//   rho~ = c(B,p) * M_p(absmax), a reduction B times smaller.  Both are fused
//   into one kernel (Fig. 8).
//
// GB300 mapping:
//  * a persistent grid of CTAs walks tiles of R whole rows.  A producer warp
//    keeps a ring of S shared-memory stages filled with one 1-D bulk TMA copy
//    per tile (the rows are contiguous); consumer warps hand a stage back
//    through an "empty" mbarrier;
//  * every consumer thread owns whole MX blocks of 16 or 32 values, so a
//    block's absmax, its scale exponent and its scale byte are
//    thread-local: no shuffles, one exponent per block; a block of 64 values
//    is split between two adjacent lanes (32 values each) that combine their
//    absmaxes with one shuffle.  A row takes 16 threads (two rows per warp)
//    or whole warps.  Without a gain the absmax runs on packed bf16 pairs
//    (max.xorsign.abs.bf16x2); the products x*rinv*2^-e run on the packed
//    f32x2 pipes, and the element cast is the hardware
//    cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32;
//  * a thread's unit (a block, or half of a 64-value block) is U 16-byte
//    vectors 16*U bytes apart from its neighbours'; thread L reads them in
//    the order k ^ ((L*U/8) mod U) so the eight lanes of each shared-memory
//    phase hit eight distinct bank groups, and writes the unit's codes back
//    in element order with one store;
//  * the row is read from shared memory twice (statistic, then cast), so no
//    thread holds more than its block absmaxes between the passes; the stage
//    is released after the second pass;
//  * the row statistic is a shuffle reduction over the row's 16 or 32
//    lanes; a row wider than one warp adds one exchange through shared
//    memory guarded by an mbarrier.
#pragma once

#include <cuda_runtime.h>

#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

// kStatusTimeout bits of the MX kernels of the including translation unit;
// every unit has its own word (no relocatable device code) and exports a
// reader built on read_and_clear_local_mx_status().
static __device__ unsigned int g_mx_status;

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
  int K;                // D / B blocks per row (units: K, or 2K for B = 64)
  int G;                // consumer threads per row: 16 (two rows per warp) or a multiple of 32
  int R;                // rows per tile
  int S;                // ring stages
  float eps;
  float corr;           // MXNorm: c(B,1) for p = 1, c(B,2)^2 for p = 2
  int post;             // MXNorm: 1 = statistic from E8M0-rounded absmaxes (post-round)
  int wide;             // 1: every codes row starts on a 32-byte boundary (32-byte stores)
  uint64_t wait_limit_ns;
  uint32_t missing_tx;  // test hook: bytes expected on the first stage but never sent
  unsigned int* sched;  // zeroed counter pair (next tile, CTAs done), or nullptr:
                        // take tiles round-robin
};

enum { kStatRms = 0, kStatMxP1 = 1, kStatMxP2 = 2 };

// Shared memory layout (bytes, in order):
//   ring [S][R][D] bf16 | full[S] | empty[S] | tile[S] i64 | rbar[2][R] |
//   red[2][R][WPR] f32
// tile[s] is the tile the producer put in stage s, or -1: no more tiles.
struct MxLayout {
  uint32_t ring, full, empty, tile, rbar, red, rcp, total;
};

// rcp: the NVFP4 scale reciprocals (128 floats; empty for the E8M0 formats).
__host__ __device__ inline MxLayout mx_layout(int S, int R, int D, int G, bool nvfp4) {
  MxLayout L;
  L.ring = 0;
  L.full = L.ring + (uint32_t)S * R * D * 2;
  L.empty = L.full + (uint32_t)S * 8;
  L.tile = L.empty + (uint32_t)S * 8;
  L.rbar = L.tile + (uint32_t)S * 8;
  L.red = L.rbar + (uint32_t)2 * R * 8;
  L.rcp = L.red + (uint32_t)2 * R * (G / 32) * 4;
  L.total = L.rcp + (nvfp4 ? 128u * 4u : 0u);
  return L;
}

// 2^round(log2 a) for a >= 0 (0 for a == 0): the power of two the E8M0
// rounding picks for a block absmax a, subnormal a included.
__device__ __forceinline__ float round_pow2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int field = (int)(b >> 23);
  const uint32_t m = b & 0x7FFFFFu;
  int k;
  if (field == 0) {
    if (m == 0) return 0.f;
    const int msb = 31 - __clz(m);                       // a = m * 2^-149
    const uint32_t frac = (m << (23 - msb)) & 0x7FFFFFu;  // significand of a, 23 bits
    k = msb - 149 + (frac >= 0x3504F4u ? 1 : 0);
  } else {
    k = field - 127 + (m >= 0x3504F4u ? 1 : 0);
  }
  if (k >= 128) return __uint_as_float(0x7F800000u);     // beyond fp32
  if (k >= -126) return __uint_as_float((uint32_t)(k + 127) << 23);
  return __uint_as_float(1u << (k + 149));
}

// 8 bf16 values (one vector) times an fp32 gain vector at `gp`, as four
// f32x2 pairs.
__device__ __forceinline__ void weigh_vector(const uint4& v, const float* gp, uint64_t (&w)[4]) {
  const float4 g0 = __ldg(reinterpret_cast<const float4*>(gp));
  const float4 g1 = __ldg(reinterpret_cast<const float4*>(gp) + 1);
  w[0] = f2_mul(bf16x2_to_f2c(v.x), f2c(g0.x, g0.y));
  w[1] = f2_mul(bf16x2_to_f2c(v.y), f2c(g0.z, g0.w));
  w[2] = f2_mul(bf16x2_to_f2c(v.z), f2c(g1.x, g1.y));
  w[3] = f2_mul(bf16x2_to_f2c(v.w), f2c(g1.z, g1.w));
}

// Element codes of one unit (UV 16-byte vectors of a row staged in shared
// memory at `base`, read in the order k ^ sig, k = 0..UV-1): q = (w * a) * c
// with w = x or fp32(x * gamma) (GAMMA), then the packed conversions (`keep`
// masks NVFP4 blocks with a zero scale).  The codes are put back in element
// order in registers (a butterfly of selects on the bits of sig) and the
// whole unit leaves in one store (32 bytes when `wide`: the codes row is
// 32-byte aligned), so that every store instruction writes whole 32-byte
// sectors.
template <int FMT, int UV, bool GAMMA>
__device__ __forceinline__ void cast_unit(const unsigned char* base, int sig, const float* gamma,
                                          int b, uint64_t a, uint64_t c, uint8_t* crow,
                                          uint32_t keep, bool wide) {
  constexpr int kU = UV * 8;
  constexpr int kW = FMT == NTS_FMT_E4M3 ? 2 : 1;   // code words per vector
  uint32_t cw[UV][kW];
#pragma unroll
  for (int k = 0; k < UV; ++k) {
    const int u = k ^ sig;
    const uint4 v = lds128(base + u * 16);
    uint64_t w[4];
    if (!GAMMA) {
      w[0] = bf16x2_to_f2c(v.x);
      w[1] = bf16x2_to_f2c(v.y);
      w[2] = bf16x2_to_f2c(v.z);
      w[3] = bf16x2_to_f2c(v.w);
    } else {
      weigh_vector(v, gamma + (size_t)b * kU + u * 8, w);
    }
    uint64_t q[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) q[h] = f2_mul(f2_mul(w[h], a), c);
    if (FMT == NTS_FMT_E4M3) {
      cw[k][0] = cvt_e4m3x4(f2_lo(q[0]), f2_hi(q[0]), f2_lo(q[1]), f2_hi(q[1]));
      cw[k][kW - 1] = cvt_e4m3x4(f2_lo(q[2]), f2_hi(q[2]), f2_lo(q[3]), f2_hi(q[3]));
    } else {
      cw[k][0] = cvt_e2m1x8(f2_lo(q[0]), f2_hi(q[0]), f2_lo(q[1]), f2_hi(q[1]), f2_lo(q[2]),
                            f2_hi(q[2]), f2_lo(q[3]), f2_hi(q[3])) & keep;
    }
  }
  // cw[k] holds vector k ^ sig: swap the pairs that differ in each set bit
#pragma unroll
  for (int bit = 1; bit < UV; bit <<= 1) {
    const bool sw = (sig & bit) != 0;
#pragma unroll
    for (int k = 0; k < UV; ++k) {
      if (k & bit) continue;
#pragma unroll
      for (int h = 0; h < kW; ++h) {
        const uint32_t x = cw[k][h], y = cw[k | bit][h];
        cw[k][h] = sw ? y : x;
        cw[k | bit][h] = sw ? x : y;
      }
    }
  }
  uint8_t* dst = crow + (size_t)b * (UV * 4 * kW);
  if (UV * kW == 8) {          // 32 bytes: E4M3 with 4 vectors
    if (wide) {
      st_global_v8(dst, cw[0][0], cw[0][kW - 1], cw[1][0], cw[1][kW - 1], cw[2 % UV][0],
                   cw[2 % UV][kW - 1], cw[3 % UV][0], cw[3 % UV][kW - 1]);
    } else {
      st_global_v4(dst, cw[0][0], cw[0][kW - 1], cw[1][0], cw[1][kW - 1]);
      st_global_v4(dst + 16, cw[2 % UV][0], cw[2 % UV][kW - 1], cw[3 % UV][0],
                   cw[3 % UV][kW - 1]);
    }
  } else if (UV * kW == 4) {   // 16 bytes: E4M3 with 2 vectors, E2M1 with 4
    if (kW == 2)
      st_global_v4(dst, cw[0][0], cw[0][kW - 1], cw[1 % UV][0], cw[1 % UV][kW - 1]);
    else
      st_global_v4(dst, cw[0][0], cw[1 % UV][0], cw[2 % UV][0], cw[3 % UV][0]);
  } else {                     // 8 bytes: E2M1 with 2 vectors
    st_global_v2(dst, cw[0][0], cw[1 % UV][0]);
  }
}

// Pass 1 over a thread's units of a staged row: the absmax of w = x (or
// fp32(x * gamma)) of every unit into am[], and for RMSNorm the packed sums
// of x^2 into acc.  Four independent chains per reduction (one per 32-bit
// lane of a vector), so that a unit is not one long dependency chain.
template <int UV, int BPT, bool GAMMA, bool SUMSQ>
__device__ __forceinline__ void mx_absmax_pass(const unsigned char* srow, const float* gamma,
                                               int G, int g, int units, bool valid, int sig,
                                               float (&am)[BPT], uint64_t (&acc)[4]) {
  constexpr int kU = UV * 8;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    const int b = i * G + g;
    am[i] = 0.f;
    if (valid && b < units) {
      const unsigned char* base = srow + (uint32_t)b * kU * 2;
      if (!GAMMA) {
        uint32_t m[4] = {0, 0, 0, 0};
#pragma unroll
        for (int k = 0; k < UV; ++k) {
          const int u = k ^ sig;
          const uint4 v = lds128(base + u * 16);
          m[0] = bf16x2_absmax(m[0], v.x);
          m[1] = bf16x2_absmax(m[1], v.y);
          m[2] = bf16x2_absmax(m[2], v.z);
          m[3] = bf16x2_absmax(m[3], v.w);
          if (SUMSQ) {
            const uint64_t a = bf16x2_to_f2c(v.x), c = bf16x2_to_f2c(v.y);
            const uint64_t d = bf16x2_to_f2c(v.z), e = bf16x2_to_f2c(v.w);
            acc[0] = f2_fma(a, a, acc[0]);
            acc[1] = f2_fma(c, c, acc[1]);
            acc[2] = f2_fma(d, d, acc[2]);
            acc[3] = f2_fma(e, e, acc[3]);
          }
        }
        am[i] = bf16x2_hmax_abs(bf16x2_absmax(bf16x2_absmax(m[0], m[1]),
                                              bf16x2_absmax(m[2], m[3])));
      } else {
        float mf[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < UV; ++k) {
          const int u = k ^ sig;
          const uint4 v = lds128(base + u * 16);
          if (SUMSQ) {
            const uint64_t a = bf16x2_to_f2c(v.x), c = bf16x2_to_f2c(v.y);
            const uint64_t d = bf16x2_to_f2c(v.z), e = bf16x2_to_f2c(v.w);
            acc[0] = f2_fma(a, a, acc[0]);
            acc[1] = f2_fma(c, c, acc[1]);
            acc[2] = f2_fma(d, d, acc[2]);
            acc[3] = f2_fma(e, e, acc[3]);
          }
          uint64_t w[4];
          weigh_vector(v, gamma + (size_t)b * kU + u * 8, w);
          mf[k & 3] = absmax8(mf[k & 3], w);
        }
        am[i] = fmaxf(fmaxf(mf[0], mf[1]), fmaxf(mf[2], mf[3]));
      }
    }
  }
}

// MXNorm statistic of a thread's block absmaxes: sum a (p = 1) or sum a^2
// (p = 2), a = the absmax, or its E8M0-rounded power of two (POST); the
// units that lead a block (every unit, or the even half of a split block).
template <int BPT, int STAT, bool POST, bool SPLIT>
__device__ __forceinline__ float mx_block_stat(const float (&am)[BPT], int G, int g, int units,
                                               bool valid) {
  float stat = 0.f;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    const int b = i * G + g;
    if (valid && b < units && (!SPLIT || (g & 1) == 0)) {
      const float a = POST ? round_pow2(am[i]) : am[i];
      if (STAT == kStatMxP1) stat += a;
      if (STAT == kStatMxP2) stat = fmaf(a, a, stat);
    }
  }
  return stat;
}

template <int VB, int BPT, int FMT, int STAT, bool GAMMA>
__global__ void __launch_bounds__(kMaxThreads, 1) mx_norm_cast_kernel(const MxParams p) {
  // A 64-value block is split between two adjacent lanes, 32 values each
  // (the layout of 32-value blocks), which combine their absmaxes by one
  // shuffle: a thread's unit is then half a block.
  constexpr bool kSplit = (VB == 8);
  constexpr int kUV = kSplit ? 4 : VB;                       // vectors per unit
  constexpr int kU = kUV * 8;                                // values per unit
  constexpr int kEmax = (FMT == NTS_FMT_E4M3) ? 8 : 2;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nconsumer = p.R * p.G;
  const int wpr = p.G >= 32 ? p.G >> 5 : 1;   // warps per row (G = 16: two rows per warp)
  const MxLayout L = mx_layout(p.S, p.R, p.D, p.G, FMT == NTS_FMT_NVFP4);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t stage_bytes = (uint32_t)p.R * p.D * 2;
  const int64_t cta = blockIdx.x, ncta = gridDim.x;
  int64_t* tile_of = reinterpret_cast<int64_t*>(smem + L.tile);

  if (tid == 0) {
    for (int s = 0; s < p.S; ++s) {
      mbar_init(sbase + L.full + 8 * s, 1);
      mbar_init(sbase + L.empty + 8 * s, nconsumer / 32);
    }
    for (int b = 0; b < 2 * p.R; ++b) mbar_init(sbase + L.rbar + 8 * b, wpr);
    fence_mbar_init();
  }
  float* rcp = reinterpret_cast<float*>(smem + L.rcp);
  if (FMT == NTS_FMT_NVFP4) fill_e4m3_reciprocals(rcp, tid, (int)blockDim.x);
  __syncthreads();
  // everything above touched shared memory only
  grid_dependency_wait();
  allow_dependent_launch();

  if (tid >= nconsumer) {
    // ------------------------------------------------------ producer warp
    if (lane == 0) {
      bool aborted = false;
      const uint64_t policy = l2_policy_evict_first();
      // ring stage s of tile j and the parity of its pass, (j / S) & 1, kept
      // incrementally (no 64-bit division in the loop)
      int s = 0;
      uint32_t ph = 0;
      int64_t n = 0;  // tiles issued
      while (true) {
        if (n >= p.S && !mbar_wait_bounded(sbase + L.empty + 8 * s, ph ^ 1u, p.wait_limit_ns)) {
          atomicOr(&g_mx_status, kStatusTimeout);
          aborted = true;
          break;
        }
        // next tile: from the launch's counter, or round-robin
        const int64_t tile = p.sched != nullptr ? (int64_t)atomicAdd(p.sched, 1u) : cta + n * ncta;
        const uint32_t bar = sbase + L.full + 8 * s;
        if (tile >= p.ntiles) {
          tile_of[s] = -1;   // published by the arrive (release) below
          mbar_arrive(bar);
          break;
        }
        tile_of[s] = tile;
        const int64_t t0 = tile * p.R;
        const uint32_t bytes = (uint32_t)min64(p.R, p.T - t0) * p.D * 2;
        mbar_arrive_expect_tx(bar, bytes + (n == 0 ? p.missing_tx : 0u));
        bulk_g2s(sbase + L.ring + (uint32_t)s * stage_bytes, p.X + (size_t)t0 * p.D, bytes, bar,
                 policy);
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
      // count this CTA out; the last one re-arms the pair for the next launch
      if (p.sched != nullptr) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
          atomicExch(p.sched, 0u);
          atomicExch(p.sched + 1, 0u);
        }
      }
    }
    __syncwarp();
    return;
  }

  // --------------------------------------------------------- consumer warps
  const int row = tid / p.G;
  const int g = tid - row * p.G;
  const int wir = g >> 5;
  const int sig = ((lane * kUV) >> 3) & (kUV - 1);   // bank-conflict-free start vector
  const int units = kSplit ? 2 * p.K : p.K;          // units per row
  const size_t cbytes = (FMT == NTS_FMT_E4M3) ? (size_t)p.D : (size_t)p.D / 2;
  bool aborted = false;

  int s = 0;          // ring stage of the j-th tile
  uint32_t ph = 0;    // (j / S) & 1
  for (int64_t j = 0;; ++j) {
    // a warp leaves together: an expired wait on one lane ends all 32 (the
    // shuffles and barriers below need the whole warp)
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(sbase + L.full + 8 * s, ph, p.wait_limit_ns))) {
      if (lane == 0) atomicOr(&g_mx_status, kStatusTimeout);
      break;
    }
    const int64_t tile = *reinterpret_cast<volatile int64_t*>(tile_of + s);
    if (tile < 0 || tile >= p.ntiles) break;   // no more tiles
    const int64_t t = tile * p.R + row;
    const bool valid = t < p.T;
    const unsigned char* srow = smem + L.ring + (uint32_t)s * stage_bytes + (uint32_t)row * p.D * 2;

    // ---- pass 1: block absmaxes (of w = x or x*gamma) and the statistic
    float am[BPT];
    uint64_t acc[4] = {0, 0, 0, 0};  // RMSNorm: packed sums of x^2
    mx_absmax_pass<kUV, BPT, GAMMA, STAT == kStatRms>(srow, p.gamma, p.G, g, units, valid, sig,
                                                      am, acc);
    // the two halves of a split block share one absmax (lanes g, g ^ 1 hold
    // units b, b ^ 1: same row, both in range or both out, as G and the
    // unit count are even)
    if (kSplit) {
#pragma unroll
      for (int i = 0; i < BPT; ++i) am[i] = fmaxf(am[i], __shfl_xor_sync(0xFFFFFFFFu, am[i], 1));
    }
    float stat;
    if (STAT == kStatRms) {
      const uint64_t a = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      stat = f2_lo(a) + f2_hi(a);
    } else if (p.post) {
      stat = mx_block_stat<BPT, STAT, true, kSplit>(am, p.G, g, units, valid);
    } else {
      stat = mx_block_stat<BPT, STAT, false, kSplit>(am, p.G, g, units, valid);
    }
    stat = group_sum(stat, min(p.G, 32));
    if (wpr > 1) {
      // a row spans several warps: add their partials in warp order
      const int bsel = (int)(j & 1);
      float* red = reinterpret_cast<float*>(smem + L.red) + (size_t)(bsel * p.R + row) * wpr;
      const uint32_t rbar = sbase + L.rbar + 8 * (bsel * p.R + row);
      if (lane == 0) {
        red[wir] = stat;
        mbar_arrive(rbar);
      }
      if (!mbar_wait_bounded(rbar, (uint32_t)((j >> 1) & 1), aborted ? 0 : p.wait_limit_ns)) {
        if (!aborted) atomicOr(&g_mx_status, kStatusTimeout);
        aborted = true;
      }
      stat = 0.f;
      for (int k = 0; k < wpr; ++k) stat += red[k];
    }

    // ---- the row's normalization factor
    float ms;
    if (STAT == kStatRms) {
      ms = stat / (float)p.D;
    } else if (STAT == kStatMxP1) {
      const float rho = p.corr * (stat / (float)p.K);
      ms = rho * rho;
    } else {
      ms = p.corr * (stat / (float)p.K);
    }
    const float rinv = 1.0f / sqrtf(ms + p.eps);
    if (valid && p.rinv_out != nullptr && g == 0) p.rinv_out[t] = rinv;

    // ---- pass 2: scales and element codes
    uint8_t* crow = p.codes + (size_t)t * cbytes;
    uint8_t* srow_sc = p.scales + (size_t)t * p.K;
    if (FMT == NTS_FMT_NVFP4) {
      if (valid) {
        const uint64_t rr = f2c(rinv, rinv);
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
          const int b = i * p.G + g;   // unit = block (B = 16)
          if (b < units) {
            float is;
            const uint32_t sc = nvfp4_scale(am[i] * rinv, rcp, &is);
            srow_sc[b] = (uint8_t)sc;
            if (p.amax_out != nullptr) p.amax_out[(size_t)t * p.K + b] = am[i];
            cast_unit<FMT, kUV, GAMMA>(srow + (uint32_t)b * kU * 2, sig, p.gamma, b, rr,
                                       f2c(is, is), crow, sc != 0 ? ~0u : 0u, false);
          }
        }
      }
    } else {
      // E8M0: every block's scale byte first, then the codes, each by the
      // two products of the definition, q = fp32(fp32(w * rinv) * 2^-e)
      // (measured on GB300: folding them into one product by a per-block
      // multiplier, with the bound checks that keep it bit-identical and a
      // warp vote, was no faster)
      float isc[BPT];   // 2^-e of every unit
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        const int b = i * p.G + g;   // unit
        isc[i] = 0.f;
        if (valid && b < units) {
          const int blk = kSplit ? (b >> 1) : b;
          const bool lead = !kSplit || (b & 1) == 0;   // writes the block's scale
          const uint32_t sbyte = (uint32_t)(e8m0_exponent(am[i] * rinv, kEmax) + 127);
          if (lead) srow_sc[blk] = (uint8_t)sbyte;
          if (p.amax_out != nullptr && lead) p.amax_out[(size_t)t * p.K + blk] = am[i];
          isc[i] = __uint_as_float((254u - sbyte) << 23);   // 2^-e, e = sbyte - 127
        }
      }
      if (valid) {
        const uint64_t rr = f2c(rinv, rinv);
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
          const int b = i * p.G + g;
          if (b < units)
            cast_unit<FMT, kUV, GAMMA>(srow + (uint32_t)b * kU * 2, sig, p.gamma, b, rr,
                                       f2c(isc[i], isc[i]), crow, ~0u, p.wide);
        }
      }
    }
    // every read of stage s by this warp is done
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + L.empty + 8 * s);
    if (aborted) break;
    if (++s == p.S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

using MxKernel = void (*)(MxParams);

// The kernel for BPT units of a thread (blocks of VB vectors; half blocks of
// 4 vectors for VB = 8), with or without a gain, or nullptr where a thread
// would hold more than 16 vectors (256 bytes) of its row (slower on GB300
// wherever measured; the launcher never picks them).
template <int FMT, int STAT, int VB, int BPT>
MxKernel mx_kernel_if_small(bool gamma) {
  if constexpr (BPT * (VB == 8 ? 4 : VB) <= 16) {
    return gamma ? mx_norm_cast_kernel<VB, BPT, FMT, STAT, true>
                 : mx_norm_cast_kernel<VB, BPT, FMT, STAT, false>;
  } else {
    return nullptr;
  }
}

template <int FMT, int STAT, int VB>
MxKernel pick_mx_bpt(int bpt, bool gamma) {
  switch (bpt) {
    case 1: return mx_kernel_if_small<FMT, STAT, VB, 1>(gamma);
    case 2: return mx_kernel_if_small<FMT, STAT, VB, 2>(gamma);
    case 3: return mx_kernel_if_small<FMT, STAT, VB, 3>(gamma);
    case 4: return mx_kernel_if_small<FMT, STAT, VB, 4>(gamma);
    case 5: return mx_kernel_if_small<FMT, STAT, VB, 5>(gamma);
    case 6: return mx_kernel_if_small<FMT, STAT, VB, 6>(gamma);
    case 7: return mx_kernel_if_small<FMT, STAT, VB, 7>(gamma);
    case 8: return mx_kernel_if_small<FMT, STAT, VB, 8>(gamma);
    default: return nullptr;
  }
}

template <int FMT, int STAT>
MxKernel pick_mx_block(int B, int bpt, bool gamma) {
  switch (B) {
    case 16: return pick_mx_bpt<FMT, STAT, 2>(bpt, gamma);
    case 32: return pick_mx_bpt<FMT, STAT, 4>(bpt, gamma);
    case 64: return pick_mx_bpt<FMT, STAT, 8>(bpt, gamma);
    default: return nullptr;
  }
}

static inline int read_and_clear_local_mx_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_mx_status, sizeof(v));
  if (e != cudaSuccess) return fail_cuda(e, "reading an MX status word");
  e = cudaMemcpyToSymbol(g_mx_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clearing an MX status word");
  *out = v;
  return NTS_OK;
}

// One translation unit per element format and statistic (mx_e4m3_rms.cu,
// ..., mx_e2m1_p2.cu; NVFP4 in mx_nvfp4.cu), so that they compile in
// parallel; each has its own status word.
#define NTS_MX_UNIT(NAME, FMT, STAT)                                            \
  MxKernel pick_##NAME(int B, int bpt, bool gamma) {                             \
    return pick_mx_block<FMT, STAT>(B, bpt, gamma);                              \
  }                                                                              \
  int read_and_clear_##NAME##_status(unsigned* out) { return read_and_clear_local_mx_status(out); }

MxKernel pick_mx_e4m3_rms(int B, int bpt, bool gamma);
MxKernel pick_mx_e4m3_p1(int B, int bpt, bool gamma);
MxKernel pick_mx_e4m3_p2(int B, int bpt, bool gamma);
MxKernel pick_mx_e2m1_rms(int B, int bpt, bool gamma);
MxKernel pick_mx_e2m1_p1(int B, int bpt, bool gamma);
MxKernel pick_mx_e2m1_p2(int B, int bpt, bool gamma);
MxKernel pick_mx_nvfp4(int stat, int B, int bpt, bool gamma);
int read_and_clear_mx_e4m3_rms_status(unsigned* out);
int read_and_clear_mx_e4m3_p1_status(unsigned* out);
int read_and_clear_mx_e4m3_p2_status(unsigned* out);
int read_and_clear_mx_e2m1_rms_status(unsigned* out);
int read_and_clear_mx_e2m1_p1_status(unsigned* out);
int read_and_clear_mx_e2m1_p2_status(unsigned* out);
int read_and_clear_mx_nvfp4_status(unsigned* out);

}  // namespace nts
