// heads_kernel.cu -- headwise QK-Norm on one GB300: one normalization factor
// per attention head of every token (SwiftQK, Sec. II.A), with the heads of a
// token kept whole inside one CTA, so no statistic leaves the warp.
//
// Method: a token row of H = nheads * head_dim values holds its heads one
// after another; head h is normalized over its own head_dim values,
//     y_j = bf16_rne((x_j * gamma_j') * 1/sqrt((1/head_dim) sum x^2 + eps)),
// with gamma (head_dim entries, j' = j mod head_dim) shared by all heads.
//
// GB300 mapping:
//  * a persistent grid of CTAs walks tiles of R whole token rows; a producer
//    warp keeps a ring of S shared-memory stages filled with one 1-D bulk TMA
//    copy per tile; consumer warps release a stage as soon as its data is in
//    registers;
//  * the G threads of a row own 16-byte vectors v = i*G + g.  A head is
//    hv = head_dim/8 consecutive vectors, i.e. hv adjacent lanes of one warp
//    (hv a power of two up to 32, G a multiple of 32): the head's sum of
//    squares is a segmented xor-shuffle reduction over those lanes, and every
//    lane meets the same gamma vector (g mod hv) on every row, so gamma sits
//    in registers for the whole kernel.
#include <cuda_runtime.h>

#include <algorithm>

#include "nts_device.cuh"
#include "nts_internal.h"

namespace nts {

namespace {

// kStatusTimeout bits of the headwise kernels.
__device__ unsigned int g_heads_status;

struct HeadsParams {
  const __nv_bfloat16* X;
  const float* gamma;   // [head_dim]
  __nv_bfloat16* Y;
  float* rinv_out;      // [T, nheads] or nullptr
  int64_t T;
  int64_t ntiles;
  int H;
  int nvec;             // H / 8
  int hv;               // vectors per head, head_dim / 8 (power of two <= 32)
  int hshift;           // log2(hv)
  int nheads;
  int G;                // consumer threads per row (multiple of 32)
  int R;                // rows per tile
  int S;                // ring stages
  float eps;
  float inv_hd;         // 1 / head_dim (exact: head_dim is a power of two)
  uint64_t wait_limit_ns;
  uint32_t missing_tx;  // test hook: bytes expected on the first stage but never sent
  unsigned int* sched;  // zeroed counter pair (next tile, CTAs done), or nullptr:
                        // take tiles round-robin
};

// Shared memory layout (bytes): ring [S][R][H] bf16 | full[S] | empty[S] |
// tile[S] i64 (the tile in stage s, or -1: no more tiles)
struct HeadsLayout {
  uint32_t ring, full, empty, tile, total;
};

HeadsLayout heads_layout(int S, int R, int H) {
  HeadsLayout L;
  L.ring = 0;
  L.full = (uint32_t)S * R * H * 2;
  L.empty = L.full + (uint32_t)S * 8;
  L.tile = L.empty + (uint32_t)S * 8;
  L.total = L.tile + (uint32_t)S * 8;
  return L;
}

template <int VPT>
__global__ void __launch_bounds__(kMaxThreads, 1) heads_kernel(const HeadsParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nconsumer = p.R * p.G;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t stage_bytes = (uint32_t)p.R * p.H * 2;
  const uint32_t full0 = sbase + (uint32_t)p.S * stage_bytes;
  const uint32_t empty0 = full0 + (uint32_t)p.S * 8;
  int64_t* tile_of = reinterpret_cast<int64_t*>(smem + (uint32_t)p.S * stage_bytes + 16 * p.S);
  const int64_t cta = blockIdx.x, ncta = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < p.S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, nconsumer / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // everything above touched shared memory only
  grid_dependency_wait();
  allow_dependent_launch();

  if (tid >= nconsumer) {
    // ------------------------------------------------------ producer warp
    if (lane == 0) {
      bool aborted = false;
      const uint64_t policy = l2_policy_evict_first();
      int s = 0;
      uint32_t ph = 0;  // (n / S) & 1
      int64_t n = 0;    // tiles issued
      while (true) {
        if (n >= p.S && !mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, p.wait_limit_ns)) {
          atomicOr(&g_heads_status, kStatusTimeout);
          aborted = true;
          break;
        }
        // next tile: from the launch's counter, or round-robin
        const int64_t tile = p.sched != nullptr ? (int64_t)atomicAdd(p.sched, 1u) : cta + n * ncta;
        if (tile >= p.ntiles) {
          tile_of[s] = -1;   // published by the arrive (release) below
          mbar_arrive(full0 + 8 * s);
          break;
        }
        tile_of[s] = tile;
        const int64_t t0 = tile * p.R;
        const uint32_t bytes = (uint32_t)min64(p.R, p.T - t0) * p.H * 2;
        mbar_arrive_expect_tx(full0 + 8 * s, bytes + (n == 0 ? p.missing_tx : 0u));
        bulk_g2s(sbase + (uint32_t)s * stage_bytes, p.X + (size_t)t0 * p.H, bytes, full0 + 8 * s,
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
        (void)mbar_wait_bounded(full0 + 8 * (int)(j % p.S), (uint32_t)((j / p.S) & 1),
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
  // this lane's place in its head, the same for every vector it owns
  const int gv = g & (p.hv - 1);
  uint64_t gm[4];
  {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p.gamma + 8 * gv));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p.gamma + 8 * gv + 4));
    gm[0] = f2(a.x, a.y);
    gm[1] = f2(a.z, a.w);
    gm[2] = f2(b.x, b.y);
    gm[3] = f2(b.z, b.w);
  }
  int s = 0;
  uint32_t ph = 0;
  while (true) {
    // a warp leaves together: an expired wait on one lane ends all 32 (the
    // shuffles and barriers below need the whole warp)
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(full0 + 8 * s, ph, p.wait_limit_ns))) {
      if (lane == 0) atomicOr(&g_heads_status, kStatusTimeout);
      break;
    }
    const int64_t tile = *reinterpret_cast<volatile int64_t*>(tile_of + s);
    if (tile < 0 || tile >= p.ntiles) break;   // no more tiles
    const int64_t t = tile * p.R + row;
    const bool valid = t < p.T;
    const unsigned char* srow = smem + (uint32_t)s * stage_bytes + (uint32_t)row * p.H * 2;

    // per vector: its sum of squares (fp32 pairs), values kept in registers
    uint64_t w[VPT][4];
    float ss[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = i * p.G + g;
      uint4 x = make_uint4(0, 0, 0, 0);
      if (valid && v < p.nvec) x = lds128(srow + v * 16);
      w[i][0] = bf16x2_to_f2(x.x);
      w[i][1] = bf16x2_to_f2(x.y);
      w[i][2] = bf16x2_to_f2(x.z);
      w[i][3] = bf16x2_to_f2(x.w);
      const uint64_t a = f2_fma(w[i][0], w[i][0], f2_mul(w[i][1], w[i][1]));
      const uint64_t b = f2_fma(w[i][2], w[i][2], f2_mul(w[i][3], w[i][3]));
      const uint64_t c = f2_add(a, b);
      ss[i] = f2_lo(c) + f2_hi(c);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);

    // each head's sum over its hv lanes (segmented butterfly, all lanes;
    // unrolled, each step guarded by the warp-uniform head size)
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1)
        if (o < p.hv) ss[i] += __shfl_xor_sync(0xFFFFFFFFu, ss[i], o);

    if (valid) {
      __nv_bfloat16* yrow = p.Y + (size_t)t * p.H;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = i * p.G + g;
        if (v < p.nvec) {
          const float rinv = rsqrtf(fmaf(ss[i], p.inv_hd, p.eps));
          const uint64_t rr = f2(rinv, rinv);
          uint64_t y[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) y[q] = f2_mul(f2_mul(w[i][q], gm[q]), rr);
          uint4 o;
          o.x = pack_bf16x2_rn(f2_lo(y[0]), f2_hi(y[0]));
          o.y = pack_bf16x2_rn(f2_lo(y[1]), f2_hi(y[1]));
          o.z = pack_bf16x2_rn(f2_lo(y[2]), f2_hi(y[2]));
          o.w = pack_bf16x2_rn(f2_lo(y[3]), f2_hi(y[3]));
          st_global_v4_stream(yrow + v * 8, o);
          if (p.rinv_out != nullptr && gv == 0)
            p.rinv_out[(size_t)t * p.nheads + (v >> p.hshift)] = rinv;
        }
      }
    }
    if (++s == p.S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

using HeadsKernel = void (*)(HeadsParams);

HeadsKernel pick_heads(int vpt) {
  switch (vpt) {
    case 1: return heads_kernel<1>;
    case 2: return heads_kernel<2>;
    case 3: return heads_kernel<3>;
    case 4: return heads_kernel<4>;
    case 5: return heads_kernel<5>;
    case 6: return heads_kernel<6>;
    case 8: return heads_kernel<8>;
    default: return nullptr;
  }
}

}  // namespace

bool heads_whole_path(int64_t H, int64_t head_dim, int N) {
  // a token row must fit the thread shapes: at most 8 vectors per thread
  if (N != 1 || H > (int64_t)kMaxConsumers * 64) return false;
  for (int hd = 8; hd <= 256; hd *= 2)
    if (head_dim == hd) return true;
  return false;
}

int launch_heads(const void* X, const float* gamma, void* Y, float* rinv, int64_t T, int64_t H,
                 int64_t head_dim, float eps, cudaStream_t stream, const LaunchTuning& tune) {
  if (const int injected = take_injected_failure()) return injected;
  const DeviceInfo& dev = device_info();
  if (!dev.ok) return fail(NTS_ERR_CUDA, "could not query the current device");
  const int nvec = (int)(H / 8);
  // Few vectors per thread and many threads per row: the per-head
  // reductions and factors are latency chains, so more warps per SM pay
  // (measured on GB300 at H = 5120: 2 vectors per thread, 320 threads per
  // row, beat 4 per thread by 25%).  Take the fewest vectors per thread
  // whose row fits 384 threads with at most 1/8 of the slots idle.
  RowShape rs;
  if (tune.force_vpt > 0) {
    rs = choose_row_shape(nvec, tune.force_vpt);
  } else {
    for (int vpt : {1, 2, 3, 4, 5, 6, 8}) {
      const int G = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
      if (G > 384 || 8 * (G * vpt - nvec) > nvec) continue;
      rs.vpt = vpt;
      rs.G = G;
      break;
    }
    if (rs.G == 0) rs = choose_row_shape(nvec, 0);
  }
  if (rs.G == 0) return fail(NTS_ERR_UNSUPPORTED, "row too wide: H = %lld", (long long)H);

  // Rows per tile: about four consumer warps and at least 8 KB per stage,
  // fewer when T is small so that the tiles spread over the GPU.
  int R = std::max(1, 128 / rs.G);
  R = std::max(R, (int)((8192 + 2 * H - 1) / (2 * H)));
  R = std::min(R, std::max(1, kMaxConsumers / rs.G));
  while (R > 1 && (T + R - 1) / R < (int64_t)2 * dev.sm_count) R /= 2;
  if (tune.force_rows > 0) R = tune.force_rows;
  if (R * rs.G > kMaxConsumers) return fail(NTS_ERR_UNSUPPORTED, "tile of %d rows too large", R);

  const int stage = (int)(R * H * 2);
  int S = stage >= 32768 ? 2 : (stage >= 12288 ? 3 : 4);
  while (S > 2 && heads_layout(S, R, (int)H).total > (uint32_t)tune.smem_budget) --S;
  while (S > 1 && heads_layout(S, R, (int)H).total > (uint32_t)dev.max_smem_optin) --S;
  if (tune.force_stages > 0) S = tune.force_stages;
  const size_t smem = heads_layout(S, R, (int)H).total;
  if (smem > (size_t)dev.max_smem_optin)
    return fail(NTS_ERR_UNSUPPORTED, "row too wide for shared memory: H = %lld", (long long)H);

  HeadsKernel kern = pick_heads(rs.vpt);
  if (kern == nullptr) return fail(NTS_ERR_UNSUPPORTED, "no headwise kernel for vpt=%d", rs.vpt);

  HeadsParams prm;
  prm.X = static_cast<const __nv_bfloat16*>(X);
  prm.gamma = gamma;
  prm.Y = static_cast<__nv_bfloat16*>(Y);
  prm.rinv_out = rinv;
  prm.T = T;
  prm.ntiles = (T + R - 1) / R;
  prm.H = (int)H;
  prm.nvec = nvec;
  prm.hv = (int)(head_dim / 8);
  prm.hshift = 0;
  while ((1 << prm.hshift) < prm.hv) ++prm.hshift;
  prm.nheads = (int)(H / head_dim);
  prm.G = rs.G;
  prm.R = R;
  prm.S = S;
  prm.eps = eps;
  prm.inv_hd = 1.0f / (float)head_dim;
  prm.wait_limit_ns = tune.wait_limit_ns;
  prm.missing_tx = tune.missing_tx;
  prm.sched = tune.dynamic ? sched_counters(stream) : nullptr;

  int rc = prepare_kernel((const void*)kern, smem);
  if (rc != NTS_OK) return rc;
  const int nthreads = R * rs.G + 32;  // consumers + producer warp
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nthreads, smem);
  if (e != cudaSuccess) return fail_cuda(e, "occupancy query for the headwise kernel");
  if (per_sm < 1) return fail(NTS_ERR_UNSUPPORTED, "headwise kernel does not fit on an SM");
  int64_t grid = std::min<int64_t>(prm.ntiles, (int64_t)per_sm * dev.sm_count);
  if (tune.force_grid > 0) grid = std::min<int64_t>(prm.ntiles, tune.force_grid);

  log_launch("qknorm_rms_heads", "T=%lld H=%lld head_dim=%lld vpt=%d G=%d R=%d S=%d smem=%zu "
             "grid=%lld (%d/SM)", (long long)T, (long long)H, (long long)head_dim, rs.vpt, rs.G,
             R, S, smem, (long long)grid, per_sm);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = tune.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return fail_cuda(e, "launching the headwise kernel");
  return NTS_OK;
}

int read_and_clear_heads_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_heads_status, sizeof(v));
  if (e != cudaSuccess) return fail_cuda(e, "reading the headwise status word");
  e = cudaMemcpyToSymbol(g_heads_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clearing the headwise status word");
  *out = v;
  return NTS_OK;
}

}  // namespace nts
