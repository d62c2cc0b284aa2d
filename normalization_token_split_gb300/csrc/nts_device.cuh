// nts_device.cuh -- inline-PTX building blocks for the sm_103a kernels:
// mbarriers with bounded waits, bulk (TMA) global->shared copies, cluster
// ranks / barriers / distributed shared memory stores, fp8/fp4 packing.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace nts {

// Status bits a kernel ORs into its device status word.
constexpr unsigned kStatusTimeout = 1u;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// `limit_ns` nanoseconds of %globaltimer.  Returns false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------- bulk async copies

// One-dimensional bulk copy global -> shared (TMA unit, no tensor map).
// Both addresses 16-byte aligned, bytes a multiple of 16.  Completion is
// signalled as transaction bytes on `bar`.  The L2 hint marks the source
// lines for early eviction: every input byte is read exactly once.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ cluster

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ------------------------------------------------------------ data movement

// Loads from this CTA's shared memory and stores of results to global
// memory as ordinary C++ accesses, not asm: the compiler then knows the
// address spaces and may interleave the loads of one vector with the stores
// of earlier ones.  The mbarrier operations' asm carries a memory clobber
// and so still orders the loads against the TMA writes that fill a stage and
// against the release of the stage to the producer.
__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint2 lds64(const unsigned char* p) {
  return *reinterpret_cast<const uint2*>(p);
}

// 16-byte store that streams through L2 (evict-first, st.global.cs).
__device__ __forceinline__ void st_global_v4_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// 8 bf16 (one 16-byte vector) -> 8 floats, element order preserved.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two floats -> two E4M3 bytes (RNE, saturating); `lo` lands in bits 0-7.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four floats -> four E4M3 bytes in one word, f0 in bits 0-7 (RNE,
// saturating); the two 16-bit conversions are packed by a register move.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float f0, float f1, float f2, float f3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(f0), "f"(f1), "f"(f2), "f"(f3));
  return r;
}

// Eight floats -> eight E2M1 nibbles in one word, f0 in bits 0-3 (RNE,
// saturating).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float f0, float f1, float f2, float f3, float f4,
                                               float f5, float f6, float f7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(f0), "f"(f1), "f"(f2), "f"(f3), "f"(f4), "f"(f5), "f"(f6), "f"(f7));
  return r;
}

// Two floats -> two E2M1 nibbles in one byte (RNE, saturating); `lo` lands
// in bits 0-3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------- more mbarrier / proxies

// Arrive once (release at CTA scope) without a transaction count.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Store a 32-bit value into the shared memory of a CTA of this cluster and
// signal 4 transaction bytes on that CTA's mbarrier (both addresses mapped
// with map_to_rank).  No fence, no barrier: the receiver's wait on its
// mbarrier makes the value visible.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
          remote_addr),
      "r"(__float_as_uint(v)), "r"(remote_bar)
      : "memory");
}

// Two 32-bit values (8 bytes) into a cluster CTA's shared memory, completing
// 8 transaction bytes on its mbarrier (address 8-byte aligned).
__device__ __forceinline__ void st_async_f32x2(uint32_t remote_addr, float a, float b,
                                               uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
          remote_addr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(remote_bar)
      : "memory");
}

// One 64-bit value into a cluster CTA's shared memory (8-byte aligned),
// completing 8 transaction bytes on its mbarrier.
__device__ __forceinline__ void st_async_u64(uint32_t remote_addr, uint64_t v,
                                             uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
          remote_addr),
      "r"((uint32_t)v), "r"((uint32_t)(v >> 32)), "r"(remote_bar)
      : "memory");
}

// 1-D bulk copy global -> shared without an L2 hint (for re-read data).
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ------------------------------------------------------- MX block scales

// E8M0 exponent of a block whose normalized absmax is `ay` (>= 0, not NaN):
// round(log2 ay) - emax, clamped to [-127, 127], where the log2 rounding goes
// up exactly when the fp32 significand is >= the first fp32 value above
// sqrt(2) (0x3504F4 in the mantissa field); zero and subnormal absmaxes give
// the smallest scale.  Adding 0x800000 - 0x3504F4 = 0x4AFB0C to the bits
// carries into the exponent field exactly when the mantissa field is
// >= 0x3504F4, so one add and one shift give field + [rounds up]; zero and
// subnormal inputs land at or below -126 - emax and clamp to -127.
__device__ __forceinline__ int e8m0_exponent(float ay, int emax) {
  const int e = (int)((__float_as_uint(ay) + 0x4AFB0Cu) >> 23) - 127 - emax;
  return max(-127, min(127, e));
}

// The same exponent by the plain definition (exponent field, mantissa
// compare, zero/subnormal special case): the reference of the self-check.
__device__ __forceinline__ int e8m0_exponent_by_fields(float ay, int emax) {
  const uint32_t b = __float_as_uint(ay);
  const int field = (int)(b >> 23);
  if (field == 0) return -127;
  const int e = field - 127 + ((b & 0x7FFFFFu) >= 0x3504F4u ? 1 : 0) - emax;
  return max(-127, min(127, e));
}

// ------------------------------------------------------- packed fp32 math
// Two fp32 lanes in one 64-bit register pair (Blackwell f32x2 pipes).

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// bf16 pair (low half = element 0) -> the two fp32 values, exactly.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v) {
  return f2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// The same two constructors in plain integer arithmetic instead of an asm
// register move: the compiler then sees which 32-bit halves form a pair and
// places them without copies.  Measured on GB300: 3-8 % faster in the MX
// kernels, slower in the split-H kernel, which keeps the asm forms.
__device__ __forceinline__ uint64_t f2c(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t bf16x2_to_f2c(uint32_t v) {
  return ((uint64_t)(v & 0xFFFF0000u) << 32) | (uint32_t)(v << 16);
}

// Two E4M3 codes (low byte = element 0) -> their exact fp32 values, via the
// hardware's exact E4M3 -> f16 conversion.
__device__ __forceinline__ uint64_t e4m3x2_to_f2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return f2(lo, hi);
}

// max(|a|, |b|) lane-wise on bf16 pairs; the sign bits of the result are the
// XOR of the inputs' (callers mask them off).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Larger magnitude of the two bf16 halves, as an exact fp32 value.
__device__ __forceinline__ float bf16x2_hmax_abs(uint32_t m) {
  m &= 0x7FFF7FFFu;
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Largest magnitude of the eight fp32 values of four pairs, folded into `m`
// (>= 0): four three-input maxima.
__device__ __forceinline__ float absmax8(float m, const uint64_t (&w)[4]) {
  m = fmax3(m, fabsf(f2_lo(w[0])), fabsf(f2_hi(w[0])));
  m = fmax3(m, fabsf(f2_lo(w[1])), fabsf(f2_hi(w[1])));
  m = fmax3(m, fabsf(f2_lo(w[2])), fabsf(f2_hi(w[2])));
  return fmax3(m, fabsf(f2_lo(w[3])), fabsf(f2_hi(w[3])));
}

__device__ __forceinline__ void st_global_v2(void* p, uint32_t a, uint32_t b) {
  *reinterpret_cast<uint2*>(p) = make_uint2(a, b);
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// 32-byte store (one whole sector; sm_100 and later), p 32-byte aligned.
// No memory clobber: the kernels never read what they store, so shared-
// memory loads may move across it.
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d, uint32_t e, uint32_t f, uint32_t g,
                                             uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a),
               "r"(b), "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h));
}

__device__ __forceinline__ void st_global_u32(void* p, uint32_t a) {
  *reinterpret_cast<uint32_t*>(p) = a;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Sum over aligned groups of `width` lanes (16 or 32, warp-uniform): for 32
// the same steps in the same order as warp_sum.
__device__ __forceinline__ float group_sum(float v, int width) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    if (o < width) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Programmatic dependent launch (PTX griddepcontrol, sm_90+).  A grid
// launched with the programmatic-serialization attribute may start while
// the grid before it in the stream is still running; it must wait here
// before its first global-memory access, until that grid has completed and
// its writes are visible.  For a launch without the attribute the wait
// returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next grid of the stream (if launched with the attribute) be
// scheduled once every CTA of this grid has called this or exited; that
// grid still waits for this one's completion before touching memory.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// fp32(a / 6) for a >= 0 by one multiply and two fmas instead of a division
// (Brisebarre, Muller and Raina, "Accelerating correctly rounded
// floating-point division when the divisor is known in advance", IEEE Trans.
// Computers 53(8), 2004): q = fl(a z) with z = fl(1/6), the remainder a - 6q
// (exact in one fma), then fl(q + r z).  For every finite a >= 0 whose
// quotient is a normal fp32 this is the IEEE quotient (checked for all such
// a); a quotient below 2^-126 may be an ulp off.
__device__ __forceinline__ float div6_rn(float a) {
  const float z = 0x1.555556p-3f;
  const float q = __fmul_rn(a, z);
  const float r = __fmaf_rn(-q, 6.0f, a);
  return __fmaf_rn(r, z, q);
}

// Reciprocals of the E4M3 scale values, for a shared-memory table that the
// threads of a CTA fill before its first nvfp4_scale: rcp[c] = fp32(1 /
// value of code c) for c = 1..126 and 0 for the zero code and the NaN code
// 127.
__device__ __forceinline__ void fill_e4m3_reciprocals(float* rcp, int tid, int nthreads) {
  for (int c = tid; c < 128; c += nthreads)
    rcp[c] = (c == 0 || c == 127) ? 0.f : __frcp_rn(f2_lo(e4m3x2_to_f2((uint16_t)c)));
}

// NVFP4 block scale of a block whose normalized absmax is `ay` (>= 0, not
// NaN): the E4M3 code of fp32(ay / 6) (RNE, saturating at 448; 6 is the
// largest E2M1 magnitude) and, in *inv, the fp32 reciprocal of that code's
// value (0 for a zero scale), read from the table above.  The code equals
// that of the IEEE quotient for every such ay: quotients below 2^-126 give
// code 0 either way, and ay is clamped at 2^32, whose quotient already
// saturates.
__device__ __forceinline__ uint32_t nvfp4_scale(float ay, const float* rcp, float* inv) {
  const uint32_t sc = cvt_e4m3x2(div6_rn(fminf(ay, 0x1p32f)), 0.f) & 0xFFu;
  *inv = rcp[sc];
  return sc;
}

}  // namespace nts
