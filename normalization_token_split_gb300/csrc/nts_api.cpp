// nts_api.cpp -- the C ABI of libnts: argument validation, launch-shape
// selection, status reporting, the host-buffer forms, and the host-side
// computation of the MXNorm correction factor c(B, p).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "nts.h"
#include "nts_debug.h"
#include "nts_internal.h"

namespace nts {

// ------------------------------------------------------------ error state

namespace {
thread_local char g_last_error[512] = "";

std::mutex g_tune_mu;
LaunchTuning g_tune;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(NTS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

void log_launch(const char* name, const char* fmt, ...) {
  static const bool on = [] {
    const char* v = std::getenv("NTS_LOG");
    return v != nullptr && v[0] != '\0' && v[0] != '0';
  }();
  if (!on) return;
  char buf[384];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  std::fprintf(stderr, "[nts] %s: %s\n", name, buf);
}

LaunchTuning current_tuning() {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  return g_tune;
}

std::atomic<int> g_inject_left{0};
std::atomic<int> g_inject_status{NTS_OK};

int take_injected_failure() {
  int left = g_inject_left.load();
  while (left > 0 && !g_inject_left.compare_exchange_weak(left, left - 1)) {
  }
  if (left <= 0) return NTS_OK;
  return fail(g_inject_status.load(), "injected failure (nts_debug_inject_failure), %d left",
              left - 1);
}

// ----------------------------------------------------------- device facts

const DeviceInfo& device_info() {
  static std::mutex mu;
  static std::map<int, DeviceInfo> cache;
  int dev = -1;
  static DeviceInfo bad;
  if (cudaGetDevice(&dev) != cudaSuccess) return bad;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  DeviceInfo d;
  d.device = dev;
  d.ok = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
         cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                dev) == cudaSuccess;
  if (!d.ok) return bad;
  return cache.emplace(dev, d).first->second;
}

RowShape choose_row_shape(int nvec, int force_vpt) {
  // Preference among shapes that waste no thread slots: 4-6 vectors
  // (32-48 values) per thread, then 8, then fewer.
  static const int order[] = {4, 5, 6, 8, 3, 2, 1};
  RowShape best;
  int best_waste = -1;
  for (int vpt : order) {
    if (force_vpt > 0 && vpt != force_vpt) continue;
    int G = (nvec + vpt - 1) / vpt;
    G = (G + 31) / 32 * 32;
    if (G > kMaxConsumers) continue;
    const int waste = G * vpt - nvec;
    if (best_waste < 0 || waste < best_waste) {
      best_waste = waste;
      best.vpt = vpt;
      best.G = G;
    }
  }
  return best;
}

int prepare_kernel(const void* kernel, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int>, size_t> done;
  const int dev = device_info().device;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_tuple(kernel, dev);
  auto it = done.find(key);
  if (it != done.end() && it->second >= smem) return NTS_OK;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return fail_cuda(e, "setting the kernel's shared memory size");
  done[key] = smem;
  return NTS_OK;
}

int kernel_registers(const void* kernel, int* regs) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int>, int> cache;
  const int dev = device_info().device;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_tuple(kernel, dev);
  auto it = cache.find(key);
  if (it == cache.end()) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, kernel);
    if (e != cudaSuccess) return fail_cuda(e, "reading a kernel's attributes");
    it = cache.emplace(key, a.numRegs).first;
  }
  *regs = it->second;
  return NTS_OK;
}

int max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg, int cluster,
                        int64_t* out) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, unsigned, size_t>, int64_t> cache;
  const int dev = device_info().device;
  auto key = std::make_tuple(kernel, dev, cfg.blockDim.x, cfg.dynamicSmemBytes);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return NTS_OK;
    }
  }
  cudaLaunchConfig_t q = cfg;
  q.gridDim = dim3((unsigned)cluster);
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
  if (e != cudaSuccess) return fail_cuda(e, "cluster occupancy query");
  if (n < 1) return fail(NTS_ERR_UNSUPPORTED, "a cluster of %d CTAs cannot be scheduled", cluster);
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  *out = n;
  return NTS_OK;
}

// ------------------------------------------------ correction factor c(B,p)

// c(B, p) = E[M^p]^(-1/p), M the maximum of B i.i.d. |N(0,1)| values.  The
// moment is integrated in its density form,
//   E[M^p] = int_0^inf x^p * B * erf(x/sqrt2)^(B-1) * sqrt(2/pi) exp(-x^2/2) dx,
// by composite 12-point Gauss-Legendre quadrature over 480 panels of [0, 12]
// (the integrand is below 1e-29 beyond 12).  Nodes come from Newton's method
// on the Legendre polynomial.
namespace {

void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
  x.assign(n, 0.0);
  w.assign(n, 0.0);
  const double pi = 3.14159265358979323846;
  for (int i = 0; i < n; ++i) {
    double z = std::cos(pi * (i + 0.75) / (n + 0.5));
    double dp = 0.0;
    for (int it = 0; it < 100; ++it) {
      double p0 = 1.0, p1 = z;
      for (int k = 2; k <= n; ++k) {
        const double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      dp = n * (z * p1 - p0) / (z * z - 1.0);
      const double dz = p1 / dp;
      z -= dz;
      if (std::fabs(dz) < 1e-16) break;
    }
    x[i] = z;
    w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
  }
}

double max_moment(int B, int p) {
  std::vector<double> gx, gw;
  gauss_legendre(12, gx, gw);
  const double c0 = std::sqrt(2.0 / 3.14159265358979323846);
  const int panels = 480;
  const double hi = 12.0, h = hi / panels;
  double total = 0.0;
  for (int k = 0; k < panels; ++k) {
    const double a = k * h, mid = a + 0.5 * h;
    double s = 0.0;
    for (size_t i = 0; i < gx.size(); ++i) {
      const double x = mid + 0.5 * h * gx[i];
      const double F = std::erf(x / std::sqrt(2.0));
      const double dens = B * std::pow(F, B - 1) * c0 * std::exp(-0.5 * x * x);
      s += gw[i] * std::pow(x, p) * dens;
    }
    total += 0.5 * h * s;
  }
  return total;
}

}  // namespace

}  // namespace nts

using namespace nts;

// ------------------------------------------------------------------ C ABI

extern "C" {

int nts_version(void) { return 100; }

const char* nts_status_string(int status) {
  switch (status) {
    case NTS_OK: return "NTS_OK";
    case NTS_ERR_INVALID_ARG: return "NTS_ERR_INVALID_ARG";
    case NTS_ERR_UNSUPPORTED: return "NTS_ERR_UNSUPPORTED";
    case NTS_ERR_CUDA: return "NTS_ERR_CUDA";
    case NTS_ERR_TIMEOUT: return "NTS_ERR_TIMEOUT";
    default: return "NTS_ERR_UNKNOWN";
  }
}

const char* nts_last_error(void) { return g_last_error; }

int nts_mxnorm_correction(int B, int p, double* c_out) {
  if (c_out == nullptr) return fail(NTS_ERR_INVALID_ARG, "c_out is NULL");
  if (B < 1 || B > 4096) return fail(NTS_ERR_INVALID_ARG, "B must be in [1, 4096], got %d", B);
  if (p != 1 && p != 2) return fail(NTS_ERR_INVALID_ARG, "p must be 1 or 2, got %d", p);
  static std::mutex mu;
  static std::map<std::pair<int, int>, double> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_pair(B, p);
  auto it = cache.find(key);
  if (it == cache.end()) {
    const double c = std::pow(max_moment(B, p), -1.0 / p);
    it = cache.emplace(key, c).first;
  }
  *c_out = it->second;
  return NTS_OK;
}

}  // extern "C"

namespace {

int validate_qk(const void* X, const float* gamma, const void* Y, const float* rinv, int64_t T,
                int64_t H, float eps, int N) {
  if (T < 0) return fail(NTS_ERR_INVALID_ARG, "T must be >= 0, got %lld", (long long)T);
  if (T > 0 && (X == nullptr || gamma == nullptr || Y == nullptr))
    return fail(NTS_ERR_INVALID_ARG, "X, gamma and Y must be non-NULL");
  if (H <= 0) return fail(NTS_ERR_INVALID_ARG, "H must be > 0, got %lld", (long long)H);
  if (N != 1 && N != 2 && N != 4 && N != 8)
    return fail(NTS_ERR_INVALID_ARG, "N must be 1, 2, 4 or 8, got %d", N);
  if (H % N != 0)
    return fail(NTS_ERR_INVALID_ARG, "H (%lld) must be a multiple of N (%d)", (long long)H, N);
  if (!(eps > 0.f) || !std::isfinite(eps))
    return fail(NTS_ERR_INVALID_ARG, "eps must be positive and finite");
  if ((H / N) % 8 != 0)
    return fail(NTS_ERR_UNSUPPORTED, "H/N (%lld) must be a multiple of 8", (long long)(H / N));
  if (H / N > 30720)
    return fail(NTS_ERR_UNSUPPORTED, "H/N (%lld) exceeds 30720", (long long)(H / N));
  if (!aligned(X, 16) || !aligned(Y, 16) || !aligned(gamma, 16) ||
      (rinv != nullptr && !aligned(rinv, 4)))
    return fail(NTS_ERR_UNSUPPORTED, "X, Y and gamma must be 16-byte aligned");
  return NTS_OK;
}

}  // namespace

// The checks of an MX call that involve no pointer.
int nts::validate_mx_scalars(int64_t T, int64_t D, float eps, int B, int fmt, int p,
                             bool mxnorm) {
  if (T < 0) return fail(NTS_ERR_INVALID_ARG, "T must be >= 0, got %lld", (long long)T);
  if (D <= 0) return fail(NTS_ERR_INVALID_ARG, "D must be > 0, got %lld", (long long)D);
  if (B != 16 && B != 32 && B != 64)
    return fail(NTS_ERR_INVALID_ARG, "B must be 16, 32 or 64, got %d", B);
  if (D % B != 0)
    return fail(NTS_ERR_INVALID_ARG, "D (%lld) must be a multiple of B (%d)", (long long)D, B);
  if (fmt != NTS_FMT_E4M3 && fmt != NTS_FMT_E2M1 && fmt != NTS_FMT_NVFP4)
    return fail(NTS_ERR_INVALID_ARG, "unknown element format %d", fmt);
  if (fmt == NTS_FMT_NVFP4 && B != 16)
    return fail(NTS_ERR_INVALID_ARG, "NVFP4 blocks have 16 elements, got B = %d", B);
  if (mxnorm && p != 1 && p != 2) return fail(NTS_ERR_INVALID_ARG, "p must be 1 or 2, got %d", p);
  if (!(eps > 0.f) || !std::isfinite(eps))
    return fail(NTS_ERR_INVALID_ARG, "eps must be positive and finite");
  if (D > 32768) return fail(NTS_ERR_UNSUPPORTED, "D (%lld) exceeds 32768", (long long)D);
  return NTS_OK;
}

namespace {

int validate_mx(const void* X, const float* gamma, const uint8_t* codes, const uint8_t* scales,
                const float* rinv, const float* amax, int64_t T, int64_t D, float eps, int B,
                int fmt, int p, bool mxnorm) {
  const int rc = validate_mx_scalars(T, D, eps, B, fmt, p, mxnorm);
  if (rc != NTS_OK) return rc;
  if (T > 0 && (X == nullptr || codes == nullptr || scales == nullptr))
    return fail(NTS_ERR_INVALID_ARG, "X, codes and scales must be non-NULL");
  if (!aligned(X, 16) || !aligned(codes, 16) || (gamma != nullptr && !aligned(gamma, 16)) ||
      (rinv != nullptr && !aligned(rinv, 4)) || (amax != nullptr && !aligned(amax, 4)))
    return fail(NTS_ERR_UNSUPPORTED, "X, gamma and codes must be 16-byte aligned");
  return NTS_OK;
}

int run_mx(const void* X, const float* gamma, uint8_t* codes, uint8_t* scales, float* rinv,
           float* amax, int64_t T, int64_t D, float eps, int B, int fmt, int p, bool mxnorm,
           void* stream, int post = 0) {
  int rc = validate_mx(X, gamma, codes, scales, rinv, amax, T, D, eps, B, fmt, p, mxnorm);
  if (rc != NTS_OK) return rc;
  if (post && fmt == NTS_FMT_NVFP4)
    return fail(NTS_ERR_INVALID_ARG, "post-round MXNorm rounds to E8M0 scales, not NVFP4");
  if (T == 0) return NTS_OK;
  MxRequest rq{X, gamma, codes, scales, rinv, amax, T, D, eps, B, fmt, mxnorm ? p : 0, 0.0, post};
  if (mxnorm) {
    rc = nts_mxnorm_correction(B, p, &rq.corr);
    if (rc != NTS_OK) return rc;
  }
  return launch_mx(rq, static_cast<cudaStream_t>(stream), current_tuning());
}

int copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, void* stream,
         const char* what) {
  if (bytes == 0) return NTS_OK;
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, what);
  return NTS_OK;
}

// ----------------------------------------------- host-buffer forms: pipeline
//
// A host-buffer call moves its rows in chunks through three streams: the
// copies to the device on `in`, the kernels on the caller's stream, the
// copies back on `out`, ordered chunk by chunk with events.  The two copy
// directions then run at once (GB300 NVLink-C2C: ~210 GB/s either way
// alone, ~330 GB/s both ways together) and the kernels hide behind them.
// The caller's stream waits for the last copy back, so the call's effects
// are ordered on that stream exactly as with one stream.

// Chunking: at least kChunkBytes of input per chunk, at most kMaxChunks
// chunks (both adjustable through nts_debug_set_host_chunks).
constexpr int kMaxChunks = 64;                      // capacity of the event arrays
constexpr int kDefaultChunks = 16;   // measured: 8 -> 16 chunks, 269 -> 274 GB/s
constexpr size_t kDefaultChunkBytes = size_t(16) << 20;
std::atomic<int> g_max_chunks{kDefaultChunks};
std::atomic<size_t> g_chunk_bytes{kDefaultChunkBytes};
constexpr int kChunkRows = 16;                     // chunk boundaries: multiples of 16 rows
constexpr int kPipeDevices = 64;

struct HostPipe {
  bool ok = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, finished = nullptr;
  cudaEvent_t loaded[kMaxChunks] = {}, done[kMaxChunks] = {};
};

// Serializes the enqueue sequences of host-buffer calls, which share the
// per-device streams and events (a wait refers to the event's record at the
// time it is enqueued, so reusing the events for the next call is safe).
std::mutex g_pipe_mu;
HostPipe g_pipe[kPipeDevices];

int host_pipe(HostPipe** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "querying the current device");
  if (dev < 0 || dev >= kPipeDevices)
    return fail(NTS_ERR_UNSUPPORTED, "device %d beyond the %d the host-buffer forms serve", dev,
                kPipeDevices);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ok) {
    const unsigned ef = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.finished, ef);
    for (int k = 0; k < kMaxChunks && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&hp.loaded[k], ef);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done[k], ef);
    }
    if (e != cudaSuccess) return fail_cuda(e, "creating the host-buffer copy streams");
    hp.ok = true;
  }
  *out = &hp;
  return NTS_OK;
}

// Runs a host-buffer call over T rows: copy_in(r0, r1, stream) enqueues the
// copies of rows [r0, r1) to the device, kernel(r0, r1, stream) the
// computation, copy_out(r0, r1, stream) the copies back.  One chunk (small
// calls) runs everything on the caller's stream.
template <typename In, typename Kernel, typename Out>
int run_host_pipeline(int64_t T, size_t in_bytes_per_row, void* stream, In copy_in,
                      Kernel kernel, Out copy_out) {
  const size_t chunk_bytes = g_chunk_bytes.load();
  int nchunks = (int)std::min<size_t>((size_t)g_max_chunks.load(), (T * in_bytes_per_row) / chunk_bytes);
  nchunks = std::max(1, std::min<int>(nchunks, (int)((T + kChunkRows - 1) / kChunkRows)));
  if (nchunks == 1) {
    int rc = copy_in(0, T, stream);
    if (rc == NTS_OK) rc = kernel(0, T, stream);
    if (rc == NTS_OK) rc = copy_out(0, T, stream);
    return rc;
  }
  int64_t rows = (T + nchunks - 1) / nchunks;
  rows = (rows + kChunkRows - 1) / kChunkRows * kChunkRows;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = nullptr;
  int rc = host_pipe(&hp);
  if (rc != NTS_OK) return rc;
  cudaError_t e = cudaEventRecord(hp->start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->start, 0);
  if (e != cudaSuccess) return fail_cuda(e, "ordering the copy streams after the caller's work");
  int k = 0;
  for (int64_t r0 = 0; r0 < T; r0 += rows, ++k) {
    const int64_t r1 = std::min(T, r0 + rows);
    rc = copy_in(r0, r1, hp->in);
    if (rc != NTS_OK) return rc;
    e = cudaEventRecord(hp->loaded[k], hp->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->loaded[k], 0);
    if (e != cudaSuccess) return fail_cuda(e, "ordering a chunk's kernel after its copy");
    rc = kernel(r0, r1, stream);
    if (rc != NTS_OK) return rc;
    e = cudaEventRecord(hp->done[k], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->done[k], 0);
    if (e != cudaSuccess) return fail_cuda(e, "ordering a chunk's copy back after its kernel");
    rc = copy_out(r0, r1, hp->out);
    if (rc != NTS_OK) return rc;
  }
  e = cudaEventRecord(hp->finished, hp->out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->finished, 0);
  if (e != cudaSuccess) return fail_cuda(e, "ordering the caller's stream after the copies");
  return NTS_OK;
}

}  // namespace

extern "C" {

int nts_qknorm_rms(const void* X_dev, const float* gamma_dev, void* Y_dev, float* rinv_dev,
                   int64_t T, int64_t H, float eps, int N, void* stream) {
  int rc = validate_qk(X_dev, gamma_dev, Y_dev, rinv_dev, T, H, eps, N);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  const QkRequest rq{X_dev, gamma_dev, Y_dev, rinv_dev, T, H};
  return launch_qknorm(&rq, 1, eps, N, QkOptions{}, static_cast<cudaStream_t>(stream),
                       current_tuning());
}

int nts_qknorm_rms_fp8(const void* X_dev, float x_scale, const float* gamma_dev, void* Y_dev,
                       float* rinv_dev, int64_t T, int64_t H, float eps, int N, void* stream) {
  int rc = validate_qk(X_dev, gamma_dev, Y_dev, rinv_dev, T, H, eps, N);
  if (rc != NTS_OK) return rc;
  if (!(x_scale > 0.f) || !std::isfinite(x_scale))
    return fail(NTS_ERR_INVALID_ARG, "x_scale must be positive and finite");
  if ((H / N) % 16 != 0)
    return fail(NTS_ERR_UNSUPPORTED, "H/N (%lld) must be a multiple of 16 for E4M3 rows",
                (long long)(H / N));
  if (T == 0) return NTS_OK;
  const QkRequest rq{X_dev, gamma_dev, Y_dev, rinv_dev, T, H};
  QkOptions opt;
  opt.in_e4m3 = 1;
  opt.x_scale = x_scale;
  return launch_qknorm(&rq, 1, eps, N, opt, static_cast<cudaStream_t>(stream), current_tuning());
}

int nts_qknorm_rms_heads(const void* X_dev, const float* gamma_dev, void* Y_dev,
                         float* rinv_dev, int64_t T, int64_t H, int64_t head_dim, float eps,
                         int N, void* stream) {
  if (head_dim <= 0) return fail(NTS_ERR_INVALID_ARG, "head_dim must be > 0");
  if (H <= 0 || H % head_dim != 0)
    return fail(NTS_ERR_INVALID_ARG, "H (%lld) must be a positive multiple of head_dim (%lld)",
                (long long)H, (long long)head_dim);
  if (T < 0) return fail(NTS_ERR_INVALID_ARG, "T must be >= 0, got %lld", (long long)T);
  // Row-major [T, H] is row-major [T * nheads, head_dim]: one row per head.
  const int64_t rows = T * (H / head_dim);
  int rc = validate_qk(X_dev, gamma_dev, Y_dev, rinv_dev, rows, head_dim, eps, N);
  if (rc != NTS_OK) return rc;
  if (rows == 0) return NTS_OK;
  // Heads kept whole in one CTA when N == 1 (no statistic leaves a warp);
  // otherwise every head is split across the N CTAs of a cluster.
  if (heads_whole_path(H, head_dim, N))
    return launch_heads(X_dev, gamma_dev, Y_dev, rinv_dev, T, H, head_dim, eps,
                        static_cast<cudaStream_t>(stream), current_tuning());
  const QkRequest rq{X_dev, gamma_dev, Y_dev, rinv_dev, rows, head_dim};
  return launch_qknorm(&rq, 1, eps, N, QkOptions{}, static_cast<cudaStream_t>(stream),
                       current_tuning());
}

int nts_layernorm_split(const void* X_dev, const float* gamma_dev, const float* beta_dev,
                        void* Y_dev, float* mean_dev, float* rstd_dev, int64_t T, int64_t H,
                        float eps, int N, void* stream) {
  int rc = validate_qk(X_dev, gamma_dev, Y_dev, rstd_dev, T, H, eps, N);
  if (rc != NTS_OK) return rc;
  if (beta_dev != nullptr && !aligned(beta_dev, 16))
    return fail(NTS_ERR_UNSUPPORTED, "beta must be 16-byte aligned");
  if (mean_dev != nullptr && !aligned(mean_dev, 4))
    return fail(NTS_ERR_UNSUPPORTED, "mean must be 4-byte aligned");
  if (beta_dev != nullptr && H / N > 20480)
    return fail(NTS_ERR_UNSUPPORTED, "H/N (%lld) exceeds 20480 with beta", (long long)(H / N));
  if (T == 0) return NTS_OK;
  QkRequest rq{X_dev, gamma_dev, Y_dev, rstd_dev, T, H};
  rq.beta = beta_dev;
  rq.mean = mean_dev;
  QkOptions opt;
  opt.layernorm = 1;
  return launch_qknorm(&rq, 1, eps, N, opt, static_cast<cudaStream_t>(stream), current_tuning());
}

int nts_qknorm_rms_qk(const void* Q_dev, const float* gamma_q_dev, void* Yq_dev,
                      float* rinv_q_dev, const void* K_dev, const float* gamma_k_dev,
                      void* Yk_dev, float* rinv_k_dev, int64_t T, int64_t Hq, int64_t Hk,
                      float eps, int N, void* stream) {
  int rc = validate_qk(Q_dev, gamma_q_dev, Yq_dev, rinv_q_dev, T, Hq, eps, N);
  if (rc != NTS_OK) return rc;
  rc = validate_qk(K_dev, gamma_k_dev, Yk_dev, rinv_k_dev, T, Hk, eps, N);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  const QkRequest rq[2] = {{Q_dev, gamma_q_dev, Yq_dev, rinv_q_dev, T, Hq},
                           {K_dev, gamma_k_dev, Yk_dev, rinv_k_dev, T, Hk}};
  return launch_qknorm(rq, 2, eps, N, QkOptions{}, static_cast<cudaStream_t>(stream),
                       current_tuning());
}

}  // extern "C"

namespace {

int validate_qk_mx(const void* X_dev, const float* gamma_dev, uint8_t* codes_dev,
                   uint8_t* scales_dev, float* rinv_dev, int64_t T, int64_t H, float eps, int N,
                   int B, int fmt) {
  int rc = validate_qk(X_dev, gamma_dev, codes_dev, rinv_dev, T, H, eps, N);
  if (rc != NTS_OK) return rc;
  if (T > 0 && scales_dev == nullptr) return fail(NTS_ERR_INVALID_ARG, "scales must be non-NULL");
  if (B != 16 && B != 32 && B != 64)
    return fail(NTS_ERR_INVALID_ARG, "B must be 16, 32 or 64, got %d", B);
  if (fmt != NTS_FMT_E4M3 && fmt != NTS_FMT_E2M1 && fmt != NTS_FMT_NVFP4)
    return fail(NTS_ERR_INVALID_ARG, "unknown element format %d", fmt);
  if (fmt == NTS_FMT_NVFP4 && B != 16)
    return fail(NTS_ERR_INVALID_ARG, "NVFP4 blocks have 16 elements, got B = %d", B);
  if ((H / N) % B != 0)
    return fail(NTS_ERR_UNSUPPORTED, "H/N (%lld) must be a multiple of B (%d)",
                (long long)(H / N), B);
  return NTS_OK;
}

}  // namespace

extern "C" {

int nts_qknorm_rms_mxcast(const void* X_dev, const float* gamma_dev, uint8_t* codes_dev,
                          uint8_t* scales_dev, float* rinv_dev, int64_t T, int64_t H, float eps,
                          int N, int B, int fmt, void* stream) {
  int rc = validate_qk_mx(X_dev, gamma_dev, codes_dev, scales_dev, rinv_dev, T, H, eps, N, B, fmt);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  QkRequest rq{X_dev, gamma_dev, nullptr, rinv_dev, T, H};
  rq.codes = codes_dev;
  rq.scales = scales_dev;
  QkOptions opt;
  opt.out_fmt = fmt;
  opt.B = B;
  return launch_qknorm(&rq, 1, eps, N, opt, static_cast<cudaStream_t>(stream), current_tuning());
}

int nts_qknorm_rms_qk_mxcast(const void* Q_dev, const float* gamma_q_dev, uint8_t* codes_q_dev,
                             uint8_t* scales_q_dev, float* rinv_q_dev, const void* K_dev,
                             const float* gamma_k_dev, uint8_t* codes_k_dev,
                             uint8_t* scales_k_dev, float* rinv_k_dev, int64_t T, int64_t Hq,
                             int64_t Hk, float eps, int N, int B, int fmt, void* stream) {
  int rc = validate_qk_mx(Q_dev, gamma_q_dev, codes_q_dev, scales_q_dev, rinv_q_dev, T, Hq, eps,
                          N, B, fmt);
  if (rc != NTS_OK) return rc;
  rc = validate_qk_mx(K_dev, gamma_k_dev, codes_k_dev, scales_k_dev, rinv_k_dev, T, Hk, eps, N,
                      B, fmt);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  QkRequest rq[2] = {{Q_dev, gamma_q_dev, nullptr, rinv_q_dev, T, Hq},
                     {K_dev, gamma_k_dev, nullptr, rinv_k_dev, T, Hk}};
  rq[0].codes = codes_q_dev;
  rq[0].scales = scales_q_dev;
  rq[1].codes = codes_k_dev;
  rq[1].scales = scales_k_dev;
  QkOptions opt;
  opt.out_fmt = fmt;
  opt.B = B;
  return launch_qknorm(rq, 2, eps, N, opt, static_cast<cudaStream_t>(stream), current_tuning());
}

int nts_rmsnorm_mxcast(const void* X_dev, const float* gamma_dev, uint8_t* codes_dev,
                       uint8_t* scales_dev, float* rinv_dev, float* amax_dev, int64_t T, int64_t D,
                       float eps, int B, int fmt, void* stream) {
  return run_mx(X_dev, gamma_dev, codes_dev, scales_dev, rinv_dev, amax_dev, T, D, eps, B, fmt,
                0, false, stream);
}

int nts_mxnorm_cast(const void* X_dev, const float* gamma_dev, uint8_t* codes_dev,
                    uint8_t* scales_dev, float* rinv_dev, float* amax_dev, int64_t T, int64_t D,
                    float eps, int B, int fmt, int p, void* stream) {
  return run_mx(X_dev, gamma_dev, codes_dev, scales_dev, rinv_dev, amax_dev, T, D, eps, B, fmt,
                p, true, stream);
}

int nts_mxnorm_postround_cast(const void* X_dev, const float* gamma_dev, uint8_t* codes_dev,
                              uint8_t* scales_dev, float* rinv_dev, float* amax_dev, int64_t T,
                              int64_t D, float eps, int B, int fmt, int p, void* stream) {
  return run_mx(X_dev, gamma_dev, codes_dev, scales_dev, rinv_dev, amax_dev, T, D, eps, B, fmt,
                p, true, stream, 1);
}

int nts_check_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "synchronizing the stream");
  unsigned qk = 0, mx = 0;
  int rc = read_and_clear_qk_status(&qk);
  if (rc != NTS_OK) return rc;
  rc = read_and_clear_mx_status(&mx);
  if (rc != NTS_OK) return rc;
  if ((qk | mx) != 0)
    return fail(NTS_ERR_TIMEOUT, "a kernel gave up on a bounded wait (qk=%u mx=%u)", qk, mx);
  return NTS_OK;
}

int nts_qknorm_rms_host(const void* X_host, const float* gamma_dev, void* Y_host,
                        float* rinv_host, void* X_dev, void* Y_dev, float* rinv_dev, int64_t T,
                        int64_t H, float eps, int N, void* stream) {
  if (T > 0 && (X_host == nullptr || Y_host == nullptr))
    return fail(NTS_ERR_INVALID_ARG, "X_host and Y_host must be non-NULL");
  if (rinv_host != nullptr && rinv_dev == nullptr)
    return fail(NTS_ERR_INVALID_ARG, "rinv_host needs a rinv_dev staging buffer");
  float* rinv_k = rinv_host != nullptr ? rinv_dev : nullptr;
  int rc = validate_qk(X_dev, gamma_dev, Y_dev, rinv_k, T, H, eps, N);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  const size_t rb = (size_t)H * 2;  // bytes per row
  auto at = [rb](const void* base, int64_t r) {
    return static_cast<const char*>(base) + (size_t)r * rb;
  };
  auto in = [&](int64_t r0, int64_t r1, void* st) {
    return copy(const_cast<char*>(at(X_dev, r0)), at(X_host, r0), (size_t)(r1 - r0) * rb,
                cudaMemcpyHostToDevice, st, "copying X to the device");
  };
  auto kern = [&](int64_t r0, int64_t r1, void* st) {
    return nts_qknorm_rms(at(X_dev, r0), gamma_dev, const_cast<char*>(at(Y_dev, r0)),
                          rinv_k != nullptr ? rinv_k + r0 : nullptr, r1 - r0, H, eps, N, st);
  };
  auto out = [&](int64_t r0, int64_t r1, void* st) {
    int c = copy(const_cast<char*>(at(Y_host, r0)), at(Y_dev, r0), (size_t)(r1 - r0) * rb,
                 cudaMemcpyDeviceToHost, st, "copying Y to the host");
    if (c == NTS_OK && rinv_host != nullptr)
      c = copy(rinv_host + r0, rinv_dev + r0, (size_t)(r1 - r0) * 4, cudaMemcpyDeviceToHost, st,
               "copying rinv to the host");
    return c;
  };
  return run_host_pipeline(T, rb, stream, in, kern, out);
}

// one_stream: every copy and the kernel on the caller's stream, in one piece
// (no chunking, so the pipeline's own streams and events are never needed).
int nts_qknorm_rms_qk_host(const void* Q_host, const float* gamma_q_dev, void* Yq_host,
                           const void* K_host, const float* gamma_k_dev, void* Yk_host,
                           void* Q_dev, void* Yq_dev, void* K_dev, void* Yk_dev, int64_t T,
                           int64_t Hq, int64_t Hk, float eps, int N, void* stream) {
  if (T > 0 && (Q_host == nullptr || Yq_host == nullptr || K_host == nullptr ||
                Yk_host == nullptr))
    return fail(NTS_ERR_INVALID_ARG, "Q_host, Yq_host, K_host and Yk_host must be non-NULL");
  int rc = validate_qk(Q_dev, gamma_q_dev, Yq_dev, nullptr, T, Hq, eps, N);
  if (rc != NTS_OK) return rc;
  rc = validate_qk(K_dev, gamma_k_dev, Yk_dev, nullptr, T, Hk, eps, N);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  const size_t qb = (size_t)Hq * 2, kb = (size_t)Hk * 2;  // bytes per row
  auto at = [](const void* base, size_t rb, int64_t r) {
    return const_cast<char*>(static_cast<const char*>(base) + (size_t)r * rb);
  };
  auto in = [&](int64_t r0, int64_t r1, void* st) {
    int c = copy(at(Q_dev, qb, r0), at(Q_host, qb, r0), (size_t)(r1 - r0) * qb,
                 cudaMemcpyHostToDevice, st, "copying Q to the device");
    if (c == NTS_OK)
      c = copy(at(K_dev, kb, r0), at(K_host, kb, r0), (size_t)(r1 - r0) * kb,
               cudaMemcpyHostToDevice, st, "copying K to the device");
    return c;
  };
  auto kern = [&](int64_t r0, int64_t r1, void* st) {
    return nts_qknorm_rms_qk(at(Q_dev, qb, r0), gamma_q_dev, at(Yq_dev, qb, r0), nullptr,
                             at(K_dev, kb, r0), gamma_k_dev, at(Yk_dev, kb, r0), nullptr, r1 - r0,
                             Hq, Hk, eps, N, st);
  };
  auto out = [&](int64_t r0, int64_t r1, void* st) {
    int c = copy(at(Yq_host, qb, r0), at(Yq_dev, qb, r0), (size_t)(r1 - r0) * qb,
                 cudaMemcpyDeviceToHost, st, "copying Yq to the host");
    if (c == NTS_OK)
      c = copy(at(Yk_host, kb, r0), at(Yk_dev, kb, r0), (size_t)(r1 - r0) * kb,
               cudaMemcpyDeviceToHost, st, "copying Yk to the host");
    return c;
  };
  return run_host_pipeline(T, qb + kb, stream, in, kern, out);
}

static int mx_host(const void* X_host, const float* gamma_dev, uint8_t* codes_host,
                   uint8_t* scales_host, void* X_dev, uint8_t* codes_dev, uint8_t* scales_dev,
                   int64_t T, int64_t D, float eps, int B, int fmt, int p, bool mxnorm,
                   void* stream, bool one_stream = false) {
  if (T > 0 && (X_host == nullptr || codes_host == nullptr || scales_host == nullptr))
    return fail(NTS_ERR_INVALID_ARG, "X_host, codes_host and scales_host must be non-NULL");
  int rc = validate_mx(X_dev, gamma_dev, codes_dev, scales_dev, nullptr, nullptr, T, D, eps, B,
                       fmt, p, mxnorm);
  if (rc != NTS_OK) return rc;
  if (T == 0) return NTS_OK;
  const size_t xr = (size_t)D * 2;                                   // bytes per row
  const size_t cr = (size_t)(fmt == NTS_FMT_E4M3 ? D : D / 2);
  const size_t sr = (size_t)(D / B);
  auto in = [&](int64_t r0, int64_t r1, void* st) {
    return copy(static_cast<char*>(X_dev) + r0 * xr, static_cast<const char*>(X_host) + r0 * xr,
                (size_t)(r1 - r0) * xr, cudaMemcpyHostToDevice, st, "copying X to the device");
  };
  auto kern = [&](int64_t r0, int64_t r1, void* st) {
    return run_mx(static_cast<const char*>(X_dev) + r0 * xr, gamma_dev, codes_dev + r0 * cr,
                  scales_dev + r0 * sr, nullptr, nullptr, r1 - r0, D, eps, B, fmt, p, mxnorm, st);
  };
  auto out = [&](int64_t r0, int64_t r1, void* st) {
    int c = copy(codes_host + r0 * cr, codes_dev + r0 * cr, (size_t)(r1 - r0) * cr,
                 cudaMemcpyDeviceToHost, st, "copying codes to the host");
    if (c == NTS_OK)
      c = copy(scales_host + r0 * sr, scales_dev + r0 * sr, (size_t)(r1 - r0) * sr,
               cudaMemcpyDeviceToHost, st, "copying scales to the host");
    return c;
  };
  if (one_stream) {
    rc = in(0, T, stream);
    if (rc == NTS_OK) rc = kern(0, T, stream);
    if (rc == NTS_OK) rc = out(0, T, stream);
    return rc;
  }
  return run_host_pipeline(T, xr, stream, in, kern, out);
}

int nts_rmsnorm_mxcast_host(const void* X_host, const float* gamma_dev, uint8_t* codes_host,
                            uint8_t* scales_host, void* X_dev, uint8_t* codes_dev,
                            uint8_t* scales_dev, int64_t T, int64_t D, float eps, int B, int fmt,
                            void* stream) {
  return mx_host(X_host, gamma_dev, codes_host, scales_host, X_dev, codes_dev, scales_dev, T, D,
                 eps, B, fmt, 0, false, stream);
}

int nts_mxnorm_cast_host(const void* X_host, const float* gamma_dev, uint8_t* codes_host,
                         uint8_t* scales_host, void* X_dev, uint8_t* codes_dev,
                         uint8_t* scales_dev, int64_t T, int64_t D, float eps, int B, int fmt,
                         int p, void* stream) {
  return mx_host(X_host, gamma_dev, codes_host, scales_host, X_dev, codes_dev, scales_dev, T, D,
                 eps, B, fmt, p, true, stream);
}

}  // extern "C"

int nts::mxnorm_cast_host_one_stream(const void* X_host, const float* gamma_dev,
                                     uint8_t* codes_host, uint8_t* scales_host, void* X_dev,
                                     uint8_t* codes_dev, uint8_t* scales_dev, int64_t T,
                                     int64_t D, float eps, int B, int fmt, int p, void* stream) {
  return mx_host(X_host, gamma_dev, codes_host, scales_host, X_dev, codes_dev, scales_dev, T, D,
                 eps, B, fmt, p, true, stream, true);
}

extern "C" {

// ------------------------------------------------------------- debug hooks

int nts_debug_set_tuning(int vpt, int rows, int stages, int64_t grid, int smem_budget) {
  if (vpt < 0 || rows < 0 || stages < 0 || grid < 0 || smem_budget < 0)
    return fail(NTS_ERR_INVALID_ARG, "tuning values must be >= 0");
  if (vpt > 8) return fail(NTS_ERR_INVALID_ARG, "vpt %d unsupported", vpt);
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.force_vpt = vpt;
  g_tune.force_rows = rows;
  g_tune.force_stages = stages;
  g_tune.force_grid = grid;
  g_tune.smem_budget = smem_budget > 0 ? smem_budget : LaunchTuning().smem_budget;
  return NTS_OK;
}

int nts_debug_set_wait_limit_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.wait_limit_ns = ns > 0 ? ns : LaunchTuning().wait_limit_ns;
  return NTS_OK;
}

int nts_debug_set_schedule(int dynamic) {
  if (dynamic != 0 && dynamic != 1) return fail(NTS_ERR_INVALID_ARG, "dynamic must be 0 or 1");
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.dynamic = dynamic;
  return NTS_OK;
}

int nts_debug_set_direct(int on) {
  if (on != 0 && on != 1) return fail(NTS_ERR_INVALID_ARG, "on must be 0 or 1");
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.direct = on;
  return NTS_OK;
}

int nts_debug_set_host_chunks(int max_chunks, int64_t min_chunk_bytes) {
  if (max_chunks < 0 || max_chunks > kMaxChunks || min_chunk_bytes < 0)
    return fail(NTS_ERR_INVALID_ARG, "max_chunks must be in [0, %d] and min_chunk_bytes >= 0",
                kMaxChunks);
  g_max_chunks = max_chunks == 0 ? kDefaultChunks : max_chunks;
  g_chunk_bytes = min_chunk_bytes == 0 ? kDefaultChunkBytes : (size_t)min_chunk_bytes;
  return NTS_OK;
}

int nts_debug_inject_failure(int status, int count) {
  if (count < 0) return fail(NTS_ERR_INVALID_ARG, "count must be >= 0");
  if (count > 0 && status != NTS_ERR_CUDA && status != NTS_ERR_UNSUPPORTED &&
      status != NTS_ERR_TIMEOUT)
    return fail(NTS_ERR_INVALID_ARG, "status must be NTS_ERR_CUDA, _UNSUPPORTED or _TIMEOUT");
  g_inject_status = status;
  g_inject_left = count;
  return NTS_OK;
}

int nts_debug_set_pdl(int on) {
  if (on != 0 && on != 1) return fail(NTS_ERR_INVALID_ARG, "on must be 0 or 1");
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.pdl = on;
  return NTS_OK;
}

int nts_debug_set_missing_tx(uint32_t bytes) {
  if (bytes % 16 != 0) return fail(NTS_ERR_INVALID_ARG, "bytes must be a multiple of 16");
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.missing_tx = bytes;
  return NTS_OK;
}

}  // extern "C"
