/*
 * nts.h -- C ABI of libnts, GB300 (sm_103a) kernels for per-token RMS
 * normalization: split-H layerwise QK-RMSNorm, fused RMSNorm + MX cast, and
 * MXNorm + MX cast.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named *_dev are device pointers (cudaMalloc'd, or owned by a
 *    framework such as PyTorch); pointers named *_host are host pointers
 *    (pinned memory gives asynchronous copies).  Entry points without a
 *    suffix take device pointers only.  The caller owns every buffer; the
 *    library allocates no device memory at run time.  Its static device
 *    state: one status word per kernel family, a 512 KB pool of tile
 *    counters (a pair per stream, and one per launch recorded into a CUDA
 *    graph), and the 16 MiB staging array of nts_mxnorm_cast_host_noalloc.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls only enqueue work and return; results are ready once
 *    the stream has reached that point.  Kernels are launched as
 *    programmatic dependents: one may be scheduled while the previous
 *    kernel in the stream drains, but it touches no global memory before
 *    that kernel has completed, so stream order holds as usual.
 *  - Matrices are row-major with one token per row: element (t, j) of a
 *    [T, H] matrix is at index t*H + j.  bf16 means IEEE-style bfloat16
 *    (uint16 storage).  Device pointers must be 16-byte aligned.
 *  - Return value: an nts_status.  Nothing is launched when the status is
 *    not NTS_OK, and no call aborts or throws.  nts_last_error() gives a
 *    human-readable detail for the calling thread.
 *  - T == 0 is valid and launches nothing; the data pointers may then be
 *    NULL (an empty tensor's storage), the other arguments are still checked.
 *
 * Sources (web pages), by title and section:
 *   SwiftQK: Fast and Communication-Efficient Tensor Parallelism for
 *   Query-Key Normalization (IEEE CAL) -- Eq. (1), Sec. III.A-D, Algorithm 1;
 *   the SwiftQK reading notes (zhongzhuzhou.org) -- Eq. (1), Sec. 3, Sec. 4b;
 *   the MXNorm paper card (arXiv 2603.13180) -- abstract, Fig. 1 caption,
 *   Fig. 8, Fig. A.1.
 */
#ifndef NTS_H
#define NTS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NTS_API __attribute__((visibility("default")))
#else
#define NTS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NTS_OK = 0,
    NTS_ERR_INVALID_ARG = 1, /* null required pointer, bad size/shape/eps/N/B/fmt/p */
    NTS_ERR_UNSUPPORTED = 2, /* valid request this build cannot run: misaligned
                                pointer, row too wide, cluster not launchable */
    NTS_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    NTS_ERR_TIMEOUT = 4      /* a kernel's bounded wait expired (nts_check_status) */
} nts_status;

typedef enum {
    NTS_FMT_E4M3 = 0, /* OCP E4M3: 1 byte per element, max 448; E8M0 scales (MXFP8) */
    NTS_FMT_E2M1 = 1, /* OCP E2M1: 4 bits per element, max 6; E8M0 scales (MXFP4) */
    NTS_FMT_NVFP4 = 2 /* E2M1 elements, B = 16, one E4M3 scale per block (NVFP4) */
} nts_elem_fmt;

/* Library version, major*10000 + minor*100 + patch. */
NTS_API int nts_version(void);

/* Static string naming a status code. */
NTS_API const char *nts_status_string(int status);

/* Detail of the calling thread's most recent failure ("" if none). */
NTS_API const char *nts_last_error(void);

/*
 * nts_qknorm_rms -- layerwise QK-RMSNorm of every token row, computed as
 * split-H scalar partial sums (SwiftQK Eq. (1) and Algorithm 1):
 *
 *     S_k    = sum over columns [k*H/N, (k+1)*H/N) of x_j^2    (Phase A, fp32)
 *     S      = S_0 + ... + S_{N-1}                            (rank order)
 *     rinv   = 1 / sqrt(S / H + eps)          (H is the FULL row width)
 *     y_j    = bf16_rne((x_j * gamma_j) * rinv)                (Phases B, C)
 *
 * The N shards of a row are N CTAs of one thread-block cluster; each keeps
 * its shard on chip, exchanges its partial sum through distributed shared
 * memory, and forms x*gamma while the exchange is in flight.  N changes only
 * the work decomposition and the fp32 summation order, never the result's
 * definition.
 *
 *   X_dev      bf16 [T, H], read.            gamma_dev  fp32 [H], read.
 *   Y_dev      bf16 [T, H], written.  Y_dev == X_dev (in place) is allowed;
 *              any other overlap is undefined.
 *   rinv_dev   fp32 [T], written, or NULL.
 *   T >= 0; H >= 8; H % N == 0; (H / N) % 8 == 0; H / N <= 30720;
 *   eps > 0 and finite; N in {1, 2, 4, 8}.
 * Errors: INVALID_ARG (null X/gamma/Y, T < 0, H <= 0, H % N, bad eps or N),
 *         UNSUPPORTED ((H/N) % 8 != 0, slice too wide, unaligned pointer,
 *         cluster shape not launchable), CUDA (launch failure).
 */
NTS_API int nts_qknorm_rms(const void *X_dev, const float *gamma_dev, void *Y_dev,
                   float *rinv_dev, int64_t T, int64_t H, float eps, int N,
                   void *stream);

/*
 * nts_qknorm_rms_fp8 -- nts_qknorm_rms on FP8-E4M3 activations (SwiftQK
 * Sec. IV.C evaluates bf16 and FP8-E4M3 activations; the squares and the
 * combine stay fp32).  X_dev holds OCP E4M3 codes, uint8 [T, H]; the
 * activation is code * x_scale (a per-tensor dequantization scale, > 0 and
 * finite).  gamma, Y (bf16), rinv, N and the errors are those of
 * nts_qknorm_rms, plus UNSUPPORTED when (H / N) % 16 != 0 (a shard's row must
 * be a whole number of 16-byte vectors).  Y must not overlap X.
 */
NTS_API int nts_qknorm_rms_fp8(const void *X_dev, float x_scale, const float *gamma_dev,
                               void *Y_dev, float *rinv_dev, int64_t T, int64_t H, float eps,
                               int N, void *stream);

/*
 * nts_qknorm_rms_heads -- headwise QK-Norm (SwiftQK Sec. II.A: one
 * normalization factor per attention head instead of one per projected
 * vector).  X holds T tokens of H = nheads * head_dim values, the heads one
 * after another; head h of token t is normalized over its own head_dim
 * values:  rinv[t][h] = 1/sqrt((1/head_dim) sum x^2 + eps),
 * y = bf16_rne((x * gamma) * rinv), with gamma of head_dim entries shared by
 * all heads.  N splits every head across the CTAs of a cluster exactly as in
 * nts_qknorm_rms (head_dim % N == 0, (head_dim / N) % 8 == 0).
 *   X_dev, Y_dev  bf16 [T, H] (in place allowed); gamma_dev fp32 [head_dim];
 *   rinv_dev      fp32 [T, H/head_dim] or NULL.
 * Errors: as nts_qknorm_rms, plus INVALID_ARG for head_dim <= 0 or
 * H % head_dim != 0.
 */
NTS_API int nts_qknorm_rms_heads(const void *X_dev, const float *gamma_dev, void *Y_dev,
                                 float *rinv_dev, int64_t T, int64_t H, int64_t head_dim,
                                 float eps, int N, void *stream);

/*
 * nts_layernorm_split -- LayerNorm with the split-H statistic exchange
 * (SwiftQK reading notes, Sec. 5e: the variance is (1/H) sum x^2 - mu^2, so
 * a shard needs only two additive scalars, its sum and its sum of squares,
 * and the Phase A/B/C structure of nts_qknorm_rms carries over with two
 * scalars per shard instead of one):
 *
 *     s1_k, s2_k = sums over shard k of x_j and x_j^2            (fp32)
 *     mu    = (s1_0 + ... + s1_{N-1}) / H
 *     var   = max((s2_0 + ... + s2_{N-1}) / H - mu^2, 0)
 *     rstd  = 1 / sqrt(var + eps)
 *     y_j   = bf16_rne((x_j * rstd - mu * rstd) * gamma_j + beta_j)
 *
 * which is (x_j - mu) * rstd * gamma_j + beta_j (fp32 fused multiply-adds).  The one-pass variance
 * loses relative accuracy when |mu| is large against the spread of the row
 * (fp32 cancellation in s2/H - mu^2); the pages' formulation is kept.
 *   X_dev      bf16 [T, H], read.     gamma_dev  fp32 [H], read.
 *   beta_dev   fp32 [H], read, or NULL (no shift).
 *   Y_dev      bf16 [T, H], written (Y == X allowed).
 *   mean_dev   fp32 [T], written, or NULL.   rstd_dev  fp32 [T], or NULL.
 *   Limits as nts_qknorm_rms, except H / N <= 20480 when beta is given (the
 *   shard's gamma and beta both stay in shared memory).
 * Errors: as nts_qknorm_rms.
 */
NTS_API int nts_layernorm_split(const void *X_dev, const float *gamma_dev,
                                const float *beta_dev, void *Y_dev, float *mean_dev,
                                float *rstd_dev, int64_t T, int64_t H, float eps, int N,
                                void *stream);

/*
 * nts_qknorm_rms_qk -- nts_qknorm_rms of a token batch's Q and K in ONE
 * launch (one persistent grid walks the tiles of both tensors).  Q and K may
 * have different widths (Hq, Hk: e.g. grouped-query attention, where K is
 * narrower) and their own gains; they share T, eps and N.  Each tensor obeys
 * the argument rules of nts_qknorm_rms (in-place Yq == Q, Yk == K allowed;
 * rinv_* nullable); the same errors apply.  Layerwise QK-Norm normalizes Q
 * and K separately (SwiftQK Sec. II.A); fusing the two calls halves the
 * launches, which dominate at decode sizes.
 */
NTS_API int nts_qknorm_rms_qk(const void *Q_dev, const float *gamma_q_dev, void *Yq_dev,
                              float *rinv_q_dev, const void *K_dev,
                              const float *gamma_k_dev, void *Yk_dev, float *rinv_k_dev,
                              int64_t T, int64_t Hq, int64_t Hk, float eps, int N,
                              void *stream);

/*
 * nts_qknorm_rms_mxcast -- layerwise QK-RMSNorm with the split-H exchange of
 * nts_qknorm_rms, whose normalized rows leave as an MX (or NVFP4) block cast
 * instead of bf16: the QK path's Phase C feeds the block stage of
 * nts_rmsnorm_mxcast (SwiftQK Sec. III.C writes only the final normalized
 * shard; the MXNorm card, Fig. 8, fuses normalization and cast into one
 * kernel).  With w_j = fp32(x_j * gamma_j) and rinv = 1/sqrt(S/H + eps),
 * S = S_0 + ... + S_{N-1} in rank order as in nts_qknorm_rms, the scales and
 * codes are exactly those nts_rmsnorm_mxcast defines for this w and rinv
 * (E8M0 scales for E4M3/E2M1, E4M3 scales for NVFP4).  Each block's absmax
 * is taken while the exchange is in flight; blocks never straddle shards.
 *   X_dev       bf16 [T, H], read.         gamma_dev  fp32 [H], read.
 *   codes_dev   uint8 [T, H] (E4M3) or [T, H/2] (E2M1, NVFP4), written,
 *               16-byte aligned.
 *   scales_dev  uint8 [T, H/B], written.   rinv_dev   fp32 [T] or NULL.
 *   Limits of nts_qknorm_rms, plus B in {16, 32, 64} (16 for NVFP4) and
 *   (H / N) % B == 0.
 * Errors: as nts_qknorm_rms; INVALID_ARG also for a null scales_dev, a bad
 *         B or fmt; UNSUPPORTED for (H / N) % B != 0.
 */
NTS_API int nts_qknorm_rms_mxcast(const void *X_dev, const float *gamma_dev,
                                  uint8_t *codes_dev, uint8_t *scales_dev, float *rinv_dev,
                                  int64_t T, int64_t H, float eps, int N, int B, int fmt,
                                  void *stream);

/*
 * nts_qknorm_rms_qk_mxcast -- nts_qknorm_rms_mxcast of a token batch's Q and
 * K in ONE launch, as nts_qknorm_rms_qk fuses nts_qknorm_rms: Q and K may
 * have different widths (Hq, Hk) and their own gains; they share T, eps, N,
 * B and fmt.  Each tensor's codes, scales and rinv follow the definition of
 * nts_qknorm_rms_mxcast.  Both tensors take the thread layout of the wider
 * shard: with Hq == Hk every result equals that of a one-tensor call bit for
 * bit; otherwise the narrower tensor's fp32 sum of squares may be added in
 * another order (rinv within fp32 rounding of the one-tensor call; its scales
 * and codes are decided with that rinv).  Each tensor obeys the argument
 * rules of nts_qknorm_rms_mxcast, and the same errors apply, for either.
 */
NTS_API int nts_qknorm_rms_qk_mxcast(const void *Q_dev, const float *gamma_q_dev,
                                     uint8_t *codes_q_dev, uint8_t *scales_q_dev,
                                     float *rinv_q_dev, const void *K_dev,
                                     const float *gamma_k_dev, uint8_t *codes_k_dev,
                                     uint8_t *scales_k_dev, float *rinv_k_dev, int64_t T,
                                     int64_t Hq, int64_t Hk, float eps, int N, int B, int fmt,
                                     void *stream);

/*
 * nts_rmsnorm_mxcast -- RMSNorm fused with the MX cast (MXNorm card,
 * Fig. 1 caption, left graph; Fig. 8, where the normalization and the cast
 * are one fused kernel):
 *
 *     rinv     = 1 / sqrt((1/D) sum_j x_j^2 + eps)      (statistic of x, fp32)
 *     w_j      = fp32(x_j * gamma_j), or x_j when gamma_dev is NULL
 *     amax_k   = max over block k (B contiguous elements) of |w_j|
 *     e_k      = round(log2(fp32(amax_k * rinv))) - emax, clamped to
 *                [-127, 127], where round() is to the nearest integer in the
 *                log2 domain (mantissa >= sqrt 2 rounds up) and emax = 8
 *                (E4M3: the scale divides the absmax by 256) or 2 (E2M1)
 *     scale_k  = e_k + 127                                   (E8M0 byte)
 *     code_j   = cast_rne_satfinite(fp32(w_j * rinv) * 2^-e_k)
 *
 *   X_dev       bf16 [T, D], read.    gamma_dev fp32 [D], read, or NULL.
 *   codes_dev   E4M3: uint8 [T, D]; E2M1: uint8 [T, D/2] with element 2i in
 *               bits 0-3 and element 2i+1 in bits 4-7 of byte i.  Written.
 *   scales_dev  uint8 [T, D/B] E8M0 codes (2^(code-127)), row-major. Written.
 *   rinv_dev    fp32 [T] or NULL.   amax_dev  fp32 [T, D/B] block absmaxes
 *               of w (before normalization) or NULL.
 *   T >= 0; D % B == 0; B in {16, 32, 64}; D <= 32768; eps > 0 and finite;
 *   fmt in nts_elem_fmt.
 *
 * fmt = NTS_FMT_NVFP4 (B must be 16; the MXNorm card lists NVFP4 among its
 * kernel cases, Table 4, without its rules; this is the reading taken):
 *     s_k      = E4M3_rne_satfinite(fp32(fp32(amax_k * rinv) / 6))
 *     scale_k  = the E4M3 code of s_k
 *     code_j   = E2M1_rne_satfinite(fp32(fp32(w_j * rinv) * fp32(1 / s_k))),
 *                or 0 for every element of a block whose s_k is 0;
 * codes are laid out as for E2M1; no per-tensor second-level scale.
 * Errors: INVALID_ARG (null X/codes/scales, T < 0, D <= 0, D % B, bad B,
 *         eps or fmt, NVFP4 with B != 16), UNSUPPORTED (row too wide,
 *         unaligned pointer), CUDA (launch failure).
 */
NTS_API int nts_rmsnorm_mxcast(const void *X_dev, const float *gamma_dev,
                       uint8_t *codes_dev, uint8_t *scales_dev,
                       float *rinv_dev, float *amax_dev, int64_t T, int64_t D,
                       float eps, int B, int fmt, void *stream);

/*
 * nts_mxnorm_cast -- MXNorm (MXNorm card, abstract and Fig. 1 caption,
 * right graph): the RMS is estimated from the K = D/B block absmaxes that the
 * MX cast computes anyway,
 *
 *     rho~  = c(B, p) * ((1/K) sum_k amax_k^p)^(1/p),   p in {1, 2}
 *     rinv  = 1 / sqrt(rho~^2 + eps)
 *
 * then the block stage of nts_rmsnorm_mxcast runs with this rinv (the
 * normalized block absmax is amax_k * rinv, so no second reduction).  w, the
 * tensor whose absmaxes are taken and which is cast, is x (gamma_dev NULL,
 * the gain folded into the next Linear layer) or fp32(x * gamma).
 * c(B, p) = E[max of B i.i.d. |N(0,1)|^p]^(-1/p) (nts_mxnorm_correction).
 * Arguments, layouts and errors as nts_rmsnorm_mxcast, plus p in {1, 2}
 * (INVALID_ARG otherwise).
 */
NTS_API int nts_mxnorm_cast(const void *X_dev, const float *gamma_dev,
                    uint8_t *codes_dev, uint8_t *scales_dev, float *rinv_dev,
                    float *amax_dev, int64_t T, int64_t D, float eps, int B,
                    int fmt, int p, void *stream);

/*
 * nts_mxnorm_postround_cast -- the "post-round" MXNorm scheme (MXNorm card,
 * Fig. A.4, which names it and reports it trains unstably; reading): the RMS
 * estimate takes every block absmax after the E8M0 power-of-two rounding,
 *     rho~ = c(B, p) * ((1/K) sum_k (2^round(log2 amax_k))^p)^(1/p),
 * with the same c(B, p); the cast (scales and codes from amax_k * rinv) is
 * that of nts_mxnorm_cast.  Arguments, layouts and errors as
 * nts_mxnorm_cast; the rounding is that of E8M0 scales, so fmt =
 * NTS_FMT_NVFP4 is INVALID_ARG here.
 */
NTS_API int nts_mxnorm_postround_cast(const void *X_dev, const float *gamma_dev,
                                      uint8_t *codes_dev, uint8_t *scales_dev,
                                      float *rinv_dev, float *amax_dev, int64_t T, int64_t D,
                                      float eps, int B, int fmt, int p, void *stream);

/*
 * nts_mxnorm_correction -- the correction factor c(B, p) used by
 * nts_mxnorm_cast (MXNorm card, Fig. 1 caption: the scalar making the
 * estimate equal the RMS for i.i.d. Gaussian rows), computed on the host by
 * quadrature.  B >= 1, p in {1, 2}; *c_out receives the value.
 * Errors: INVALID_ARG.
 */
NTS_API int nts_mxnorm_correction(int B, int p, double *c_out);

/*
 * nts_check_status -- synchronizes `stream`, then reads and clears the
 * device status words.  Returns NTS_ERR_TIMEOUT if any kernel since the last
 * check gave up on a bounded wait (its outputs are then undefined),
 * NTS_ERR_CUDA if the stream reported an error, NTS_OK otherwise.
 */
NTS_API int nts_check_status(void *stream);

/*
 * Host-buffer forms: the same operations for callers whose inputs and
 * outputs live in host memory.  Each enqueues the host->device copy of the
 * input rows, the kernel, and the device->host copies of the outputs, all
 * ordered on `stream`: the caller synchronizes the stream before reading
 * *_host outputs.  Calls of more than 32 MB move their rows in up to 16
 * chunks through two internal copy streams (one per direction, created on
 * the first such call on a device) while the kernels run on `stream`, so
 * both copy directions and the kernels overlap; the enqueueing of such calls
 * from several host threads is serialized.  Host buffers should be pinned
 * for the copies to run asynchronously.
 * The device staging buffers (*_dev) are caller-owned and sized like the
 * corresponding host buffers; gamma stays a device pointer (a parameter,
 * uploaded once).  Optional outputs follow the device forms: a NULL *_host
 * output skips that output (its *_dev may then be NULL too).
 * Errors: as the device forms; CUDA also covers a failed copy.
 */
NTS_API int nts_qknorm_rms_host(const void *X_host, const float *gamma_dev,
                        void *Y_host, float *rinv_host, void *X_dev,
                        void *Y_dev, float *rinv_dev, int64_t T, int64_t H,
                        float eps, int N, void *stream);

/*
 * nts_qknorm_rms_qk_host -- nts_qknorm_rms_qk on host buffers: the copies of
 * Q and K to the device, the one launch that normalizes both, and the copies
 * of Yq and Yk back, enqueued as nts_qknorm_rms_host enqueues its work (in
 * row chunks through the library's copy streams for large calls; the
 * caller's stream is ordered after the last copy back).
 *   Q_host bf16 [T, Hq], K_host bf16 [T, Hk]: read.
 *   Yq_host, Yk_host: written once the stream reaches the end of the call.
 *   Q_dev, Yq_dev, K_dev, Yk_dev: caller-owned device staging of the same
 *   sizes (16-byte aligned); gamma_q_dev, gamma_k_dev: device gains.
 * Errors: as nts_qknorm_rms_qk; CUDA also covers a failed copy.
 */
NTS_API int nts_qknorm_rms_qk_host(const void *Q_host, const float *gamma_q_dev,
                                   void *Yq_host, const void *K_host,
                                   const float *gamma_k_dev, void *Yk_host, void *Q_dev,
                                   void *Yq_dev, void *K_dev, void *Yk_dev, int64_t T,
                                   int64_t Hq, int64_t Hk, float eps, int N, void *stream);

NTS_API int nts_rmsnorm_mxcast_host(const void *X_host, const float *gamma_dev,
                            uint8_t *codes_host, uint8_t *scales_host,
                            void *X_dev, uint8_t *codes_dev,
                            uint8_t *scales_dev, int64_t T, int64_t D,
                            float eps, int B, int fmt, void *stream);

NTS_API int nts_mxnorm_cast_host(const void *X_host, const float *gamma_dev,
                         uint8_t *codes_host, uint8_t *scales_host,
                         void *X_dev, uint8_t *codes_dev, uint8_t *scales_dev,
                         int64_t T, int64_t D, float eps, int B, int fmt,
                         int p, void *stream);

/*
 * nts_mxnorm_cast_host_noalloc -- nts_mxnorm_cast_host with no caller-owned
 * device buffers: the device staging for X, gamma, codes and scales is a
 * fixed 16 MiB array inside the library (one per device).  The pages have
 * no counterpart; it serves callers that cannot allocate device memory at
 * the call: processes whose device memory another framework's pool has
 * already reserved, latency-bound loops that must not call the allocator
 * after start-up (cudaFree synchronizes the device, cudaMalloc may), and
 * host-only callers with no device allocator.
 *
 *   X_host      bf16 [T, D], read.   gamma_host  fp32 [D], read, or NULL.
 *   codes_host, scales_host: as nts_mxnorm_cast_host, written once the
 *   stream reaches the end of the call's work.  Other arguments as
 *   nts_mxnorm_cast.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (and fills the library's host-side launch caches: device facts, kernel
 * attributes, c(B, p), the stream's tile counters).  Its copies and its
 * kernel all run on `stream` in one piece, never chunked, so it never
 * creates the copy streams of the other host-buffer forms.  Make that first
 * call before any stream capture; later calls on that device and stream
 * allocate nothing, host or device.
 * Sharing: every call on a device uses the same array, so calls that overlap
 * in time (other streams, unordered host threads) race and corrupt each
 * other's staging; serialize them.  Nothing in the array needs to start at
 * zero: each call copies in all the kernel reads.
 * Errors: as nts_mxnorm_cast_host, and every argument is checked before
 * anything is enqueued; UNSUPPORTED when the call needs more than 16 MiB of
 * staging (2*T*D bytes of X, 4*D of gamma, T*D or T*D/2 of codes,
 * T*D/B of scales, each rounded up to 256 bytes), or for a device ordinal
 * of 64 or more.
 */
NTS_API int nts_mxnorm_cast_host_noalloc(const void *X_host, const float *gamma_host,
                                         uint8_t *codes_host, uint8_t *scales_host, int64_t T,
                                         int64_t D, float eps, int B, int fmt, int p,
                                         void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NTS_H */
