/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the two
 * per-token normalization paths.  TEST INFRASTRUCTURE ONLY: nothing in the
 * product library links, includes or calls this file.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * Every quantity is computed in double precision with plain loops, in the
 * order the defining passage states.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Sources (web pages), cited by title and section:
 *   [SQK]  "SwiftQK: Fast and Communication-Efficient Tensor Parallelism for
 *          Query-Key Normalization" (IEEE CAL), Sec. II.A Eq. (1),
 *          Sec. III.A-C and Algorithm 1.
 *   [SQKN] SwiftQK reading notes (zhongzhuzhou.org), Eq. (1) (clean form),
 *          Sec. 3 (Algorithm 1 restated), Sec. 4b worked example Eqs. (2)-(8).
 *   [MXN]  MXNorm paper card (arXiv 2603.13180): abstract, Fig. 1 caption
 *          (RMSNorm + MXCast vs MXNorm, absmax/256, 2^round(log2), c(B,p)),
 *          Fig. A.1 (MX block: B E4M3 values sharing one E8M0 scale).
 *   [OCP]  OCP Microscaling Formats (MX) v1.0 element encodings
 *          (E4M3: bias 7, max 448, no infinities; E2M1: bias 1, max 6).
 *
 * Parity pins live in tests/test_oracle_*.py; which function is pinned by
 * what is written above each function below.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* Nearest value of a binary floating-point format with `p` significand bits
 * (the implicit leading bit included) whose smallest normal power of two is
 * 2^emin, ties to even.  Magnitudes above `maxfinite` after rounding become
 * `maxfinite` when `satfinite` is set (the OCP "saturating" cast), otherwise
 * infinity.  Subnormals of the format fall out of clamping the exponent at
 * emin: the quantum stays 2^(emin-p+1) below 2^emin. */
static double round_to_format(double v, int p, int emin, double maxfinite,
                              int satfinite) {
    if (v == 0.0 || isnan(v)) return v;
    double a = fabs(v);
    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1)       */
    int E = e2 - 1;               /* floor(log2 a)                      */
    if (E < emin) E = emin;       /* subnormal range: fixed quantum     */
    double quantum = ldexp(1.0, E - (p - 1));
    double r = nearbyint(a / quantum) * quantum; /* default mode: ties-to-even */
    if (r > maxfinite) r = satfinite ? maxfinite : INFINITY;
    return copysign(r, v);
}

/* bfloat16: 8 significand bits, min normal 2^-126, max (2-2^-7)*2^127,
 * overflow to infinity (the round-to-nearest-even cast). */
ORACLE_EXPORT uint16_t oracle_double_to_bf16(double v) {
    double r = round_to_format(v, 8, -126, ldexp(2.0 - ldexp(1.0, -7), 127), 0);
    float f = (float)r;           /* exact: every bf16 value is an fp32 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

ORACLE_EXPORT double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP E4M3 (FN variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * normal range 2^-6 .. 448, subnormal quantum 2^-9, no infinities.
 * Saturating, round-to-nearest-even cast; the sign of zero is kept. */
ORACLE_EXPORT uint8_t oracle_double_to_e4m3(double v) {
    double r = round_to_format(v, 4, -6, 448.0, 1);
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(r);
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -6)) {                     /* subnormal: exp field 0 */
        return (uint8_t)(sign | (uint8_t)(a / ldexp(1.0, -9)));
    }
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    uint8_t field = (uint8_t)(E + 7);
    uint8_t mant = (uint8_t)((a / ldexp(1.0, E) - 1.0) * 8.0);
    return (uint8_t)(sign | (field << 3) | mant);
}

ORACLE_EXPORT double oracle_e4m3_to_double(uint8_t c) {
    int s = c >> 7, field = (c >> 3) & 0xF, mant = c & 7;
    double a;
    if (field == 0xF && mant == 7) return NAN;
    if (field == 0) a = ldexp((double)mant, -9);
    else a = ldexp(1.0 + mant / 8.0, field - 7);
    return s ? -a : a;
}

/* OCP E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Saturating RNE cast, sign of zero kept.
 * Returns the 4-bit code in the low nibble. */
ORACLE_EXPORT uint8_t oracle_double_to_e2m1(double v) {
    double r = round_to_format(v, 2, 0, 6.0, 1);
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(r);
    if (a == 0.0) return sign;
    if (a < 1.0) return (uint8_t)(sign | 0x1);    /* the one subnormal, 0.5 */
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    uint8_t field = (uint8_t)(E + 1);
    uint8_t mant = (uint8_t)((a / ldexp(1.0, E) - 1.0) * 2.0);
    return (uint8_t)(sign | (field << 1) | mant);
}

ORACLE_EXPORT double oracle_e2m1_to_double(uint8_t c) {
    int s = (c >> 3) & 1, field = (c >> 1) & 3, mant = c & 1;
    double a = field == 0 ? 0.5 * mant : ldexp(1.0 + mant / 2.0, field - 1);
    return s ? -a : a;
}

/* round(log2 v) to the nearest integer, for v > 0 ([MXN] Fig. 1 caption:
 * the E8M0 cast uses the power-of-two rounding 2^round(log2 .)).  With
 * v = m * 2^E, m in [1, 2): log2 v = E + log2 m, and log2 m > 1/2 exactly
 * when m > sqrt(2), i.e. m*m - 2 > 0.  fma() evaluates m*m - 2 with one
 * rounding, which cannot change its sign, so the comparison is exact.
 * A tie (m == sqrt 2) is impossible for a binary m. */
ORACLE_EXPORT int oracle_round_log2(double v) {
    int e2;
    double m = 2.0 * frexp(v, &e2);               /* m in [1, 2)   */
    int E = e2 - 1;
    return E + (fma(m, m, -2.0) > 0.0 ? 1 : 0);
}

/* Unbiased E8M0 exponent of an MX block whose normalized absmax is v:
 * divide by the largest power of two of the element format (2^emax: 256 for
 * E4M3 per [MXN] Fig. 1 caption; 4 for E2M1 by the same rule), round in the
 * log2 domain, clamp to the E8M0 range [-127, 127] (code 255 = NaN is never
 * produced).  v == 0 gives the smallest scale, 2^-127. */
ORACLE_EXPORT int oracle_e8m0_exponent(double v, int emax) {
    if (!(v > 0.0)) return -127;
    int e = oracle_round_log2(v) - emax;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* ------------------------------------------------------------------------ */
/* Path 1: layerwise QK-RMSNorm with split-H scalar partial sums             */
/* ------------------------------------------------------------------------ */

/* RMSNorm of each token row x (length H), [SQKN] Eq. (1):
 *     y_j = x_j / sqrt((1/H) sum_j x_j^2 + eps) * gamma_j,
 * evaluated in the three phases of [SQK] Algorithm 1 / Sec. III:
 *   Phase A  each of the N shards (columns [kH/N, (k+1)H/N)) forms its local
 *            sum of squares S_k;
 *   combine  S = S_0 + S_1 + ... + S_{N-1} (rank order), RMS^-1 =
 *            1/sqrt(S/H_total + eps) with H_total the FULL row width;
 *   Phase B  the weight product x_j * gamma_j, independent of S;
 *   Phase C  y_j = (x_j * gamma_j) * RMS^-1, rounded once to bfloat16.
 * X, Y: bf16 bit patterns [T][H] row-major; gamma: fp32 [H];
 * rinv: [T] (nullable); partials: [T][N] per-shard S_k (nullable). */
ORACLE_EXPORT void oracle_qknorm_rms(const uint16_t *X, const float *gamma,
                                     uint16_t *Y, double *rinv, double *partials,
                                     int64_t T, int64_t H, double eps, int N) {
    int64_t W = H / N;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *x = X + t * H;
        double S = 0.0;
        for (int k = 0; k < N; ++k) {                       /* Phase A */
            double Sk = 0.0;
            for (int64_t j = k * W; j < (k + 1) * W; ++j) {
                double xj = oracle_bf16_to_double(x[j]);
                Sk += xj * xj;
            }
            if (partials) partials[t * N + k] = Sk;
            S += Sk;                                        /* combine */
        }
        double r = 1.0 / sqrt(S / (double)H + eps);
        if (rinv) rinv[t] = r;
        for (int64_t j = 0; j < H; ++j) {                   /* Phases B, C */
            double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];
            Y[t * H + j] = oracle_double_to_bf16(w * r);
        }
    }
}

/* QK-RMSNorm of FP8-E4M3 activations ([SQK] Sec. IV.C evaluates bf16 and
 * FP8-E4M3 activations with fp32 accumulation).  X holds E4M3 codes; the
 * activation is code * x_scale (a per-tensor dequantization scale).  The
 * phases and outputs are those of oracle_qknorm_rms. */
ORACLE_EXPORT void oracle_qknorm_rms_fp8(const uint8_t *X, double x_scale,
                                         const float *gamma, uint16_t *Y, double *rinv,
                                         double *partials, int64_t T, int64_t H,
                                         double eps, int N) {
    int64_t W = H / N;
    for (int64_t t = 0; t < T; ++t) {
        const uint8_t *x = X + t * H;
        double S = 0.0;
        for (int k = 0; k < N; ++k) {                       /* Phase A */
            double Sk = 0.0;
            for (int64_t j = k * W; j < (k + 1) * W; ++j) {
                double xj = oracle_e4m3_to_double(x[j]) * x_scale;
                Sk += xj * xj;
            }
            if (partials) partials[t * N + k] = Sk;
            S += Sk;                                        /* combine */
        }
        double r = 1.0 / sqrt(S / (double)H + eps);
        if (rinv) rinv[t] = r;
        for (int64_t j = 0; j < H; ++j) {                   /* Phases B, C */
            double w = oracle_e4m3_to_double(x[j]) * x_scale * (double)gamma[j];
            Y[t * H + j] = oracle_double_to_bf16(w * r);
        }
    }
}

/* LayerNorm split over H ([SQKN] Sec. 5e: LayerNorm's statistics reduce to
 * two additive scalars per shard, sum x and sum x^2, exchanged and combined
 * like the single sum of squares):
 *     mu = (1/H) sum_j x_j,   var = (1/H) sum_j (x_j - mu)^2,
 *     y_j = (x_j - mu) / sqrt(var + eps) * gamma_j + beta_j.
 * The oracle takes the definition (mean first, then the centred sum, in
 * double); partials [T][N][2] are each shard's (sum x, sum x^2).  beta is
 * nullable (zero); mean / rstd are [T] (nullable). */
ORACLE_EXPORT void oracle_layernorm_split(const uint16_t *X, const float *gamma,
                                          const float *beta, uint16_t *Y, double *mean,
                                          double *rstd, double *partials, int64_t T,
                                          int64_t H, double eps, int N) {
    int64_t W = H / N;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *x = X + t * H;
        double S1 = 0.0;
        for (int k = 0; k < N; ++k) {
            double s1 = 0.0, s2 = 0.0;
            for (int64_t j = k * W; j < (k + 1) * W; ++j) {
                double xj = oracle_bf16_to_double(x[j]);
                s1 += xj;
                s2 += xj * xj;
            }
            if (partials) {
                partials[(t * N + k) * 2] = s1;
                partials[(t * N + k) * 2 + 1] = s2;
            }
            S1 += s1;
        }
        double mu = S1 / (double)H;
        double var = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double d = oracle_bf16_to_double(x[j]) - mu;
            var += d * d;
        }
        var /= (double)H;
        double r = 1.0 / sqrt(var + eps);
        if (mean) mean[t] = mu;
        if (rstd) rstd[t] = r;
        for (int64_t j = 0; j < H; ++j) {
            double y = (oracle_bf16_to_double(x[j]) - mu) * r * (double)gamma[j];
            if (beta) y += (double)beta[j];
            Y[t * H + j] = oracle_double_to_bf16(y);
        }
    }
}

/* Headwise QK-Norm ([SQK] Sec. II.A): one normalization factor per attention
 * head instead of one per projected vector.  A token row of H = nheads *
 * head_dim values holds the heads one after another; head h of token t is
 * normalized over its own head_dim values,
 *     y_j = x_j / sqrt((1/head_dim) sum_{j in head} x_j^2 + eps) * gamma_j',
 * where gamma has head_dim entries shared by all heads (j' = j mod head_dim).
 * rinv: [T][nheads] (nullable). */
ORACLE_EXPORT void oracle_qknorm_rms_heads(const uint16_t *X, const float *gamma,
                                           uint16_t *Y, double *rinv, int64_t T,
                                           int64_t H, int64_t head_dim, double eps) {
    int64_t nheads = H / head_dim;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < nheads; ++h) {
            const uint16_t *x = X + t * H + h * head_dim;
            double S = 0.0;
            for (int64_t j = 0; j < head_dim; ++j) {
                double xj = oracle_bf16_to_double(x[j]);
                S += xj * xj;
            }
            double r = 1.0 / sqrt(S / (double)head_dim + eps);
            if (rinv) rinv[t * nheads + h] = r;
            for (int64_t j = 0; j < head_dim; ++j) {
                double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];
                Y[t * H + h * head_dim + j] = oracle_double_to_bf16(w * r);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Path 2: RMSNorm + MX cast, and MXNorm                                     */
/* ------------------------------------------------------------------------ */

/* Correction factor c(B, p) of [MXN] Fig. 1 caption: the scalar that makes
 * the MXNorm estimate equal the RMS for i.i.d. Gaussian inputs.  For
 * X ~ N(0, sigma^2) the block absmax is sigma * M with M the maximum of B
 * i.i.d. |N(0,1)|; requiring c * E[(sigma M)^p]^(1/p) = sigma gives
 *     c(B, p) = E[M^p]^(-1/p),
 *     E[M^p]  = integral_0^inf p x^(p-1) (1 - erf(x/sqrt 2)^B) dx
 * (the survival-function form of the moment).  1 - erf^B is evaluated as
 * -expm1(B log1p(-erfc)) to keep the tail accurate.  The integral is taken
 * by adaptive Simpson quadrature on [0, 40]; the integrand is below 1e-300
 * past that. */
static double cpb_integrand(double x, int B, int p) {
    double q = erfc(x / sqrt(2.0));
    double tail = -expm1((double)B * log1p(-q));
    return (double)p * pow(x, (double)(p - 1)) * tail;
}

static double simpson(double a, double b, double fa, double fm, double fb) {
    return (b - a) / 6.0 * (fa + 4.0 * fm + fb);
}

static double adaptive_simpson(int B, int p, double a, double b, double fa,
                               double fm, double fb, double whole, double tol,
                               int depth) {
    double m = 0.5 * (a + b);
    double lm = 0.5 * (a + m), rm = 0.5 * (m + b);
    double flm = cpb_integrand(lm, B, p), frm = cpb_integrand(rm, B, p);
    double left = simpson(a, m, fa, flm, fm);
    double right = simpson(m, b, fm, frm, fb);
    double delta = left + right - whole;
    if (depth <= 0 || fabs(delta) <= 15.0 * tol)
        return left + right + delta / 15.0;
    return adaptive_simpson(B, p, a, m, fa, flm, fm, left, 0.5 * tol, depth - 1) +
           adaptive_simpson(B, p, m, b, fm, frm, fb, right, 0.5 * tol, depth - 1);
}

ORACLE_EXPORT double oracle_mx_correction(int B, int p) {
    double total = 0.0;
    /* unit panels keep the recursion shallow where the integrand bends */
    for (int i = 0; i < 40; ++i) {
        double a = i, b = i + 1;
        double fa = cpb_integrand(a, B, p), fb = cpb_integrand(b, B, p);
        double fm = cpb_integrand(0.5 * (a + b), B, p);
        total += adaptive_simpson(B, p, a, b, fa, fm, fb,
                                  simpson(a, b, fa, fm, fb), 1e-15, 40);
    }
    return pow(total, -1.0 / (double)p);
}

/* Shared block stage of both MX functions ([MXN] Fig. 1 caption, Fig. A.1):
 * for one row whose values (already multiplied by gamma when given) are
 * w[0..D) and whose normalization factor is r, every block k of B contiguous
 * values gets
 *     amax_k  = max_b |w_kb|                        (before normalization)
 *     e_k     = round(log2(amax_k * r / 2^emax))    (E8M0, clamped)
 *     code_kb = cast(w_kb * r * 2^-e_k; E4M3 or E2M1).
 * `in_float` selects where the normalized values are formed:
 *   0: in double, r given in double (the definition);
 *   1: in fp32, as fl32(w * r) with r an fp32 value -- the precision the
 *      decision is taken in when comparing against a device result whose
 *      fp32 r is known (integer codes decided in the same precision).
 * Output layout: codes row-major (E4M3 one byte per element; E2M1 two per
 * byte, element 2i in the low nibble), scales [K] bytes, amax [K] floats. */
/* NVFP4 block (fmt 2; a reading: the MXNorm card names NVFP4 among its
 * kernel cases, Table 4, without its rules): B = 16 E2M1 values share one
 * E4M3 scale
 *     s_k    = E4M3(amax_k * r / 6)        (6 = largest E2M1 magnitude;
 *                                            RNE, saturating at 448)
 *     code_kb = E2M1(w_kb * r / s_k)        (code 0 when s_k == 0),
 * with no second, per-tensor scale: the normalized absmaxes lie far inside
 * the E4M3 range.  In fp32 mode every step is an fp32 operation:
 * fl32(fl32(amax*r)/6), then fl32(fl32(w*r) * fl32(1/s)). */
static void nvfp4_cast_block(const float *w, int B, double r, int in_float,
                             double amax, uint8_t *codes, int64_t j0,
                             uint8_t *scale) {
    double v = in_float ? (double)(float)(amax * r) : amax * r;
    double sv = in_float ? (double)(float)(v / 6.0) : v / 6.0;
    uint8_t sc = oracle_double_to_e4m3(sv);
    double s = oracle_e4m3_to_double(sc);
    double inv = 0.0;
    if (s > 0.0) inv = in_float ? (double)(float)(1.0 / s) : 1.0 / s;
    *scale = sc;
    for (int b = 0; b < B; ++b) {
        int64_t j = j0 + b;
        double y = in_float ? (double)(float)((double)w[b] * r) : (double)w[b] * r;
        uint8_t c = 0;
        if (s > 0.0) c = oracle_double_to_e2m1(in_float ? (double)(float)(y * inv) : y / s);
        if ((j & 1) == 0) codes[j / 2] = c;
        else codes[j / 2] = (uint8_t)(codes[j / 2] | (c << 4));
    }
}

static void mx_cast_row(const float *w, int64_t D, double r, int in_float,
                        int B, int fmt, uint8_t *codes, uint8_t *scales,
                        float *amax_out) {
    int emax = fmt == 0 ? 8 : 2;
    int64_t K = D / B;
    for (int64_t k = 0; k < K; ++k) {
        double amax = 0.0;
        for (int b = 0; b < B; ++b) {
            double a = fabs((double)w[k * B + b]);
            if (a > amax) amax = a;
        }
        if (amax_out) amax_out[k] = (float)amax;
        if (fmt == 2) {
            nvfp4_cast_block(w + k * B, B, r, in_float, amax, codes, k * B, scales + k);
            continue;
        }
        double v = in_float ? (double)(float)(amax * r) : amax * r;
        int e = oracle_e8m0_exponent(v, emax);
        scales[k] = (uint8_t)(e + 127);
        for (int b = 0; b < B; ++b) {
            int64_t j = k * B + b;
            double y = in_float ? (double)(float)((double)w[j] * r)
                                : (double)w[j] * r;
            double q = ldexp(y, -e);
            if (fmt == 0) {
                codes[j] = oracle_double_to_e4m3(q);
            } else {
                uint8_t c = oracle_double_to_e2m1(q);
                if ((j & 1) == 0) codes[j / 2] = c;
                else codes[j / 2] = (uint8_t)(codes[j / 2] | (c << 4));
            }
        }
    }
}

/* w_j = fl32(x_j * gamma_j), or x_j when gamma is NULL (the gain folded into
 * the next Linear layer, [MXN] Fig. 1 top right).  The product of a bf16 and
 * an fp32 value is exact in double, so one cast gives the fp32 product. */
static void weight_row(const uint16_t *x, const float *gamma, int64_t D,
                       float *w) {
    for (int64_t j = 0; j < D; ++j) {
        double xj = oracle_bf16_to_double(x[j]);
        w[j] = gamma ? (float)(xj * (double)gamma[j]) : (float)xj;
    }
}

static int64_t codes_row_bytes(int64_t D, int fmt) { return fmt == 0 ? D : D / 2; }

/* RMSNorm followed by the MX cast ([MXN] Fig. 1 caption, left-hand graph;
 * fused as one kernel in Fig. 8): r = 1/sqrt((1/D) sum_j x_j^2 + eps), the
 * statistic of x itself as in Eq. (1), then the block stage above on
 * w = x * gamma.  `work` holds D floats. */
ORACLE_EXPORT void oracle_rmsnorm_mxcast(const uint16_t *X, const float *gamma,
                                         uint8_t *codes, uint8_t *scales,
                                         double *rinv, float *amax, float *work,
                                         int64_t T, int64_t D, double eps,
                                         int B, int fmt) {
    int64_t K = D / B, cb = codes_row_bytes(D, fmt);
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *x = X + t * D;
        double S = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double xj = oracle_bf16_to_double(x[j]);
            S += xj * xj;
        }
        double r = 1.0 / sqrt(S / (double)D + eps);
        if (rinv) rinv[t] = r;
        weight_row(x, gamma, D, work);
        mx_cast_row(work, D, r, 0, B, fmt, codes + t * cb, scales + t * K,
                    amax ? amax + t * K : NULL);
    }
}

/* MXNorm ([MXN] abstract and Fig. 1 caption, right-hand graph): the RMS is
 * estimated from the K = D/B block absmaxes a_k of the values being cast,
 *     rho~ = c(B,p) * ((1/K) sum_k a_k^p)^(1/p),   p = 1 or 2,
 * and r = 1/sqrt(rho~^2 + eps) (eps enters like Eq. (1): added to the
 * estimated mean square).  The output is the MX cast of w * r, whose block
 * absmaxes are a_k * r, so no second reduction is needed.  `c` is the
 * correction factor (oracle_mx_correction(B, p)). */
static void mxnorm_rows(const uint16_t *X, const float *gamma, uint8_t *codes,
                        uint8_t *scales, double *rinv, float *amax, float *work,
                        int64_t T, int64_t D, double eps, int B, int fmt, int p,
                        double c, int post_round) {
    int64_t K = D / B, cb = codes_row_bytes(D, fmt);
    for (int64_t t = 0; t < T; ++t) {
        weight_row(X + t * D, gamma, D, work);
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = 0.0;
            for (int b = 0; b < B; ++b) {
                double v = fabs((double)work[k * B + b]);
                if (v > a) a = v;
            }
            /* post-round: the block absmax as its E8M0 power of two */
            if (post_round && a > 0.0) a = ldexp(1.0, oracle_round_log2(a));
            acc += p == 1 ? a : a * a;
        }
        double Mp = p == 1 ? acc / (double)K : sqrt(acc / (double)K);
        double rho = c * Mp;
        double r = 1.0 / sqrt(rho * rho + eps);
        if (rinv) rinv[t] = r;
        mx_cast_row(work, D, r, 0, B, fmt, codes + t * cb, scales + t * K,
                    amax ? amax + t * K : NULL);
    }
}

ORACLE_EXPORT void oracle_mxnorm_cast(const uint16_t *X, const float *gamma,
                                      uint8_t *codes, uint8_t *scales,
                                      double *rinv, float *amax, float *work,
                                      int64_t T, int64_t D, double eps, int B,
                                      int fmt, int p, double c) {
    mxnorm_rows(X, gamma, codes, scales, rinv, amax, work, T, D, eps, B, fmt, p, c, 0);
}

/* Post-round MXNorm ([MXN] Fig. A.4 names the scheme; reading): the RMS
 * estimate takes each block absmax after the E8M0 power-of-two rounding,
 * a_k -> 2^round(log2 a_k), with the same c(B, p); the cast itself is the
 * block stage above, on the unrounded absmaxes. */
ORACLE_EXPORT void oracle_mxnorm_postround_cast(const uint16_t *X, const float *gamma,
                                                uint8_t *codes, uint8_t *scales,
                                                double *rinv, float *amax, float *work,
                                                int64_t T, int64_t D, double eps,
                                                int B, int fmt, int p, double c) {
    mxnorm_rows(X, gamma, codes, scales, rinv, amax, work, T, D, eps, B, fmt, p, c, 1);
}

/* The block stage alone with a given fp32 normalization factor per row,
 * every normalized value formed in fp32 (fl32(amax * r), fl32(w * r)).
 * This is the stage where floating point decides integers (E8M0 exponents
 * and element codes); fed a device's own fp32 factors it takes the same
 * decisions in the same precision. */
ORACLE_EXPORT void oracle_mx_cast_given_rinv(const uint16_t *X,
                                             const float *gamma,
                                             const float *rinv_f32,
                                             uint8_t *codes, uint8_t *scales,
                                             float *amax, float *work,
                                             int64_t T, int64_t D, int B,
                                             int fmt) {
    int64_t K = D / B, cb = codes_row_bytes(D, fmt);
    for (int64_t t = 0; t < T; ++t) {
        weight_row(X + t * D, gamma, D, work);
        mx_cast_row(work, D, (double)rinv_f32[t], 1, B, fmt, codes + t * cb,
                    scales + t * K, amax ? amax + t * K : NULL);
    }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar encoders, for exhaustive encoder checks         */
/* ------------------------------------------------------------------------ */

ORACLE_EXPORT void oracle_encode_array(const double *v, uint8_t *out, int64_t n,
                                       int fmt) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = fmt == 0 ? oracle_double_to_e4m3(v[i]) : oracle_double_to_e2m1(v[i]);
}

ORACLE_EXPORT void oracle_bf16_array(const double *v, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16(v[i]);
}

ORACLE_EXPORT void oracle_e8m0_array(const double *v, int32_t *out, int64_t n,
                                     int emax) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e8m0_exponent(v[i], emax);
}
