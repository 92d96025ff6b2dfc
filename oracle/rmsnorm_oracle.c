/*
 * rmsnorm_oracle.c -- plain CPU oracle for row-wise RMSNorm, forward and backward.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline use this file. The GPU library never links, includes or calls it, and
 * it shares no code with the GPU library (its own dtype codes, its own number
 * format conversions, its own loops).
 *
 * What it computes (page "Check an AI model calculation before accelerating it",
 * sections "Problem and reference formula", "Why do we need a forward and a
 * backward pass?", "Where does the cube of r come from?" and "A sum is not an
 * average"), for a row-major M x N matrix x, a per-column weight gamma and an
 * upstream gradient dy:
 *
 *     r      = 1 / sqrt(mean_j(x_j^2) + eps)          one number per row
 *     y      = x * r * gamma                          elementwise
 *     u      = dy * gamma
 *     dx     = r * u - x * r^3 * mean_j(u_j * x_j)     mean over the N columns of a row
 *     dgamma = sum over the M rows of dy * x * r       a sum, not a mean
 *
 * The offset variant (page "torchtitan kernel numerics verification", section on
 * the golden / reference / target implementations) replaces gamma by (1 + w)
 * wherever gamma appears; dgamma keeps the same formula because d(1+w)/dw = 1.
 *
 * Two arithmetic levels, following the three-implementation method of the
 * torchtitan page:
 *
 *   golden     every input element is promoted exactly to fp64 and every step is
 *              done in fp64; outputs stay fp64.
 *   reference  every input element is converted to fp32 at load, every product,
 *              sum, square root and division is an fp32 operation, sums run left
 *              to right in index order, and each output (y, dx, dgamma) is rounded
 *              once, to nearest-even, into the I/O dtype. rstd stays fp32.
 *
 * This file must be compiled with floating-point contraction disabled
 * (-ffp-contract=off) so that every fp32 operation above is rounded on its own.
 *
 * Dtype codes used by this file: 0 = float32, 1 = float16, 2 = bfloat16.
 * Element storage: float32 as IEEE binary32, float16 as IEEE binary16 bits,
 * bfloat16 as the upper 16 bits of an IEEE binary32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* Exact value of an IEEE binary16 bit pattern. */
static double half_bits_to_double(uint16_t h) {
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25); /* (1024 + m) * 2^(e - 15 - 10) */
    return sign ? -v : v;
}

/* Exact value of a bfloat16 bit pattern (the top half of a binary32). */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/*
 * Round v to the nearest value of a binary floating-point format with `prec`
 * significand bits (implicit bit included), smallest normal exponent `emin` and
 * largest exponent `emax`; ties go to the even significand; values beyond the
 * largest finite number become infinities (IEEE 754 round-to-nearest-even).
 */
static double round_to_format(double v, int prec, int emin, int emax) {
    if (v != v || v == 0.0 || isinf(v)) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);            /* a = f * 2^e with f in [0.5, 1) */
    int lead = e - 1;        /* exponent of the leading bit */
    if (lead < emin) lead = emin;   /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, lead - (prec - 1));
    double r = nearbyint(a / quantum) * quantum;   /* default mode: ties to even */
    double max_finite = ldexp(2.0 - ldexp(1.0, 1 - prec), emax);
    if (r > max_finite) r = INFINITY;
    return v < 0 ? -r : r;
}

static double round_to_dtype(double v, int dt) {
    switch (dt) {
    case OR_F16:  return round_to_format(v, 11, -14, 15);
    case OR_BF16: return round_to_format(v, 8, -126, 127);
    default:      return round_to_format(v, 24, -126, 127);
    }
}

static uint16_t double_to_bf16_bits(double v) {
    if (v != v) return 0x7fc0;
    double r = round_to_format(v, 8, -126, 127);   /* representable in binary32 */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static uint16_t double_to_half_bits(double v) {
    if (v != v) return 0x7e00;
    double r = round_to_format(v, 11, -14, 15);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a)) return sign | 0x7c00;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int lead = e - 1;
    if (lead < -14)                              /* subnormal: a = m * 2^-24 */
        return sign | (uint16_t)(a * 16777216.0);
    uint16_t m = (uint16_t)((ldexp(a, -lead) - 1.0) * 1024.0);
    return sign | (uint16_t)((lead + 15) << 10) | m;
}

/* Value of element i of an array of dtype dt. */
static double load_elem(const void* base, int64_t i, int dt) {
    if (dt == OR_F32) {
        float f;
        memcpy(&f, (const char*)base + 4 * i, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * i, 2);
    return dt == OR_F16 ? half_bits_to_double(h) : bf16_bits_to_double(h);
}

/* Store v, rounded to nearest-even, as element i of an array of dtype dt. */
static void store_elem(void* base, int64_t i, int dt, double v) {
    if (dt == OR_F32) {
        float f = (float)v;   /* C conversion: round to nearest-even */
        memcpy((char*)base + 4 * i, &f, 4);
    } else {
        uint16_t h = dt == OR_F16 ? double_to_half_bits(v) : double_to_bf16_bits(v);
        memcpy((char*)base + 2 * i, &h, 2);
    }
}

/* --- exported format helpers (used by the tests and the gate) ------------ */

void oracle_decode(const void* src, int dt, int64_t n, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, i, dt);
}

void oracle_encode(const double* src, int64_t n, int dt, void* dst) {
    for (int64_t i = 0; i < n; ++i) store_elem(dst, i, dt, src[i]);
}

/* dst[i] = value of src[i] after rounding into dtype dt (the gate's rounding floor). */
void oracle_round(const double* src, int64_t n, int dt, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = round_to_dtype(src[i], dt);
}

/* ------------------------------------------------------------------------- */
/* Golden: fp64 throughout                                                   */
/* ------------------------------------------------------------------------- */

/*
 * y[M*N] (fp64), rstd[M] (fp64). gamma has dtype dt like x.
 * Forward formula: "Problem and reference formula" (r and y); offset variant from
 * the torchtitan page's golden implementation, (1 + w) * x * r.
 */
void oracle_fwd_golden(const void* x, const void* gamma, int64_t M, int64_t N,
                       double eps, int dt, int offset, double* y, double* rstd) {
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(x, row + j, dt);
            ss += xv * xv;
        }
        double r = 1.0 / sqrt(ss / (double)N + eps);
        if (rstd) rstd[i] = r;
        if (!y) continue;
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(x, row + j, dt);
            double w = load_elem(gamma, j, dt);
            y[row + j] = offset ? (1.0 + w) * xv * r : xv * r * w;
        }
    }
}

/*
 * dx[M*N] (fp64, may be NULL to skip), dgamma[N] (fp64, may be NULL).
 * r is recomputed from x exactly as in the forward pass.
 * Backward formula: "Why do we need a forward and a backward pass?" with
 * u = dy * gamma, dx = r*u - x*r^3*mean(u*x); dgamma = sum over rows of dy*x*r.
 */
void oracle_bwd_golden(const void* dy, const void* x, const void* gamma, int64_t M,
                       int64_t N, double eps, int dt, int offset, double* dx,
                       double* dgamma) {
    if (dgamma)
        for (int64_t j = 0; j < N; ++j) dgamma[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(x, row + j, dt);
            ss += xv * xv;
        }
        double r = 1.0 / sqrt(ss / (double)N + eps);
        double sux = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double w = load_elem(gamma, j, dt);
            double g = offset ? 1.0 + w : w;
            double u = load_elem(dy, row + j, dt) * g;
            sux += u * load_elem(x, row + j, dt);
        }
        double mean_ux = sux / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(x, row + j, dt);
            double dyv = load_elem(dy, row + j, dt);
            double w = load_elem(gamma, j, dt);
            double g = offset ? 1.0 + w : w;
            double u = dyv * g;
            if (dx) dx[row + j] = r * u - xv * r * r * r * mean_ux;
            if (dgamma) dgamma[j] += dyv * xv * r;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Reference: I/O dtype, fp32 intermediates, sequential sums                 */
/* ------------------------------------------------------------------------- */

static float ld32(const void* base, int64_t i, int dt) {
    return (float)load_elem(base, i, dt);   /* exact for all three dtypes */
}

/* fp32 r of one row: sequential sum of squares, mean, add eps, sqrt, reciprocal. */
static float row_rstd_f32(const void* x, int64_t row, int64_t N, float eps, int dt) {
    float ss = 0.0f;
    for (int64_t j = 0; j < N; ++j) {
        float xv = ld32(x, row + j, dt);
        float sq = xv * xv;
        ss = ss + sq;
    }
    float ms = ss / (float)N;
    float den = sqrtf(ms + eps);
    return 1.0f / den;
}

/*
 * y[M*N] in dtype dt, rstd[M] fp32. Multiplication order follows the pages'
 * reference code: (x * r) * gamma, and for the offset variant ((1 + w) * x) * r.
 */
void oracle_fwd_reference(const void* x, const void* gamma, int64_t M, int64_t N,
                          float eps, int dt, int offset, void* y, float* rstd) {
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        float r = row_rstd_f32(x, row, N, eps, dt);
        if (rstd) rstd[i] = r;
        if (!y) continue;
        for (int64_t j = 0; j < N; ++j) {
            float xv = ld32(x, row + j, dt);
            float w = ld32(gamma, j, dt);
            float out;
            if (offset) {
                float g = 1.0f + w;
                float gx = g * xv;
                out = gx * r;
            } else {
                float xr = xv * r;
                out = xr * w;
            }
            store_elem(y, row + j, dt, (double)out);
        }
    }
}

/*
 * dx[M*N] in dtype dt (may be NULL), dgamma[N] in dtype dt (may be NULL).
 * r is recomputed in fp32 from x exactly as oracle_fwd_reference does.
 * dx = (r * u) - ((x * r^3) * c) with r^3 = (r * r) * r and c = (sum u*x) / N;
 * dgamma accumulates (dy * x) * r over rows in row order, in one fp32 sum per
 * column, and is rounded into dtype dt once at the end.
 */
void oracle_bwd_reference(const void* dy, const void* x, const void* gamma, int64_t M,
                          int64_t N, float eps, int dt, int offset, void* dx,
                          void* dgamma) {
    float* acc = NULL;
    if (dgamma) {
        acc = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
        for (int64_t j = 0; j < N; ++j) acc[j] = 0.0f;
    }
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        float r = row_rstd_f32(x, row, N, eps, dt);
        float sux = 0.0f;
        for (int64_t j = 0; j < N; ++j) {
            float w = ld32(gamma, j, dt);
            float g = offset ? 1.0f + w : w;
            float u = ld32(dy, row + j, dt) * g;
            float ux = u * ld32(x, row + j, dt);
            sux = sux + ux;
        }
        float c = sux / (float)N;
        float r2 = r * r;
        float r3 = r2 * r;
        for (int64_t j = 0; j < N; ++j) {
            float xv = ld32(x, row + j, dt);
            float dyv = ld32(dy, row + j, dt);
            float w = ld32(gamma, j, dt);
            float g = offset ? 1.0f + w : w;
            float u = dyv * g;
            if (dx) {
                float t1 = r * u;
                float xr3 = xv * r3;
                float t2 = xr3 * c;
                float d = t1 - t2;
                store_elem(dx, row + j, dt, (double)d);
            }
            if (acc) {
                float dyx = dyv * xv;
                float term = dyx * r;
                acc[j] = acc[j] + term;
            }
        }
    }
    if (acc) {
        for (int64_t j = 0; j < N; ++j) store_elem(dgamma, j, dt, (double)acc[j]);
        free(acc);
    }
}

/* ------------------------------------------------------------------------- */
/* LayerNorm (page "torch.compile performance leap: optimizing LayerNorm and  */
/* RMSNorm kernels", sections 1.1 "LayerNorm" and 2 "Backward": per-row mean  */
/* and variance, learned gamma and beta; gradients for the input, the weight  */
/* and the bias). The pages print no formula; this is the standard one:       */
/*     mu = mean_j x_j;  var = mean_j (x_j - mu)^2;  r = 1/sqrt(var + eps)     */
/*     xhat = (x - mu) * r;  y = xhat * gamma + beta                          */
/*     u = dy * gamma;  dx = r * (u - mean_j u_j - xhat * mean_j(u_j xhat_j))  */
/*     dgamma = sum_rows dy * xhat;  dbeta = sum_rows dy                       */
/* The variance is the two-pass one (mean first).                             */
/* ------------------------------------------------------------------------- */

/* y[M*N], mean[M], rstd[M] in fp64 (any of them may be NULL). */
void oracle_ln_fwd_golden(const void* x, const void* gamma, const void* beta, int64_t M, int64_t N,
                          double eps, int dt, double* y, double* mean, double* rstd) {
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) s += load_elem(x, row + j, dt);
        const double mu = s / (double)N;
        double v = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double d = load_elem(x, row + j, dt) - mu;
            v += d * d;
        }
        const double r = 1.0 / sqrt(v / (double)N + eps);
        if (mean) mean[i] = mu;
        if (rstd) rstd[i] = r;
        if (!y) continue;
        for (int64_t j = 0; j < N; ++j) {
            const double xh = (load_elem(x, row + j, dt) - mu) * r;
            y[row + j] = xh * load_elem(gamma, j, dt) + load_elem(beta, j, dt);
        }
    }
}

/* dx[M*N] (may be NULL), dgamma[N], dbeta[N] in fp64; mu and r recomputed from x. */
void oracle_ln_bwd_golden(const void* dy, const void* x, const void* gamma, int64_t M, int64_t N, double eps,
                          int dt, double* dx, double* dgamma, double* dbeta) {
    for (int64_t j = 0; j < N; ++j) {
        if (dgamma) dgamma[j] = 0.0;
        if (dbeta) dbeta[j] = 0.0;
    }
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        double mu, r;
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) s += load_elem(x, row + j, dt);
        mu = s / (double)N;
        double v = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double d = load_elem(x, row + j, dt) - mu;
            v += d * d;
        }
        r = 1.0 / sqrt(v / (double)N + eps);
        double su = 0.0, suxh = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double u = load_elem(dy, row + j, dt) * load_elem(gamma, j, dt);
            const double xh = (load_elem(x, row + j, dt) - mu) * r;
            su += u;
            suxh += u * xh;
        }
        const double mean_u = su / (double)N, mean_uxh = suxh / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            const double dyv = load_elem(dy, row + j, dt);
            const double u = dyv * load_elem(gamma, j, dt);
            const double xh = (load_elem(x, row + j, dt) - mu) * r;
            if (dx) dx[row + j] = r * (u - mean_u - xh * mean_uxh);
            if (dgamma) dgamma[j] += dyv * xh;
            if (dbeta) dbeta[j] += dyv;
        }
    }
}

/* fp32 mean and r of one row: sequential sums, two-pass variance. */
static void ln_row_stats_f32(const void* x, int64_t row, int64_t N, float eps, int dt, float* mu_out,
                             float* r_out) {
    float s = 0.0f;
    for (int64_t j = 0; j < N; ++j) s = s + ld32(x, row + j, dt);
    const float mu = s / (float)N;
    float v = 0.0f;
    for (int64_t j = 0; j < N; ++j) {
        const float d = ld32(x, row + j, dt) - mu;
        const float d2 = d * d;
        v = v + d2;
    }
    const float var = v / (float)N;
    const float den = sqrtf(var + eps);
    *mu_out = mu;
    *r_out = 1.0f / den;
}

/* y[M*N] in dtype dt, mean[M] and rstd[M] fp32. y = ((x - mu) * r) * gamma + beta. */
void oracle_ln_fwd_reference(const void* x, const void* gamma, const void* beta, int64_t M, int64_t N,
                             float eps, int dt, void* y, float* mean, float* rstd) {
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        float mu, r;
        ln_row_stats_f32(x, row, N, eps, dt, &mu, &r);
        if (mean) mean[i] = mu;
        if (rstd) rstd[i] = r;
        if (!y) continue;
        for (int64_t j = 0; j < N; ++j) {
            const float d = ld32(x, row + j, dt) - mu;
            const float xh = d * r;
            const float t = xh * ld32(gamma, j, dt);
            const float out = t + ld32(beta, j, dt);
            store_elem(y, row + j, dt, (double)out);
        }
    }
}

/* dx[M*N] (may be NULL), dgamma[N], dbeta[N] in dtype dt; fp32 intermediates,
 * sequential sums; dx = r * ((u - mean(u)) - xhat * mean(u*xhat)). */
void oracle_ln_bwd_reference(const void* dy, const void* x, const void* gamma, int64_t M, int64_t N, float eps,
                             int dt, void* dx, void* dgamma, void* dbeta) {
    float* ag = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    float* ab = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    for (int64_t j = 0; j < N; ++j) ag[j] = ab[j] = 0.0f;
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        float mu, r;
        ln_row_stats_f32(x, row, N, eps, dt, &mu, &r);
        float su = 0.0f, suxh = 0.0f;
        for (int64_t j = 0; j < N; ++j) {
            const float u = ld32(dy, row + j, dt) * ld32(gamma, j, dt);
            const float xh = (ld32(x, row + j, dt) - mu) * r;
            const float uxh = u * xh;
            su = su + u;
            suxh = suxh + uxh;
        }
        const float mean_u = su / (float)N;
        const float mean_uxh = suxh / (float)N;
        for (int64_t j = 0; j < N; ++j) {
            const float dyv = ld32(dy, row + j, dt);
            const float u = dyv * ld32(gamma, j, dt);
            const float xh = (ld32(x, row + j, dt) - mu) * r;
            if (dx) {
                const float a = u - mean_u;
                const float b = xh * mean_uxh;
                const float c = a - b;
                store_elem(dx, row + j, dt, (double)(r * c));
            }
            const float g = dyv * xh;
            ag[j] = ag[j] + g;
            ab[j] = ab[j] + dyv;
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        if (dgamma) store_elem(dgamma, j, dt, (double)ag[j]);
        if (dbeta) store_elem(dbeta, j, dt, (double)ab[j]);
    }
    free(ag);
    free(ab);
}

/* ------------------------------------------------------------------------- */
/* RMSNorm double backward (page "Check an AI model calculation before        */
/* accelerating it", section "Adapting the kernel and moving to production",  */
/* which lists double backward among the extensions not yet validated). The   */
/* backward maps (dy, x, g) to (dx, dgamma); its own gradient, for cotangents */
/* ddx [M x N] of dx and ddg [N] of dgamma, is obtained by differentiating    */
/* the backward formula (r depends on x: dr/dx_j = -r^3 x_j / N):             */
/*     u = dy*g, c = mean(u*x), A = mean(ddx*x), B = mean(ddx*u),             */
/*     D = mean(ddg*dy*x)                                  (per row)          */
/*     d_dy = g*r*(ddx - r^2*x*A) + r*x*ddg                                   */
/*     d_x  = r*ddg*dy - r^3*(c*ddx + u*A + x*(B + D)) + 3*r^5*c*A*x          */
/*     d_g  = sum over rows of r*dy*(ddx - r^2*x*A)                           */
/* g = gamma, or 1 + w with offset (then d_w = d_g). ddg may be NULL (zero).   */
/* ------------------------------------------------------------------------- */

/* d_dy[M*N], d_x[M*N], d_gamma[N] in fp64 (each may be NULL). */
void oracle_bwd_bwd_golden(const void* ddx, const void* ddg, const void* dy, const void* x, const void* gamma,
                           int64_t M, int64_t N, double eps, int dt, int offset, double* d_dy, double* d_x,
                           double* d_gamma) {
    if (d_gamma)
        for (int64_t j = 0; j < N; ++j) d_gamma[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double xv = load_elem(x, row + j, dt);
            ss += xv * xv;
        }
        const double r = 1.0 / sqrt(ss / (double)N + eps);
        double sc = 0.0, sa = 0.0, sb = 0.0, sd = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double w = load_elem(gamma, j, dt);
            const double g = offset ? 1.0 + w : w;
            const double xv = load_elem(x, row + j, dt);
            const double dyv = load_elem(dy, row + j, dt);
            const double u = dyv * g;
            const double t = load_elem(ddx, row + j, dt);
            const double q = ddg ? load_elem(ddg, j, dt) : 0.0;
            sc += u * xv;
            sa += t * xv;
            sb += t * u;
            sd += q * dyv * xv;
        }
        const double c = sc / (double)N, A = sa / (double)N, Bm = sb / (double)N, D = sd / (double)N;
        const double r2 = r * r, r3 = r2 * r, r5 = r3 * r2;
        for (int64_t j = 0; j < N; ++j) {
            const double w = load_elem(gamma, j, dt);
            const double g = offset ? 1.0 + w : w;
            const double xv = load_elem(x, row + j, dt);
            const double dyv = load_elem(dy, row + j, dt);
            const double u = dyv * g;
            const double t = load_elem(ddx, row + j, dt);
            const double q = ddg ? load_elem(ddg, j, dt) : 0.0;
            const double e = t - r2 * xv * A;
            if (d_dy) d_dy[row + j] = g * r * e + r * xv * q;
            if (d_x) d_x[row + j] = r * q * dyv - r3 * (c * t + u * A + xv * (Bm + D)) + 3.0 * r5 * c * A * xv;
            if (d_gamma) d_gamma[j] += r * dyv * e;
        }
    }
}

/* Same outputs in dtype dt from fp32 intermediates: r recomputed as in the
 * forward reference, the four row sums sequential, then, step by step,
 *   e = t - (r2*x)*A;  d_dy = (g*r)*e + (r*x)*q;
 *   d_x = ((r*q)*dy - r3*((c*t + u*A) + x*(B + D))) + ((3*r5)*(c*A))*x;
 *   d_gamma accumulates (r*dy)*e over rows in row order. */
void oracle_bwd_bwd_reference(const void* ddx, const void* ddg, const void* dy, const void* x, const void* gamma,
                              int64_t M, int64_t N, float eps, int dt, int offset, void* d_dy, void* d_x,
                              void* d_gamma) {
    float* acc = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0f;
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * N;
        const float r = row_rstd_f32(x, row, N, eps, dt);
        float sc = 0.0f, sa = 0.0f, sb = 0.0f, sd = 0.0f;
        for (int64_t j = 0; j < N; ++j) {
            const float w = ld32(gamma, j, dt);
            const float g = offset ? 1.0f + w : w;
            const float xv = ld32(x, row + j, dt);
            const float dyv = ld32(dy, row + j, dt);
            const float u = dyv * g;
            const float t = ld32(ddx, row + j, dt);
            const float q = ddg ? ld32(ddg, j, dt) : 0.0f;
            const float ux = u * xv;
            const float tx = t * xv;
            const float tu = t * u;
            const float qd = q * dyv;
            const float qdx = qd * xv;
            sc = sc + ux;
            sa = sa + tx;
            sb = sb + tu;
            sd = sd + qdx;
        }
        const float c = sc / (float)N, A = sa / (float)N, Bm = sb / (float)N, D = sd / (float)N;
        const float r2 = r * r;
        const float r3 = r2 * r;
        const float r5 = r3 * r2;
        const float k5 = (3.0f * r5) * (c * A);
        const float bd = Bm + D;
        for (int64_t j = 0; j < N; ++j) {
            const float w = ld32(gamma, j, dt);
            const float g = offset ? 1.0f + w : w;
            const float xv = ld32(x, row + j, dt);
            const float dyv = ld32(dy, row + j, dt);
            const float u = dyv * g;
            const float t = ld32(ddx, row + j, dt);
            const float q = ddg ? ld32(ddg, j, dt) : 0.0f;
            const float r2x = r2 * xv;
            const float r2xa = r2x * A;
            const float e = t - r2xa;
            if (d_dy) {
                const float a1 = (g * r) * e;
                const float a2 = (r * xv) * q;
                store_elem(d_dy, row + j, dt, (double)(a1 + a2));
            }
            if (d_x) {
                const float b1 = (r * q) * dyv;
                const float ct = c * t;
                const float ua = u * A;
                const float xbd = xv * bd;
                const float inner = (ct + ua) + xbd;
                const float b2 = r3 * inner;
                const float b3 = k5 * xv;
                store_elem(d_x, row + j, dt, (double)((b1 - b2) + b3));
            }
            const float re = (r * dyv) * e;
            acc[j] = acc[j] + re;
        }
    }
    if (d_gamma)
        for (int64_t j = 0; j < N; ++j) store_elem(d_gamma, j, dt, (double)acc[j]);
    free(acc);
}

/* ------------------------------------------------------------------------- */
/* dgamma with pairwise row sums (a report-only second reference)             */
/* ------------------------------------------------------------------------- */

/* fp32 pairwise (recursive halving) sum of t[lo .. hi). */
static float pairwise_sum_f32(const float* t, int64_t lo, int64_t hi) {
    const int64_t n = hi - lo;
    if (n <= 0) return 0.0f;
    if (n == 1) return t[lo];
    const int64_t mid = lo + n / 2;
    const float a = pairwise_sum_f32(t, lo, mid);
    const float b = pairwise_sum_f32(t, mid, hi);
    return a + b;
}

/*
 * dgamma[N] in dtype dt: the same fp32 terms as oracle_bwd_reference,
 * (dy * x) * r with r recomputed in fp32 per row, but summed over the rows by a
 * pairwise tree (error growing with log2 M rather than M), rounded once. The
 * gate reports the target's distance from it next to the sequential reference
 * (the pages leave the summation order of the reference open).
 */
void oracle_dgamma_pairwise_reference(const void* dy, const void* x, const void* gamma, int64_t M, int64_t N,
                                      float eps, int dt, int offset, void* dgamma) {
    (void)gamma;
    (void)offset;  /* dgamma has the same formula with and without the offset */
    float* r = (float*)malloc((size_t)(M > 0 ? M : 1) * sizeof(float));
    float* t = (float*)malloc((size_t)(M > 0 ? M : 1) * sizeof(float));
    for (int64_t i = 0; i < M; ++i) r[i] = row_rstd_f32(x, i * N, N, eps, dt);
    for (int64_t j = 0; j < N; ++j) {
        for (int64_t i = 0; i < M; ++i) {
            const float dyx = ld32(dy, i * N + j, dt) * ld32(x, i * N + j, dt);
            t[i] = dyx * r[i];
        }
        store_elem(dgamma, j, dt, (double)pairwise_sum_f32(t, 0, M));
    }
    free(r);
    free(t);
}
