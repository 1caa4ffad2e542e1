/*
 * Oracle for the Quant VideoGen KV-cache compression path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, fp64 CPU statement of what
 * the method computes.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load it.  The CUDA library shares no code, header,
 * table or constant with this file, and never calls it.
 *
 * Sources, by page and section (the pages are web write-ups of arXiv 2602.02958):
 *   [notes/SAS]   "Quant VideoGen" (note.zhuruihan.top), section Semantic-Aware Smoothing:
 *                 k-means over the sequence axis; each group's centroid is its mean; the
 *                 residual is the token minus its group's centroid.
 *   [notes/PRQ]   same page, section Progressive Residual Quantization: the smoothing is
 *                 re-applied to the residual for T stages, only the last residual is
 *                 quantized, and reconstruction adds the centroids back from stage T to 1.
 *   [notes/co-design] same page, section Algorithm-System Co-design: per-group scales are
 *                 FP8 E4M3; the previous chunk's centroids seed the next chunk's k-means.
 *   [review/pipeline] "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成"
 *                 (paper.rainbus.top), the pipeline paragraph: X in R^{N x d}, C groups,
 *                 R^(0) = X, stage t gives (R^(t), C^(t), pi^(t)), X_INT, S_x = Q(R^(T)),
 *                 X^(t-1) = X^(t) + C^(t)_{pi_i}.
 *   [explainer/steps] "Quant VideoGen: Auto-Regressive Long Video Generation via 2-Bit
 *                 KV-Cache Quantization" (howistudyai.com), Step-by-step: per-group scales
 *                 in FP8, INT2/INT4 codes, block size B, pi stored as uint8 with K = 256.
 *
 * Readings taken where the pages say nothing (each one is also listed in the design notes):
 *   - k-means is Lloyd's algorithm on squared Euclidean distance, computed directly as
 *     sum_k (r_k - c_k)^2, ties going to the lowest cluster index.  One round is an
 *     assignment followed by a mean update; `iters` rounds are run.  The stored pi is the
 *     last assignment and the stored centroid is the mean under it.  An empty cluster
 *     keeps its previous centroid.
 *   - Centroids are stored as fp32, rounded to nearest even after every update.  Residuals
 *     are taken against those stored fp32 centroids, exactly (in fp64).  A 16-bit storage
 *     variant (the explainer page's compression ratios count centroids in 16 bits) keeps
 *     them as IEEE binary16 or bfloat16 instead (centroid_format 1 / 2): the exact mean,
 *     and the cold-start rows and warm tables, are rounded once to that format, and the
 *     residuals are taken against the rounded values.
 *   - Cold start: C distinct rows of R^(t-1), chosen by a partial Fisher-Yates shuffle
 *     driven by SplitMix64 (Steele, Lea, Flood 2014; Vigna's published constants), seeded
 *     with seed ^ (tensor_id * 0x9E3779B97F4A7C15) ^ t.  Warm start: the caller's
 *     centroids for stage t.
 *   - Q(.) is symmetric on the restricted grid q in [-qmax, qmax], qmax = 2^(b-1) - 1.
 *     A group is `group` contiguous channels of one token.  s = max|r| / qmax; the stored
 *     scale is E4M3(s), rounded to nearest even and saturated to +-448; q is r / s_q
 *     rounded half-to-even and clamped; the stored code is u = q + 2^(b-1).  When
 *     s_q == 0 every code is 2^(b-1).
 *   - Scheme 1 (mid-rise, the reading of a critique's "only 4 quantization levels" at 2
 *     bits): the 2^b levels sit at half-integers, x = s_q * (u - 2^(b-1) + 1/2) for
 *     u = 0 .. 2^b - 1.  s = max|r| / (2^(b-1) - 1/2), so the largest |r| maps to the
 *     outermost level; u = floor(r / s_q) + 2^(b-1), clamped to [0, 2^b - 1], the nearest
 *     level (a value exactly between two levels takes the upper one).  When s_q == 0 every
 *     code is 2^(b-1).
 *   - Codes are packed little-endian inside a byte: channel k sits at bit (k*b) mod 8 of
 *     byte (k*b)/8 of its token's row.
 *
 * Everything is fp64 except where the method stores a narrower type (fp32 centroids,
 * E4M3 scales, integer codes).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------------------ */
/* FP8 E4M3 as defined by the OCP 8-bit floating point specification: 1 sign bit, 4     */
/* exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN.         */
/* ------------------------------------------------------------------------------------ */

double orc_e4m3_decode(uint8_t b) {
    int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* subnormal: (m / 8) * 2^(1 - 7) */
    else
        v = ldexp((double)(8 + m), e - 10); /* normal: (1 + m / 8) * 2^(e - 7) */
    return sign ? -v : v;
}

/* Nearest E4M3 value, ties to the even code, magnitudes past the largest finite value
 * clamp to it (saturate-to-finite).  Done by plain search over the 127 finite
 * non-negative codes so that it can be checked by eye. */
uint8_t orc_e4m3_encode(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* saturate to the largest finite value */
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; c++) {
        double err = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

void orc_e4m3_encode_n(const double *x, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_n(const uint8_t *b, int64_t n, double *out) {
    for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_decode(b[i]);
}

/* ------------------------------------------------------------------------------------ */
/* Seeded cold start.                                                                     */
/* ------------------------------------------------------------------------------------ */

uint64_t orc_splitmix64_next(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* idx[0..C) = the first C entries of a partial Fisher-Yates shuffle of 0..N-1. */
int orc_init_indices(uint64_t seed, int64_t tensor_id, int stage, int64_t N, int C,
                     int64_t *idx) {
    if (N < 1 || C < 1 || C > N) return -1;
    int64_t *perm = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    if (!perm) return -2;
    for (int64_t i = 0; i < N; i++) perm[i] = i;
    uint64_t state = seed ^ ((uint64_t)tensor_id * 0x9E3779B97F4A7C15ULL) ^ (uint64_t)stage;
    for (int j = 0; j < C; j++) {
        uint64_t r = orc_splitmix64_next(&state);
        int64_t k = j + (int64_t)(r % (uint64_t)(N - j));
        int64_t tmp = perm[j];
        perm[j] = perm[k];
        perm[k] = tmp;
        idx[j] = perm[j];
    }
    free(perm);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Semantic-Aware Smoothing building blocks [notes/SAS], [review/pipeline] (a)-(c).      */
/* ------------------------------------------------------------------------------------ */

static double orc_sqdist(const double *r, const float *c, int d) {
    double s = 0.0;
    for (int k = 0; k < d; k++) {
        double diff = r[k] - (double)c[k];
        s += diff * diff;
    }
    return s;
}

/* (a) pi_i = argmin_j ||R_i - cent_j||^2, lowest j on ties.  dist, if given, receives the
 * chosen squared distance. */
void orc_assign(const double *R, int64_t N, int d, const float *cent, int C, int32_t *pi,
                double *dist) {
    for (int64_t i = 0; i < N; i++) {
        double best = INFINITY;
        int bj = 0;
        for (int j = 0; j < C; j++) {
            double D = orc_sqdist(R + i * d, cent + (int64_t)j * d, d);
            if (D < best) {
                best = D;
                bj = j;
            }
        }
        pi[i] = bj;
        if (dist) dist[i] = best;
    }
}

/* (b) cent_j = fp32(mean of the rows assigned to j); empty clusters keep cent_j.
 * counts, if given, receives the cluster sizes. */
/* ------------------------------------------------------------------------------------ */
/* Centroid storage formats: 0 fp32, 1 IEEE binary16, 2 bfloat16.  A stored centroid is   */
/* the exact mean rounded once to the format, to nearest even; residuals are then taken   */
/* against that stored value.  The rounding is written from the formats' definitions:    */
/* p significand bits, smallest normal exponent emin (subnormals keep emin's quantum),    */
/* and values past the largest finite one rounding to infinity.                           */
/* ------------------------------------------------------------------------------------ */

static double orc_round_p(double x, int p, int emin, double maxfinite) {
    if (x != x || x == 0.0 || isinf(x)) return x;
    int ex;
    frexp(fabs(x), &ex); /* |x| = m 2^ex, m in [0.5, 1): the leading bit has weight 2^(ex-1) */
    int e = ex - 1;
    if (e < emin) e = emin;
    const double q = ldexp(1.0, e - (p - 1));
    double r = nearbyint(fabs(x) / q) * q; /* exact scaling; nearest, ties to even */
    if (r > maxfinite) r = INFINITY;
    return copysign(r, x);
}

float orc_store(double v, int format) {
    if (format == 1) return (float)orc_round_p(v, 11, -14, 65504.0);
    if (format == 2) return (float)orc_round_p(v, 8, -126, ldexp(255.0, 120));
    return (float)v;
}

void orc_store_n(const double *x, int64_t n, int format, float *out) {
    for (int64_t i = 0; i < n; i++) out[i] = orc_store(x[i], format);
}

static void orc_update_fmt(const double *R, int64_t N, int d, const int32_t *pi, int C,
                           float *cent, int64_t *counts, int format);

void orc_update(const double *R, int64_t N, int d, const int32_t *pi, int C, float *cent,
                int64_t *counts) {
    orc_update_fmt(R, N, d, pi, C, cent, counts, 0);
}

static void orc_update_fmt(const double *R, int64_t N, int d, const int32_t *pi, int C,
                           float *cent, int64_t *counts, int format) {
    double *sum = (double *)calloc((size_t)C * d, sizeof(double));
    int64_t *n = (int64_t *)calloc((size_t)C, sizeof(int64_t));
    for (int64_t i = 0; i < N; i++) {
        int j = pi[i];
        n[j] += 1;
        for (int k = 0; k < d; k++) sum[(int64_t)j * d + k] += R[i * d + k];
    }
    for (int j = 0; j < C; j++) {
        if (n[j] == 0) continue;
        for (int k = 0; k < d; k++)
            cent[(int64_t)j * d + k] = orc_store(sum[(int64_t)j * d + k] / (double)n[j], format);
    }
    if (counts)
        for (int j = 0; j < C; j++) counts[j] = n[j];
    free(sum);
    free(n);
}

/* Lloyd objective sum_i ||R_i - cent_{pi_i}||^2. */
double orc_objective(const double *R, int64_t N, int d, const int32_t *pi, const float *cent) {
    double J = 0.0;
    for (int64_t i = 0; i < N; i++) J += orc_sqdist(R + i * d, cent + (int64_t)pi[i] * d, d);
    return J;
}

/* (c) R_i <- R_i - cent_{pi_i}, exact in fp64. */
void orc_subtract(double *R, int64_t N, int d, const int32_t *pi, const float *cent) {
    for (int64_t i = 0; i < N; i++)
        for (int k = 0; k < d; k++) R[i * d + k] -= (double)cent[(int64_t)pi[i] * d + k];
}

/* One smoothing stage: `iters` Lloyd rounds from the centroids already in `cent`. */
static void orc_lloyd_fmt(const double *R, int64_t N, int d, int C, int iters, float *cent,
                          int32_t *pi, int format) {
    for (int it = 0; it < iters; it++) {
        orc_assign(R, N, d, cent, C, pi, NULL);
        orc_update_fmt(R, N, d, pi, C, cent, NULL, format);
    }
}

void orc_lloyd(const double *R, int64_t N, int d, int C, int iters, float *cent, int32_t *pi) {
    orc_lloyd_fmt(R, N, d, C, iters, cent, pi, 0);
}

/* ------------------------------------------------------------------------------------ */
/* Q(.) of the final residual [review/pipeline], [notes/co-design], [explainer/steps].    */
/* ------------------------------------------------------------------------------------ */

void orc_encode(const double *R, int64_t N, int d, int bits, int group, int scheme,
                uint8_t *codes, uint8_t *scales) {
    const int qmax = (1 << (bits - 1)) - 1, mid = 1 << (bits - 1);
    /* the outermost level: qmax for the symmetric grid, 2^(b-1) - 1/2 for mid-rise */
    const double top = scheme == 1 ? (double)mid - 0.5 : (double)qmax;
    const int row_bytes = d * bits / 8, ngroups = d / group;
    memset(codes, 0, (size_t)N * row_bytes);
    for (int64_t i = 0; i < N; i++) {
        const double *r = R + i * d;
        for (int g = 0; g < ngroups; g++) {
            double a = 0.0;
            for (int k = g * group; k < (g + 1) * group; k++)
                if (fabs(r[k]) > a) a = fabs(r[k]);
            uint8_t sb = orc_e4m3_encode(a / top);
            double sq = orc_e4m3_decode(sb);
            scales[i * ngroups + g] = sb;
            for (int k = g * group; k < (g + 1) * group; k++) {
                int u = mid;
                if (sq != 0.0 && scheme == 1) {
                    double f = floor(r[k] / sq) + mid;
                    if (f > 2 * mid - 1) f = 2 * mid - 1;
                    if (f < 0) f = 0;
                    u = (int)f;
                } else if (sq != 0.0) {
                    double q = nearbyint(r[k] / sq); /* default rounding: half to even */
                    if (q > qmax) q = qmax;
                    if (q < -qmax) q = -qmax;
                    u = (int)q + mid;
                }
                codes[i * row_bytes + (k * bits) / 8] |= (uint8_t)(u << ((k * bits) % 8));
            }
        }
    }
}

/* deQ(X_INT, S_x) in fp64. */
void orc_decode_codes(const uint8_t *codes, const uint8_t *scales, int64_t N, int d, int bits,
                      int group, int scheme, double *out) {
    const int mid = 1 << (bits - 1), row_bytes = d * bits / 8, ngroups = d / group;
    const double off = scheme == 1 ? 0.5 : 0.0;
    for (int64_t i = 0; i < N; i++)
        for (int k = 0; k < d; k++) {
            int u = (codes[i * row_bytes + (k * bits) / 8] >> ((k * bits) % 8)) & ((1 << bits) - 1);
            double sq = orc_e4m3_decode(scales[i * ngroups + k / group]);
            out[i * d + k] = sq * ((double)(u - mid) + off);
        }
}

/* Reconstruction: X^(T) = deQ, then X^(t-1) = X^(t) + C^(t)_{pi_i} for t = T..1
 * [review/pipeline], [notes/PRQ].  pi is [T][N], cent is [T][C][d]. */
void orc_dequantize(const uint8_t *codes, const uint8_t *scales, const uint8_t *pi,
                    const float *cent, int64_t N, int d, int C, int T, int bits, int group,
                    int scheme, double *out) {
    orc_decode_codes(codes, scales, N, d, bits, group, scheme, out);
    for (int t = T; t >= 1; t--) {
        const uint8_t *p = pi + (int64_t)(t - 1) * N;
        const float *c = cent + (int64_t)(t - 1) * C * d;
        for (int64_t i = 0; i < N; i++)
            for (int k = 0; k < d; k++) out[i * d + k] += (double)c[(int64_t)p[i] * d + k];
    }
}

/* ------------------------------------------------------------------------------------ */
/* The whole quantize path for one tensor [review/pipeline] steps 1-3.                   */
/* ------------------------------------------------------------------------------------ */

typedef struct {
    int64_t N;
    int d, C, T, bits, group, iters;
    uint64_t seed;
    int scheme;          /* 0: symmetric restricted grid, 1: mid-rise */
    int centroid_format; /* 0: fp32, 1: binary16, 2: bfloat16 (see orc_store) */
} orc_cfg;

/* X [N][d] fp64 (decoded input); warm [T][C][d] or NULL; outputs codes [N][d*bits/8],
 * scales [N][d/group], pi [T][N], cent [T][C][d], J [T] (objective of each stage, may be
 * NULL), Rfin [N][d] (final residual, may be NULL). */
int orc_quantize_tensor(const orc_cfg *cfg, int64_t tensor_id, const double *X,
                        const float *warm, uint8_t *codes, uint8_t *scales, uint8_t *pi,
                        float *cent, double *J, double *Rfin) {
    const int64_t N = cfg->N;
    const int d = cfg->d, C = cfg->C;
    double *R = (double *)malloc((size_t)N * d * sizeof(double));
    int32_t *p = (int32_t *)malloc((size_t)N * sizeof(int32_t));
    int64_t *idx = (int64_t *)malloc((size_t)C * sizeof(int64_t));
    if (!R || !p || !idx) {
        free(R), free(p), free(idx);
        return -2;
    }
    memcpy(R, X, (size_t)N * d * sizeof(double)); /* R^(0) = X */
    for (int t = 1; t <= cfg->T; t++) {
        float *c = cent + (int64_t)(t - 1) * C * d;
        if (warm) {
            const float *w = warm + (int64_t)(t - 1) * C * d;
            for (int64_t x = 0; x < (int64_t)C * d; x++) c[x] = orc_store((double)w[x], cfg->centroid_format);
        } else {
            if (orc_init_indices(cfg->seed, tensor_id, t, N, C, idx) != 0) {
                free(R), free(p), free(idx);
                return -1;
            }
            for (int j = 0; j < C; j++)
                for (int k = 0; k < d; k++)
                    c[(int64_t)j * d + k] = orc_store(R[idx[j] * d + k], cfg->centroid_format);
        }
        orc_lloyd_fmt(R, N, d, C, cfg->iters, c, p, cfg->centroid_format);
        if (J) J[t - 1] = orc_objective(R, N, d, p, c);
        for (int64_t i = 0; i < N; i++) pi[(int64_t)(t - 1) * N + i] = (uint8_t)p[i];
        orc_subtract(R, N, d, p, c); /* R^(t) */
    }
    orc_encode(R, N, d, cfg->bits, cfg->group, cfg->scheme, codes, scales);
    if (Rfin) memcpy(Rfin, R, (size_t)N * d * sizeof(double));
    free(R), free(p), free(idx);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* A batch of independent tensors, spread over host threads.                             */
/* ------------------------------------------------------------------------------------ */

typedef struct {
    const orc_cfg *cfg;
    int64_t H, tensor_id_base;
    const double *X;
    const float *warm;
    uint8_t *codes, *scales, *pi;
    float *cent;
    double *J;
    int tid, nthreads, status;
} orc_job;

static void *orc_worker(void *arg) {
    orc_job *jb = (orc_job *)arg;
    const orc_cfg *c = jb->cfg;
    const int64_t N = c->N;
    for (int64_t h = jb->tid; h < jb->H; h += jb->nthreads) {
        int rc = orc_quantize_tensor(
            c, jb->tensor_id_base + h, jb->X + h * N * c->d,
            jb->warm ? jb->warm + h * (int64_t)c->T * c->C * c->d : NULL,
            jb->codes + h * N * (c->d * c->bits / 8), jb->scales + h * N * (c->d / c->group),
            jb->pi + h * (int64_t)c->T * N, jb->cent + h * (int64_t)c->T * c->C * c->d,
            jb->J ? jb->J + h * c->T : NULL, NULL);
        if (rc != 0) jb->status = rc;
    }
    return NULL;
}

int orc_num_cores(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

int orc_quantize(int64_t H, int64_t N, int d, int C, int T, int bits, int group, int iters,
                 uint64_t seed, int64_t tensor_id_base, const double *X, const float *warm,
                 uint8_t *codes, uint8_t *scales, uint8_t *pi, float *cent, double *J,
                 int nthreads, int scheme, int centroid_format) {
    if (H < 0 || N < 1 || d < 1 || T < 0 || iters < 1) return -1;
    if (T > 0 && (C < 1 || C > 256 || C > N)) return -1;
    if ((bits != 2 && bits != 4) || group < 1 || d % group != 0 || (d * bits) % 8 != 0) return -1;
    if (scheme != 0 && scheme != 1) return -1;
    if (centroid_format < 0 || centroid_format > 2) return -1;
    orc_cfg cfg = {N, d, C, T, bits, group, iters, seed, scheme, centroid_format};
    if (nthreads <= 0) nthreads = orc_num_cores();
    if (nthreads > H) nthreads = (int)(H > 0 ? H : 1);
    orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (orc_job){&cfg, H, tensor_id_base, X, warm, codes, scales, pi, cent, J,
                            i, nthreads, 0};
        pthread_create(&th[i], NULL, orc_worker, &jobs[i]);
    }
    int status = 0;
    for (int i = 0; i < nthreads; i++) {
        pthread_join(th[i], NULL);
        if (jobs[i].status) status = jobs[i].status;
    }
    free(jobs);
    free(th);
    return status;
}
