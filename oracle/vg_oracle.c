/*
 * vg_oracle.c -- CPU reference for the NVFP4 / row-scaled FP8 verify GEMV.
 *
 * TEST INFRASTRUCTURE ONLY (see vg_oracle.h).  Plain C99, no blocking, no
 * fusion, no reordering beyond the definitions below.  Build with
 * -ffp-contract=off so that every FP32 step of the quantisation recipe is
 * one IEEE operation with one rounding.
 *
 * Sources for what is computed:
 *  - The product and the 1-8 column widths: mtp7-device-confidence engine
 *    card, Design table ("GEMVs": FP8 and NVFP4 bytes fed to BF16 MMA
 *    fragments) and Decode row (verify pass over 2-8 columns).
 *  - Checks against FP64: same card, Checks section.
 *  - Round-to-nearest post-training quantisation to NVFP4 / FP8: crit
 *    landing page, "Models" paragraph; row-scaled FP8: card, Model section.
 *  - The pages do not define the bit formats.  E2M1 and E4M3 follow the
 *    public OCP Microscaling and OCP 8-bit floating point definitions; the
 *    quantisation order (tensor scale amax/(6*448), block scale
 *    blockamax/6 in tensor-scale units, RNE with saturation) is the plainest
 *    reading of the recipe.
 */
#include "vg_oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decode */

/* E2M1 magnitudes indexed by the low three bits of the code. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double vgo_e2m1_value(int code)
{
    double v = E2M1_MAG[code & 7];
    return (code & 8) ? -v : v;
}

double vgo_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int f = byte & 7;
    double v;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);                 /* subnormal: f * 2^-9 */
    else
        v = ldexp(1.0 + f / 8.0, e - 7);          /* 2^(e-7) * (1 + f/8) */
    return s ? -v : v;
}

double vgo_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------- encode */

int vgo_e4m3_encode(float v)
{
    int sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    int ex, E, n;
    double quantum, r;
    if (isnan(v))
        return sign | 0x7F;
    if (a >= 448.0)
        return sign | 0x7E;                       /* satfinite */
    if (a == 0.0)
        return sign;
    /* binade of a: a = m * 2^ex with m in [0.5, 1) -> a in [2^(ex-1), 2^ex) */
    frexp(a, &ex);
    E = ex - 1;
    if (E < -6)
        E = -6;                                   /* subnormal spacing 2^-9 */
    quantum = ldexp(1.0, E - 3);                  /* 3 mantissa bits */
    r = nearbyint(a / quantum);                   /* ties to even multiple */
    n = (int)r;
    /* value = n * quantum; n in [0, 16].  Re-express as an E4M3 code. */
    if (E == -6 && n < 8)
        return sign | n;                          /* subnormal f = n */
    if (n == 16) {                                /* rounded up a binade */
        n = 8;
        E += 1;
    }
    /* n in [8, 15]: value = 2^E * n/8 = 2^E * (1 + (n-8)/8) */
    return sign | ((E + 7) << 3) | (n - 8);
}

int vgo_e2m1_encode(float v)
{
    int sign = signbit(v) ? 8 : 0;
    float a = fabsf(v);
    int mag;
    /* nearest of {0,.5,1,1.5,2,3,4,6}; a midpoint goes to the code with an
     * even mantissa bit (codes 0,2,4,6 have mantissa 0); above 6 saturates */
    if (a <= 0.25f)       mag = 0;
    else if (a < 0.75f)   mag = 1;
    else if (a <= 1.25f)  mag = 2;
    else if (a < 1.75f)   mag = 3;
    else if (a <= 2.5f)   mag = 4;
    else if (a < 3.5f)    mag = 5;
    else if (a <= 5.0f)   mag = 6;
    else                  mag = 7;
    return sign | mag;
}

/* ------------------------------------------------------------- quantise */

static int all_finite(const float *W, int64_t n)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        if (!(fabsf(W[i]) <= FLT_MAX))
            return 0;
    return 1;
}

float vgo_amax(const float *W, int64_t n)
{
    int64_t i;
    float amax = 0.0f;
    for (i = 0; i < n; ++i)
        if (fabsf(W[i]) > amax)
            amax = fabsf(W[i]);
    return amax;
}

void vgo_nvfp4_quantise_gs(const float *W, int64_t M, int64_t K, float gs,
                           uint8_t *nib, uint8_t *sc)
{
    int64_t m, b;
    memset(nib, 0, (size_t)(M * (K / 2)));
    for (m = 0; m < M; ++m) {
        for (b = 0; b < K / 16; ++b) {
            const float *w = W + m * K + b * 16;
            float bamax = 0.0f, d;
            int code, j;
            for (j = 0; j < 16; ++j)
                if (fabsf(w[j]) > bamax)
                    bamax = fabsf(w[j]);
            if (gs == 0.0f) {
                code = 0;
            } else {
                float t = bamax / gs;             /* block max in gs units */
                float s = t / 6.0f;               /* scale for a max of 6 */
                code = vgo_e4m3_encode(s);
            }
            sc[m * (K / 16) + b] = (uint8_t)code;
            d = (float)vgo_e4m3_value(code) * gs; /* one FP32 rounding */
            for (j = 0; j < 16; ++j) {
                int c = (d == 0.0f) ? 0 : vgo_e2m1_encode(w[j] / d);
                int64_t k = b * 16 + j;
                uint8_t *p = nib + m * (K / 2) + k / 2;
                if (k & 1)
                    *p = (uint8_t)(*p | (c << 4));
                else
                    *p = (uint8_t)(*p | c);
            }
        }
    }
}

int vgo_nvfp4_quantise(const float *W, int64_t M, int64_t K,
                       uint8_t *nib, uint8_t *sc, float *gs_out)
{
    float gs;
    if (!all_finite(W, M * K))
        return -1;
    gs = vgo_amax(W, M * K) / 2688.0f;            /* 2688 = 6 * 448 */
    *gs_out = gs;
    vgo_nvfp4_quantise_gs(W, M, K, gs, nib, sc);
    return 0;
}

int vgo_fp8_quantise(const float *W, int64_t M, int64_t K,
                     uint8_t *q, float *rs_out)
{
    int64_t m, k;
    if (!all_finite(W, M * K))
        return -1;
    for (m = 0; m < M; ++m) {
        const float *w = W + m * K;
        float ramax = 0.0f, rs;
        for (k = 0; k < K; ++k)
            if (fabsf(w[k]) > ramax)
                ramax = fabsf(w[k]);
        rs = ramax / 448.0f;
        rs_out[m] = rs;
        for (k = 0; k < K; ++k)
            q[m * K + k] = (uint8_t)((rs == 0.0f) ? 0 : vgo_e4m3_encode(w[k] / rs));
    }
    return 0;
}

/* -------------------------------------------------------------- dequant */

void vgo_nvfp4_dequant(const uint8_t *nib, const uint8_t *sc, float gs,
                       int64_t M, int64_t K, double *What)
{
    int64_t m, k;
    for (m = 0; m < M; ++m)
        for (k = 0; k < K; ++k) {
            uint8_t byte = nib[m * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            What[m * K + k] = vgo_e2m1_value(code)
                            * vgo_e4m3_value(sc[m * (K / 16) + k / 16])
                            * (double)gs;
        }
}

void vgo_fp8_dequant(const uint8_t *q, const float *rs,
                     int64_t M, int64_t K, double *What)
{
    int64_t m, k;
    for (m = 0; m < M; ++m)
        for (k = 0; k < K; ++k)
            What[m * K + k] = vgo_e4m3_value(q[m * K + k]) * (double)rs[m];
}

/* ----------------------------------------------------------------- gemv */

typedef struct {
    int fp8;                                      /* 1 FP8 row-scaled, 2 MXFP8, 3 INT4 groups */
    const uint8_t *nib, *sc, *q;
    const uint16_t *gsc;                          /* INT4 group scales (BF16) */
    const float *rs;
    float gs;
    const uint16_t *x;
    int N;
    int64_t M, K;
    const int64_t *rows;
    int64_t nrows, r0, r1;
    double *y, *a;
    double *xd;                                   /* x decoded, [N][K] */
} gemv_job;

/* One output row: decode row m of W to FP64, then for every column n the
 * FP64 sum over k of w*x and of |w*x|, k in increasing order. */
static void gemv_row(const gemv_job *j, int64_t r, double *wrow)
{
    int64_t m = j->rows ? j->rows[r] : r;
    int64_t k;
    int n;
    for (k = 0; k < j->K; ++k) {
        if (j->fp8 == 1) {
            wrow[k] = vgo_e4m3_value(j->q[m * j->K + k]) * (double)j->rs[m];
        } else if (j->fp8 == 2) {
            wrow[k] = vgo_e4m3_value(j->q[m * j->K + k])
                    * vgo_e8m0_value(j->sc[m * (j->K / 32) + k / 32]);
        } else if (j->fp8 == 3) {
            uint8_t byte = j->nib[m * (j->K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            wrow[k] = (double)(code - 8) * vgo_bf16_value(j->gsc[m * (j->K / 128) + k / 128]);
        } else {
            uint8_t byte = j->nib[m * (j->K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            wrow[k] = vgo_e2m1_value(code)
                    * vgo_e4m3_value(j->sc[m * (j->K / 16) + k / 16])
                    * (double)j->gs;
        }
    }
    for (n = 0; n < j->N; ++n) {
        const double *xn = j->xd + (int64_t)n * j->K;
        double s = 0.0, sa = 0.0;
        for (k = 0; k < j->K; ++k) {
            double p = wrow[k] * xn[k];               /* exact in FP64 */
            s += p;
            sa += fabs(p);
        }
        j->y[(int64_t)n * j->nrows + r] = s;
        j->a[(int64_t)n * j->nrows + r] = sa;
    }
}

static void *gemv_worker(void *arg)
{
    const gemv_job *j = (const gemv_job *)arg;
    double *wrow = (double *)malloc(sizeof(double) * (size_t)(j->K ? j->K : 1));
    int64_t r;
    for (r = j->r0; r < j->r1; ++r)
        gemv_row(j, r, wrow);
    free(wrow);
    return NULL;
}

static void gemv_run(gemv_job *base, int threads)
{
    int64_t i, total = (int64_t)base->N * base->K;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(total ? total : 1));
    int t;
    for (i = 0; i < total; ++i)
        xd[i] = vgo_bf16_value(base->x[i]);
    base->xd = xd;
    if (threads <= 1 || base->nrows < 2 * threads) {
        base->r0 = 0;
        base->r1 = base->nrows;
        gemv_worker(base);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
        gemv_job *jobs = (gemv_job *)malloc(sizeof(gemv_job) * (size_t)threads);
        for (t = 0; t < threads; ++t) {
            jobs[t] = *base;
            jobs[t].r0 = base->nrows * t / threads;
            jobs[t].r1 = base->nrows * (t + 1) / threads;
            pthread_create(&tid[t], NULL, gemv_worker, &jobs[t]);
        }
        for (t = 0; t < threads; ++t)
            pthread_join(tid[t], NULL);
        free(tid);
        free(jobs);
    }
    free(xd);
}

void vgo_gemv_nvfp4(const uint8_t *nib, const uint8_t *sc, float gs,
                    const uint16_t *x, int N, int64_t M, int64_t K,
                    const int64_t *rows, int64_t nrows,
                    double *y, double *a, int threads)
{
    gemv_job j;
    memset(&j, 0, sizeof j);
    j.nib = nib; j.sc = sc; j.gs = gs; j.x = x; j.N = N; j.M = M; j.K = K;
    j.rows = rows; j.nrows = rows ? nrows : M; j.y = y; j.a = a;
    gemv_run(&j, threads);
}

void vgo_gemv_mxfp8(const uint8_t *q, const uint8_t *sc, const uint16_t *x, int N, int64_t M,
                    int64_t K, const int64_t *rows, int64_t nrows, double *y, double *a,
                    int threads)
{
    gemv_job j;
    memset(&j, 0, sizeof j);
    j.fp8 = 2; j.q = q; j.sc = sc; j.x = x; j.N = N; j.M = M; j.K = K;
    j.rows = rows; j.nrows = rows ? nrows : M; j.y = y; j.a = a;
    gemv_run(&j, threads);
}

void vgo_gemv_int4g(const uint8_t *nib, const uint16_t *sc, const uint16_t *x, int N, int64_t M,
                    int64_t K, const int64_t *rows, int64_t nrows, double *y, double *a,
                    int threads)
{
    gemv_job j;
    memset(&j, 0, sizeof j);
    j.fp8 = 3; j.nib = nib; j.gsc = sc; j.x = x; j.N = N; j.M = M; j.K = K;
    j.rows = rows; j.nrows = rows ? nrows : M; j.y = y; j.a = a;
    gemv_run(&j, threads);
}

void vgo_gemv_fp8(const uint8_t *q, const float *rs,
                  const uint16_t *x, int N, int64_t M, int64_t K,
                  const int64_t *rows, int64_t nrows,
                  double *y, double *a, int threads)
{
    gemv_job j;
    memset(&j, 0, sizeof j);
    j.fp8 = 1; j.q = q; j.rs = rs; j.x = x; j.N = N; j.M = M; j.K = K;
    j.rows = rows; j.nrows = rows ? nrows : M; j.y = y; j.a = a;
    gemv_run(&j, threads);
}

/* ---------------------------------------------------------------- check */

int64_t vgo_check(const uint16_t *y, const double *yref, const double *a,
                  int64_t n, double rel, double abs_tol, double *worst)
{
    int64_t i, bad = 0;
    double w = 0.0;
    for (i = 0; i < n; ++i) {
        double err = fabs(vgo_bf16_value(y[i]) - yref[i]);
        double tol = rel * a[i] + abs_tol;
        double ratio = err / tol;
        if (!(err <= tol))
            ++bad;
        if (!(ratio <= w))                        /* also catches NaN */
            w = isnan(ratio) ? INFINITY : ratio;
    }
    if (worst)
        *worst = w;
    return bad;
}

/* --------------------------------------------------------- other formats */

double vgo_e8m0_value(int byte)
{
    if (byte == 255)
        return NAN;
    return ldexp(1.0, byte - 127);
}

int vgo_mxfp8_quantise(const float *W, int64_t M, int64_t K, uint8_t *q, uint8_t *sc)
{
    int64_t m, b;
    if (!all_finite(W, M * K))
        return -1;
    for (m = 0; m < M; ++m) {
        for (b = 0; b < K / 32; ++b) {
            const float *w = W + m * K + b * 32;
            float amax = 0.0f, X;
            int e, ex, j;
            for (j = 0; j < 32; ++j)
                if (fabsf(w[j]) > amax)
                    amax = fabsf(w[j]);
            if (amax == 0.0f) {
                e = 127;
            } else {
                frexp((double)amax, &ex);         /* amax in [2^(ex-1), 2^ex) */
                e = (ex - 1) - 8 + 127;           /* floor(log2 amax) - emax(E4M3) */
                if (e < 10)
                    e = 10;
                if (e > 134)
                    e = 134;
            }
            sc[m * (K / 32) + b] = (uint8_t)e;
            X = (float)ldexp(1.0, e - 127);       /* exact */
            for (j = 0; j < 32; ++j)
                q[m * K + b * 32 + j] = (uint8_t)vgo_e4m3_encode(w[j] / X);
        }
    }
    return 0;
}

int vgo_int4g_quantise(const float *W, int64_t M, int64_t K, uint8_t *nib, uint16_t *sc)
{
    int64_t m, b;
    if (!all_finite(W, M * K))
        return -1;
    memset(nib, 0, (size_t)(M * (K / 2)));
    for (m = 0; m < M; ++m) {
        for (b = 0; b < K / 128; ++b) {
            const float *w = W + m * K + b * 128;
            float amax = 0.0f, s;
            uint16_t sbits;
            int j;
            for (j = 0; j < 128; ++j)
                if (fabsf(w[j]) > amax)
                    amax = fabsf(w[j]);
            sbits = vgo_bf16_round((double)(amax / 7.0f));   /* FP32 division, then BF16 */
            sc[m * (K / 128) + b] = sbits;
            s = (float)vgo_bf16_value(sbits);
            for (j = 0; j < 128; ++j) {
                int code = 8;
                if (s != 0.0f) {
                    float r = nearbyintf(w[j] / s);       /* ties to even */
                    if (r < -8.0f)
                        r = -8.0f;
                    if (r > 7.0f)
                        r = 7.0f;
                    code = (int)r + 8;
                }
                {
                    int64_t k = b * 128 + j;
                    uint8_t *p = nib + m * (K / 2) + k / 2;
                    *p = (uint8_t)(*p | ((k & 1) ? code << 4 : code));
                }
            }
        }
    }
    return 0;
}

void vgo_mxfp8_dequant(const uint8_t *q, const uint8_t *sc, int64_t M, int64_t K, double *What)
{
    int64_t m, k;
    for (m = 0; m < M; ++m)
        for (k = 0; k < K; ++k)
            What[m * K + k] = vgo_e4m3_value(q[m * K + k]) * vgo_e8m0_value(sc[m * (K / 32) + k / 32]);
}

void vgo_int4g_dequant(const uint8_t *nib, const uint16_t *sc, int64_t M, int64_t K,
                       double *What)
{
    int64_t m, k;
    for (m = 0; m < M; ++m)
        for (k = 0; k < K; ++k) {
            uint8_t byte = nib[m * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            What[m * K + k] = (double)(code - 8) * vgo_bf16_value(sc[m * (K / 128) + k / 128]);
        }
}

/* ------------------------------------------------------ fused neighbours */

uint16_t vgo_bf16_round(double v)
{
    int ex;
    double a = fabs(v), q, r;
    uint32_t u;
    float f;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v))
        return 0x7FC0;
    if (a == 0.0)
        return sign;
    frexp(a, &ex);                                /* a in [2^(ex-1), 2^ex) */
    if (ex - 1 < -126)
        ex = -125;                                /* subnormal spacing 2^-133 */
    q = ldexp(1.0, ex - 1 - 7);                   /* 7 fraction bits */
    r = nearbyint(a / q) * q;                     /* ties to the even multiple */
    if (r > 3.3895313892515355e38)                /* past the largest finite BF16 */
        return sign | 0x7F80;
    f = (float)r;                                 /* exact: r has <= 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

double vgo_silu(double g)
{
    return g / (1.0 + exp(-g));
}

void vgo_swiglu(const double *g, const double *u, const double *ag, const double *au,
                int64_t n, double *h, double *bound)
{
    int64_t i;
    for (i = 0; i < n; ++i) {
        double s = vgo_silu(g[i]);
        double eg = 4e-3 * ag[i] + 1e-6, eu = 4e-3 * au[i] + 1e-6;
        h[i] = s * u[i];
        bound[i] = 1.1 * eg * (fabs(u[i]) + eu) + fabs(s) * eu + ldexp(fabs(h[i]), -8) + 1e-6;
    }
}

void vgo_rmsnorm(const uint16_t *x, const uint16_t *gamma, int N, int64_t K, double eps,
                 uint16_t *out)
{
    int n;
    int64_t k;
    for (n = 0; n < N; ++n) {
        double ss = 0.0, inv;
        for (k = 0; k < K; ++k) {
            double v = vgo_bf16_value(x[n * K + k]);
            ss += v * v;
        }
        inv = 1.0 / sqrt(ss / (double)K + eps);
        for (k = 0; k < K; ++k)
            out[n * K + k] = vgo_bf16_round(vgo_bf16_value(x[n * K + k]) * inv
                                            * vgo_bf16_value(gamma[k]));
    }
}
