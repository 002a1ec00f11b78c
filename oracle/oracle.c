/*
 * oracle.c -- plain fp64 CPU oracle for RMSNorm (forward, residual-fused
 * forward, backward).  TEST INFRASTRUCTURE: only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load this file.  It shares no
 * code, header, table or helper with the CUDA library and never touches a GPU.
 *
 * What it computes follows "Skill: Write a Triton RMSNorm Kernel" (ahel.ai,
 * write-triton-rmsnorm-kernel):
 *   - Purpose:                 y = x * rsqrt(mean(x^2 over the last axis) + eps) * weight
 *   - Required reasoning 5-8:  mean of squares over the full row length H,
 *                              eps inside the square root, weight indexed by
 *                              column only, apply order (x * rrms) * w
 *   - Kernel design rules:     fused residual: add the two inputs before squaring
 *   - Required reasoning 10:   the saved per-row statistic is rrms (reciprocal)
 *   - Required reasoning 12:   dx = rrms*(dy*w) - (xhat*rrms/H) * sum_h(dy*w*xhat),
 *                              xhat = x*rrms;  dweight = sum over rows of dy*xhat
 *   - Use this when, third bullet (the post-add sum is written back as the
 *     next block's residual stream): its gradient adds to ds in the backward
 *     of the fused forward (orc_rmsnorm_bwd_residual)
 * and the PyTorch one-liner printed on the "Rocm Kernels" page
 * (skillselion.com huggingface/kernels/rocm-kernels, "Compare with PyTorch
 * reference"), which states the same forward.  It also holds that page's
 * AdaLN forward and a residual + LayerNorm forward (see their sections).
 *
 * Everything is evaluated in IEEE binary64, in plain ascending index order,
 * with no blocking or reordering.  Storage formats are decoded to binary64 on
 * entry and results are returned in binary64; rounding back to a storage
 * format is a separate call (orc_encode), written from the IEEE 754 format
 * definitions (binary16, and bfloat16 = the upper 16 bits of binary32).
 *
 * Threads: rows are independent, so row loops are split into contiguous row
 * ranges, one per thread.  Each row is computed exactly as in the
 * single-thread case, so results do not depend on the thread count.  The
 * cross-row dweight sum is split by column ranges; every column is summed
 * over rows in ascending row order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };

#define ORC_MAX_THREADS 256

/* ------------------------------------------------------------------------ */
/* Storage-format codec (IEEE 754-2008 binary16; bfloat16 = binary32's top  */
/* half; binary32 and binary64 as the C types).                             */
/* ------------------------------------------------------------------------ */

static double decode_f16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 10) & 0x1f;
    int m = b & 0x3ff;
    double v;
    if (e == 0)              /* zero or subnormal: m * 2^-24 */
        v = ldexp((double)m, -24);
    else if (e == 31)        /* infinity or NaN */
        v = (m == 0) ? INFINITY : NAN;
    else                     /* normal: (1024 + m) * 2^(e - 15 - 10) */
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

static double decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)              /* zero or subnormal: m * 2^-133 */
        v = ldexp((double)m, -133);
    else if (e == 255)
        v = (m == 0) ? INFINITY : NAN;
    else                     /* normal: (128 + m) * 2^(e - 127 - 7) */
        v = ldexp((double)(128 + m), e - 134);
    return sign ? -v : v;
}

/*
 * Round |v| to a binary format with `p` significand bits (including the
 * implicit one), minimum normal exponent `emin`, maximum exponent `emax`,
 * round-to-nearest, ties to even.  Returns the encoded magnitude bits
 * (exponent field << (p-1) | fraction) or -1 for overflow to infinity.
 * Scaling by powers of two is exact in binary64 for every value used here,
 * so the only rounding step is rint() in the default (nearest-even) mode.
 */
static long round_to_format(double a, int p, int emin, int emax, int bias)
{
    if (a == 0.0)
        return 0;
    int e2;
    frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;          /* a in [2^e, 2^(e+1)) */
    if (e < emin) {
        /* subnormal range: integer multiple of 2^(emin - p + 1) */
        double q = rint(ldexp(a, -(emin - p + 1)));
        /* q may reach 2^(p-1): that is the smallest normal, whose encoding
           (exponent field 1, fraction 0) equals q as an integer. */
        return (long)q;
    }
    double q = rint(ldexp(a, (p - 1) - e));    /* in [2^(p-1), 2^p] */
    if (q == ldexp(1.0, p)) {                  /* rounded up to the next binade */
        q = ldexp(1.0, p - 1);
        e += 1;
    }
    if (e > emax)
        return -1;
    return ((long)(e + bias) << (p - 1)) | ((long)q - (1L << (p - 1)));
}

static uint16_t encode_f16(double v)
{
    if (isnan(v))
        return 0x7e00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    long mag = round_to_format(fabs(v), 11, -14, 15, 15);
    if (mag < 0 || isinf(v))
        return sign | 0x7c00;
    return sign | (uint16_t)mag;
}

static uint16_t encode_bf16(double v)
{
    if (isnan(v))
        return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    long mag = round_to_format(fabs(v), 8, -126, 127, 127);
    if (mag < 0 || isinf(v))
        return sign | 0x7f80;
    return sign | (uint16_t)mag;
}

static size_t elem_size(int dtype)
{
    switch (dtype) {
    case ORC_F32: return 4;
    case ORC_F16: return 2;
    case ORC_BF16: return 2;
    case ORC_F64: return 8;
    default: return 0;
    }
}

/* element k of a storage array, as binary64 */
static double load_elem(int dtype, const void *base, int64_t k)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)base)[k];
    case ORC_F16: return decode_f16(((const uint16_t *)base)[k]);
    case ORC_BF16: return decode_bf16(((const uint16_t *)base)[k]);
    default: return ((const double *)base)[k];
    }
}

int orc_decode(int dtype, const void *src, double *dst, int64_t n)
{
    if (!elem_size(dtype))
        return 1;
    for (int64_t k = 0; k < n; ++k)
        dst[k] = load_elem(dtype, src, k);
    return 0;
}

/* binary64 -> storage format, each value rounded once (nearest, ties even) */
int orc_encode(int dtype, const double *src, void *dst, int64_t n)
{
    for (int64_t k = 0; k < n; ++k) {
        switch (dtype) {
        case ORC_F32: ((float *)dst)[k] = (float)src[k]; break;
        case ORC_F16: ((uint16_t *)dst)[k] = encode_f16(src[k]); break;
        case ORC_BF16: ((uint16_t *)dst)[k] = encode_bf16(src[k]); break;
        case ORC_F64: ((double *)dst)[k] = src[k]; break;
        default: return 1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver                                                      */
/* ------------------------------------------------------------------------ */

typedef void (*range_fn)(void *ctx, int64_t begin, int64_t end);

struct range_job {
    range_fn fn;
    void *ctx;
    int64_t begin, end;
};

static void *range_thread(void *p)
{
    struct range_job *j = (struct range_job *)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

/* run fn over [0, n) split into at most nthreads contiguous ranges */
static void parallel_ranges(range_fn fn, void *ctx, int64_t n, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > ORC_MAX_THREADS)
        nthreads = ORC_MAX_THREADS;
    if ((int64_t)nthreads > n)
        nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t tid[ORC_MAX_THREADS];
    struct range_job job[ORC_MAX_THREADS];
    int started[ORC_MAX_THREADS];
    for (int t = 0; t < nthreads; ++t) {
        job[t].fn = fn;
        job[t].ctx = ctx;
        job[t].begin = n * t / nthreads;
        job[t].end = n * (t + 1) / nthreads;
        started[t] = pthread_create(&tid[t], NULL, range_thread, &job[t]) == 0;
        if (!started[t])
            fn(ctx, job[t].begin, job[t].end);   /* no thread: run it here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (started[t])
            pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* Forward                                                                  */
/* ------------------------------------------------------------------------ */

struct fwd_ctx {
    int dtype;
    const void *x, *r, *w;
    int64_t H, stride;
    double eps;
    double *y, *s_out, *rrms;
};

static void fwd_rows(void *p, int64_t i0, int64_t i1)
{
    const struct fwd_ctx *c = (const struct fwd_ctx *)p;
    const int64_t H = c->H;
    double *s = (double *)malloc((size_t)H * sizeof(double));
    if (!s)
        abort();
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t row = i * c->stride;
        /* input row; fused residual: s = x + r, added before squaring */
        for (int64_t h = 0; h < H; ++h) {
            s[h] = load_elem(c->dtype, c->x, row + h);
            if (c->r)
                s[h] += load_elem(c->dtype, c->r, row + h);
        }
        /* mean of squares over the full row length H */
        double ss = 0.0;
        for (int64_t h = 0; h < H; ++h)
            ss += s[h] * s[h];
        const double ms = ss / (double)H;
        /* reciprocal RMS, eps inside the square root */
        const double rrms = 1.0 / sqrt(ms + c->eps);
        if (c->rrms)
            c->rrms[i] = rrms;
        /* y = (s * rrms) * w, weight indexed by column only */
        for (int64_t h = 0; h < H; ++h) {
            double w = c->w ? load_elem(c->dtype, c->w, h) : 1.0;
            c->y[i * H + h] = (s[h] * rrms) * w;
            if (c->s_out)
                c->s_out[i * H + h] = s[h];
        }
    }
    free(s);
}

/*
 * x, r (nullable: no residual), w (nullable: no weight) are storage arrays;
 * element (i, h) of x and r sits at index i*stride + h, element h of w at h.
 * eps is the binary64 value of the binary32 eps the library receives.
 * Outputs are dense M x H binary64 (y, s_out) and M binary64 (rrms);
 * s_out and rrms are nullable.
 */
int orc_rmsnorm_fwd(int dtype, const void *x, const void *r, const void *w,
                    int64_t M, int64_t H, int64_t stride, double eps,
                    double *y, double *s_out, double *rrms, int nthreads)
{
    if (!elem_size(dtype) || !x || !y || M < 0 || H <= 0 || stride < H)
        return 1;
    struct fwd_ctx c = {dtype, x, r, w, H, stride, eps, y, s_out, rrms};
    parallel_ranges(fwd_rows, &c, M, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* AdaLN forward ("Rocm Kernels" page, section 4. AdaLN / Template 4):      */
/*   out = norm(x) * weight * (1 + scale) + shift                           */
/* evaluated left to right on norm(x) = x * rrms; scale and shift are       */
/* conditioning rows: token row i uses conditioning row i / rows_per_cond   */
/* (1 = per token, [B, S, H]; S = one row per sequence, [B, 1, H]).         */
/* ------------------------------------------------------------------------ */

struct adaln_ctx {
    int dtype;
    const void *x, *w, *scale, *shift;
    int64_t H, stride, cond_stride, rows_per_cond;
    double eps;
    double *y, *y_scale, *rrms;
};

static void adaln_rows(void *p, int64_t i0, int64_t i1)
{
    const struct adaln_ctx *c = (const struct adaln_ctx *)p;
    const int64_t H = c->H;
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t row = i * c->stride;
        const int64_t crow = (i / c->rows_per_cond) * c->cond_stride;
        double ss = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            const double v = load_elem(c->dtype, c->x, row + h);
            ss += v * v;
        }
        const double rrms = 1.0 / sqrt(ss / (double)H + c->eps);
        if (c->rrms)
            c->rrms[i] = rrms;
        for (int64_t h = 0; h < H; ++h) {
            const double w = c->w ? load_elem(c->dtype, c->w, h) : 1.0;
            const double sc = load_elem(c->dtype, c->scale, crow + h);
            const double sh = load_elem(c->dtype, c->shift, crow + h);
            const double t = ((load_elem(c->dtype, c->x, row + h) * rrms) * w) * (1.0 + sc);
            c->y[i * H + h] = t + sh;
            /* size of the two terms whose sum is y (bounds any rounding order) */
            if (c->y_scale)
                c->y_scale[i * H + h] = fabs(t) + fabs(sh);
        }
    }
}

/*
 * x: M x H at `stride`; scale, shift: conditioning rows at `cond_stride`;
 * w nullable (no weight).  Outputs y (dense M x H), y_scale (nullable),
 * rrms (nullable).
 */
int orc_rmsnorm_adaln_fwd(int dtype, const void *x, const void *w, const void *scale, const void *shift,
                          int64_t M, int64_t H, int64_t stride, int64_t cond_stride, int64_t rows_per_cond,
                          double eps, double *y, double *y_scale, double *rrms, int nthreads)
{
    if (!elem_size(dtype) || !x || !scale || !shift || !y || M < 0 || H <= 0 || stride < H ||
        cond_stride < H || rows_per_cond < 1)
        return 1;
    struct adaln_ctx c = {dtype, x, w, scale, shift, H, stride, cond_stride, rows_per_cond, eps, y, y_scale,
                          rrms};
    parallel_ranges(adaln_rows, &c, M, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Residual + LayerNorm forward (the devpost "SpeedROCm" page, How the      */
/* solution addresses the problem, item 4: each residual add fused with the */
/* LayerNorm that consumes it; the model's reference LayerNorm is PyTorch's,*/
/* Development tools).  The pages print no formula; this is the textbook    */
/* definition with the mean subtraction the RMSNorm skill page says         */
/* LayerNorm has (Do not use this when, second bullet):                     */
/*   s = x (+ r);  mean = sum(s) / H;  var = sum((s - mean)^2) / H          */
/*   rstd = 1 / sqrt(var + eps);  y = (s - mean) * rstd * w + b             */
/* (biased variance, eps inside the square root, per-column weight and      */
/* bias), both sums in one pass each over the row, ascending.               */
/* ------------------------------------------------------------------------ */

struct ln_ctx {
    int dtype;
    const void *x, *r, *w, *b;
    int64_t H, stride;
    double eps;
    double *y, *y_scale, *s_out, *mean, *rstd;
};

static void ln_rows(void *p, int64_t i0, int64_t i1)
{
    const struct ln_ctx *c = (const struct ln_ctx *)p;
    const int64_t H = c->H;
    double *s = (double *)malloc((size_t)H * sizeof(double));
    if (!s)
        abort();
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t row = i * c->stride;
        for (int64_t h = 0; h < H; ++h) {
            s[h] = load_elem(c->dtype, c->x, row + h);
            if (c->r)
                s[h] += load_elem(c->dtype, c->r, row + h);
        }
        double sum = 0.0, abs_sum = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            sum += s[h];
            abs_sum += fabs(s[h]);
        }
        const double mean = sum / (double)H;
        const double mean_abs = abs_sum / (double)H;   /* condition scale of the mean */
        double sq = 0.0;
        for (int64_t h = 0; h < H; ++h)
            sq += (s[h] - mean) * (s[h] - mean);
        const double rstd = 1.0 / sqrt(sq / (double)H + c->eps);
        if (c->mean)
            c->mean[i] = mean;
        if (c->rstd)
            c->rstd[i] = rstd;
        for (int64_t h = 0; h < H; ++h) {
            const double w = c->w ? load_elem(c->dtype, c->w, h) : 1.0;
            const double b = c->b ? load_elem(c->dtype, c->b, h) : 0.0;
            c->y[i * H + h] = ((s[h] - mean) * rstd) * w + b;
            /* size of the terms whose differences and sum make y: s_h, the
             * mean (whose rounding error in any evaluation scales with the
             * mean of |s|) and the bias */
            if (c->y_scale)
                c->y_scale[i * H + h] = (fabs(s[h]) + mean_abs) * rstd * fabs(w) + fabs(b);
            if (c->s_out)
                c->s_out[i * H + h] = s[h];
        }
    }
    free(s);
}

/*
 * x, r (nullable), w (nullable: no weight), b (nullable: no bias) are storage
 * arrays with the layout of orc_rmsnorm_fwd.  Outputs: y, y_scale, s_out
 * (dense M x H), mean and rstd (M); all but y nullable.
 */
int orc_layernorm_fwd(int dtype, const void *x, const void *r, const void *w, const void *b,
                      int64_t M, int64_t H, int64_t stride, double eps, double *y, double *y_scale,
                      double *s_out, double *mean, double *rstd, int nthreads)
{
    if (!elem_size(dtype) || !x || !y || M < 0 || H <= 0 || stride < H)
        return 1;
    struct ln_ctx c = {dtype, x, r, w, b, H, stride, eps, y, y_scale, s_out, mean, rstd};
    parallel_ranges(ln_rows, &c, M, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward                                                                 */
/* ------------------------------------------------------------------------ */

struct bwd_ctx {
    int dtype;
    const void *dy, *dres, *x, *w;
    int64_t M, H, stride;
    double eps;
    double *dx, *dx_scale, *dweight, *dweight_abs, *rrms;
};

/* rrms per row, recomputed in binary64 from the stored input row */
static void bwd_rrms_rows(void *p, int64_t i0, int64_t i1)
{
    const struct bwd_ctx *c = (const struct bwd_ctx *)p;
    for (int64_t i = i0; i < i1; ++i) {
        double ss = 0.0;
        for (int64_t h = 0; h < c->H; ++h) {
            double v = load_elem(c->dtype, c->x, i * c->stride + h);
            ss += v * v;
        }
        c->rrms[i] = 1.0 / sqrt(ss / (double)c->H + c->eps);
    }
}

/* dx_h = rrms*g_h - xhat_h*(rrms/H)*sum_k g_k*xhat_k, g = dy*w, xhat = x*rrms.
   dx_scale_h = |rrms*g_h| + |xhat_h*(rrms/H)| * sum_k |g_k*xhat_k| is the size
   of the two terms whose difference is dx_h: the rounding error of any
   binary32 evaluation of dx_h is a small multiple of u * dx_scale_h, even
   where the difference cancels (H = 1, or x parallel to g). */
static void bwd_dx_rows(void *p, int64_t i0, int64_t i1)
{
    const struct bwd_ctx *c = (const struct bwd_ctx *)p;
    const int64_t H = c->H;
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t row = i * c->stride;
        const double rrms = c->rrms[i];
        double dot = 0.0, dot_abs = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double w = c->w ? load_elem(c->dtype, c->w, h) : 1.0;
            double g = load_elem(c->dtype, c->dy, row + h) * w;
            double xhat = load_elem(c->dtype, c->x, row + h) * rrms;
            dot += g * xhat;
            dot_abs += fabs(g * xhat);
        }
        for (int64_t h = 0; h < H; ++h) {
            double w = c->w ? load_elem(c->dtype, c->w, h) : 1.0;
            double g = load_elem(c->dtype, c->dy, row + h) * w;
            double xhat = load_elem(c->dtype, c->x, row + h) * rrms;
            c->dx[i * H + h] = rrms * g - xhat * (rrms / (double)H) * dot;
            if (c->dx_scale)
                c->dx_scale[i * H + h] = fabs(rrms * g) + fabs(xhat * (rrms / (double)H)) * dot_abs;
            if (c->dres) {   /* gradient arriving through residual_out adds to ds */
                const double d = load_elem(c->dtype, c->dres, row + h);
                c->dx[i * H + h] += d;
                if (c->dx_scale)
                    c->dx_scale[i * H + h] += fabs(d);
            }
        }
    }
}

/* dweight_h = sum over rows i (ascending) of dy_ih * xhat_ih; also the sum of
   absolute terms, which bounds the rounding error of any summation order.
   A thread owns a column range and walks the rows in ascending order, so
   every column is summed in ascending row order. */
static void bwd_dweight_cols(void *p, int64_t h0, int64_t h1)
{
    const struct bwd_ctx *c = (const struct bwd_ctx *)p;
    const int64_t n = h1 - h0;
    double *acc = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    double *acc_abs = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    if (!acc || !acc_abs)
        abort();
    for (int64_t i = 0; i < c->M; ++i) {
        const int64_t row = i * c->stride;
        for (int64_t h = h0; h < h1; ++h) {
            double t = load_elem(c->dtype, c->dy, row + h) *
                       (load_elem(c->dtype, c->x, row + h) * c->rrms[i]);
            acc[h - h0] += t;
            acc_abs[h - h0] += fabs(t);
        }
    }
    for (int64_t h = h0; h < h1; ++h) {
        if (c->dweight)
            c->dweight[h] = acc[h - h0];
        if (c->dweight_abs)
            c->dweight_abs[h] = acc_abs[h - h0];
    }
    free(acc);
    free(acc_abs);
}

/*
 * dy, x storage arrays with row stride `stride`; w nullable (no weight: g = dy).
 * Outputs (all nullable): dx and dx_scale dense M x H binary64 (dx_scale is
 * only written together with dx), dweight and dweight_abs H binary64, rrms M
 * binary64 (recomputed from x; scratch is allocated here if the caller passes
 * NULL).
 */
static int bwd_common(int dtype, const void *dy, const void *dres, const void *x, const void *w,
                      int64_t M, int64_t H, int64_t stride, double eps,
                      double *dx, double *dx_scale, double *dweight, double *dweight_abs,
                      double *rrms, int nthreads);

int orc_rmsnorm_bwd(int dtype, const void *dy, const void *x, const void *w,
                    int64_t M, int64_t H, int64_t stride, double eps,
                    double *dx, double *dx_scale, double *dweight, double *dweight_abs,
                    double *rrms, int nthreads)
{
    return bwd_common(dtype, dy, NULL, x, w, M, H, stride, eps, dx, dx_scale, dweight, dweight_abs, rrms,
                      nthreads);
}

/*
 * Backward of the residual-fused forward (s = x + residual feeds both the
 * norm and residual_out): ds = (the norm's dx for dy) + dres, where dres is
 * the gradient arriving through residual_out; ds is the gradient of x and
 * of residual alike.  x here is the stored residual_out; dweight as for
 * orc_rmsnorm_bwd (dres does not reach the weight).
 */
int orc_rmsnorm_bwd_residual(int dtype, const void *dy, const void *dres, const void *x, const void *w,
                             int64_t M, int64_t H, int64_t stride, double eps,
                             double *dx, double *dx_scale, double *dweight, double *dweight_abs,
                             double *rrms, int nthreads)
{
    if (!dres)
        return 1;
    return bwd_common(dtype, dy, dres, x, w, M, H, stride, eps, dx, dx_scale, dweight, dweight_abs, rrms,
                      nthreads);
}

static int bwd_common(int dtype, const void *dy, const void *dres, const void *x, const void *w,
                      int64_t M, int64_t H, int64_t stride, double eps,
                      double *dx, double *dx_scale, double *dweight, double *dweight_abs,
                      double *rrms, int nthreads)
{
    if (!elem_size(dtype) || !dy || !x || M < 0 || H <= 0 || stride < H)
        return 1;
    double *rr = rrms;
    if (!rr) {
        rr = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
        if (!rr)
            return 2;
    }
    struct bwd_ctx c = {dtype, dy, dres, x, w, M, H, stride, eps, dx, dx_scale, dweight, dweight_abs, rr};
    parallel_ranges(bwd_rrms_rows, &c, M, nthreads);
    if (dx)
        parallel_ranges(bwd_dx_rows, &c, M, nthreads);
    if (dweight || dweight_abs)
        parallel_ranges(bwd_dweight_cols, &c, H, nthreads);
    if (!rrms)
        free(rr);
    return 0;
}
