/*
 * dg_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of DiffusionGemma's canvas-forward attention
 * block, written from the page "inferencelayer 0.2.3, src/diffusion_gemma_gpu.rs" (docs.rs).
 * It exists to check the CUDA library against; nothing in the product links or calls it.
 * Only the tests, the smoke check and the bench's CPU-baseline leg may use it.
 *
 * It shares no code with the CUDA path: no headers, helpers, tables or constants.
 * Every step follows its definition directly, in the page's order, with fp64 arithmetic on
 * the fp32 inputs:
 *
 *   1. per-(token, head) RMSNorm with an optional weight
 *      (item DG_HEADNORM_ROPE: x * (mean x^2 + eps)^-1/2, then * w when "weighted");
 *   2. NeoX rotate-half RoPE at position pos0 + t (same item: v*cos + rot*sin with
 *      rot = -x[i + hd/2] for i < hd/2 and x[i - hd/2] otherwise); the per-token cos|sin row is
 *      either given, or built from the standard NeoX frequencies theta^(-2i/hd) with both halves
 *      equal (the table builder rope_cos_sin is imported, not shown, on the page);
 *   3. the weightless, un-roped V norm (canvas_forward, third head-norm dispatch: flags 0);
 *   4. GQA bidirectional softmax attention with scaling 1.0 over the split key set
 *      [cache (ctx rows, layout [nkv, ctx, hd], used as given) | canvas (T rows, [T, nkv*hd])],
 *      kv head = q head / (nh / nkv) (item DG_ATTN).
 *
 * The attention is the plain definition: scores for every key, the maximum subtracted, the
 * exponentials, their sum, the weighted sum of values, one division. No tiling, no online
 * rescaling, no reordering beyond the natural loops.
 *
 * OpenMP (when compiled with -fopenmp) splits the (canvas row, head) loop of step 4 across
 * threads; each output element is still computed by one thread in the same order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Step 1 (DG_HEADNORM_ROPE, first half): y = x * (mean(x^2) + eps)^-1/2, times w[i] if w. */
static void rms_head(const float *x, int hd, const float *w, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < hd; ++i) ss += (double)x[i] * (double)x[i];
    double r = 1.0 / sqrt(ss / (double)hd + eps);
    for (int i = 0; i < hd; ++i) {
        double v = (double)x[i] * r;
        if (w) v *= (double)w[i];
        y[i] = v;
    }
}

/* Step 2 (DG_HEADNORM_ROPE, second half): rotate-half with per-element cos c[i], sin s[i]. */
static void rope_head(const double *y, int hd, const double *c, const double *s, double *z)
{
    int half = hd / 2;
    for (int i = 0; i < hd; ++i) {
        double rot = (i < half) ? -y[i + half] : y[i - half];
        z[i] = y[i] * c[i] + rot * s[i];
    }
}

/* The cos|sin row for one token.  With a table: the row's two halves verbatim.  Without: the
 * standard NeoX frequencies, angle_i = p * theta^(-2 (i mod hd/2) / hd), computed in fp64. */
static void cos_sin_row(int hd, long long p, double theta, const float *table_row, double *c,
                        double *s)
{
    int half = hd / 2;
    for (int i = 0; i < hd; ++i) {
        if (table_row) {
            c[i] = (double)table_row[i];
            s[i] = (double)table_row[hd + i];
        } else {
            int k = i % half;
            double inv_freq = pow(theta, -2.0 * (double)k / (double)hd);
            double ang = (double)p * inv_freq;
            c[i] = cos(ang);
            s[i] = sin(ang);
        }
    }
}

/* Steps 1+2 over a [rows, heads*hd] block: out[(r*heads + h)*hd + i] (fp64).
 * rope != 0 applies RoPE at position pos0 + r (or the table row r). */
void dgo_norm_rope(const float *x, int rows, int heads, int hd, const float *w, double eps,
                   int rope, long long pos0, double theta, const float *cos_sin, double *out)
{
    double *y = (double *)malloc(sizeof(double) * hd);
    double *c = (double *)malloc(sizeof(double) * hd);
    double *s = (double *)malloc(sizeof(double) * hd);
    for (int r = 0; r < rows; ++r) {
        if (rope) cos_sin_row(hd, pos0 + r, theta, cos_sin ? cos_sin + (size_t)r * 2 * hd : NULL, c, s);
        for (int h = 0; h < heads; ++h) {
            const float *xr = x + ((size_t)r * heads + h) * hd;
            double *o = out + ((size_t)r * heads + h) * hd;
            rms_head(xr, hd, w, eps, y);
            if (rope) rope_head(y, hd, c, s, o);
            else memcpy(o, y, sizeof(double) * hd);
        }
    }
    free(y); free(c); free(s);
}

/* Step 4 (DG_ATTN): for canvas rows [row_begin, row_end) and every q head h, with
 * g = h / (nh/nkv):  keys j < ctx come from k_cache[g, j, :] (as given), keys ctx + t from the
 * normed canvas khat[t, g, :]; s_j = q . K_j (scaling 1.0, no mask);
 * out = sum_j exp(s_j - max s) V_j / sum_j exp(s_j - max s).
 * qhat [T, nh, hd], khat/vhat [T, nkv, hd] (fp64); k_cache/v_cache [nkv, ctx, hd] (fp32);
 * out [T, nh, hd] (fp64; only the requested rows are written). */
void dgo_attention(const double *qhat, const double *khat, const double *vhat,
                   const float *k_cache, const float *v_cache, int T, int ctx, int nh, int nkv,
                   int hd, int row_begin, int row_end, double *out)
{
    int G = nh / nkv;
    int S = ctx + T;
    long long units = (long long)(row_end - row_begin) * nh;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)S);
        double *acc = (double *)malloc(sizeof(double) * (size_t)hd);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (long long u = 0; u < units; ++u) {
            int t = row_begin + (int)(u / nh);
            int h = (int)(u % nh);
            int g = h / G;
            const double *q = qhat + ((size_t)t * nh + h) * hd;
            double mx = -INFINITY;
            for (int j = 0; j < S; ++j) {
                double d = 0.0;
                if (j < ctx) {
                    const float *k = k_cache + ((size_t)g * ctx + j) * hd;
                    for (int i = 0; i < hd; ++i) d += q[i] * (double)k[i];
                } else {
                    const double *k = khat + ((size_t)(j - ctx) * nkv + g) * hd;
                    for (int i = 0; i < hd; ++i) d += q[i] * k[i];
                }
                sc[j] = d;
                if (d > mx) mx = d;
            }
            double den = 0.0;
            for (int j = 0; j < S; ++j) { sc[j] = exp(sc[j] - mx); den += sc[j]; }
            for (int i = 0; i < hd; ++i) acc[i] = 0.0;
            for (int j = 0; j < S; ++j) {
                double p = sc[j];
                if (j < ctx) {
                    const float *v = v_cache + ((size_t)g * ctx + j) * hd;
                    for (int i = 0; i < hd; ++i) acc[i] += p * (double)v[i];
                } else {
                    const double *v = vhat + ((size_t)(j - ctx) * nkv + g) * hd;
                    for (int i = 0; i < hd; ++i) acc[i] += p * v[i];
                }
            }
            double *o = out + ((size_t)t * nh + h) * hd;
            for (int i = 0; i < hd; ++i) o[i] = acc[i] / den;
        }
        free(sc); free(acc);
    }
}

/* The whole block: q/k norm + rope (weights optional), v norm, attention.  pos0 is the
 * position of canvas row 0 (the cache length by default).  Returns 0, or -1 on bad sizes. */
int dgo_forward(int nh, int nkv, int hd, int ctx, int T, double eps, double theta, long long pos0,
                const float *q, const float *k_canvas, const float *v_canvas,
                const float *k_cache, const float *v_cache, const float *q_norm_w,
                const float *k_norm_w, const float *cos_sin, int row_begin, int row_end,
                double *out)
{
    if (nh <= 0 || nkv <= 0 || nh % nkv || hd <= 0 || hd % 2 || ctx < 0 || T <= 0) return -1;
    if (row_begin < 0 || row_end > T || row_begin > row_end) return -1;
    double *qh = (double *)malloc(sizeof(double) * (size_t)T * nh * hd);
    double *kh = (double *)malloc(sizeof(double) * (size_t)T * nkv * hd);
    double *vh = (double *)malloc(sizeof(double) * (size_t)T * nkv * hd);
    if (!qh || !kh || !vh) { free(qh); free(kh); free(vh); return -1; }
    /* Only the requested query rows need normalising; keys and values need all T rows. */
    int nrows = row_end - row_begin;
    if (nrows > 0)
        dgo_norm_rope(q + (size_t)row_begin * nh * hd, nrows, nh, hd, q_norm_w, eps, 1,
                      pos0 + row_begin, theta,
                      cos_sin ? cos_sin + (size_t)row_begin * 2 * hd : NULL,
                      qh + (size_t)row_begin * nh * hd);
    dgo_norm_rope(k_canvas, T, nkv, hd, k_norm_w, eps, 1, pos0, theta, cos_sin, kh);
    dgo_norm_rope(v_canvas, T, nkv, hd, NULL, eps, 0, 0, theta, NULL, vh);
    dgo_attention(qh, kh, vh, k_cache, v_cache, T, ctx, nh, nkv, hd, row_begin, row_end, out);
    free(qh); free(kh); free(vh);
    return 0;
}

/* The step before the block (canvas_forward, attention branch): the input RMSNorm of the
 * residual stream, `rms!(&cur, &l.ln_in, 1, &nb)` (item DG_RMSNORM: x * (mean x^2 + eps)^-1/2,
 * times w[i] when weighted), then the q / k / v projections, `gemm!` on GLin weights, which
 * compute y = x W^T with W stored [n, k] (the page's "y = x.W^T", bias zero).
 * x [rows, h] fp32, w [h] or NULL; xhat [rows, h] fp64. */
void dgo_rmsnorm_rows(const float *x, int rows, int h, const float *w, double eps, double *xhat)
{
    for (int r = 0; r < rows; ++r) {
        const float *xr = x + (size_t)r * h;
        double ss = 0.0;
        for (int i = 0; i < h; ++i) ss += (double)xr[i] * (double)xr[i];
        double inv = 1.0 / sqrt(ss / (double)h + eps);
        for (int i = 0; i < h; ++i) {
            double v = (double)xr[i] * inv;
            if (w) v *= (double)w[i];
            xhat[(size_t)r * h + i] = v;
        }
    }
}

/* y[r, j] = sum_i xhat[r, i] * W[j, i] for W [n, k] fp32 (GLin layout before its upload
 * transpose); fp64 accumulation in index order. */
void dgo_linear(const double *xhat, int rows, int k, const float *W, int n, double *y)
{
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (long long u = 0; u < (long long)rows * n; ++u) {
        int r = (int)(u / n), j = (int)(u % n);
        const double *xr = xhat + (size_t)r * k;
        const float *wr = W + (size_t)j * k;
        double acc = 0.0;
        for (int i = 0; i < k; ++i) acc += xr[i] * (double)wr[i];
        y[u] = acc;
    }
}

/* The step after the block (canvas_forward, attention branch): `gemm!(&sb, &l.o, t_len, &nb)`
 * (o_proj, y = attn W_o^T with W_o [h, nh*hd]), `rms!(&nb, &l.ln_post_attn, 1, &sb)` (weighted
 * RMSNorm of the projection, item DG_RMSNORM) and `add_scale!(&cur, &sb, 1.0)` (item DG_ADD_SCALE:
 * cur = (cur + sb) * 1.0).  attn [rows, k] fp32, Wo [h, k], w [h] or NULL, resid [rows, h] fp32;
 * out [rows, h] fp64 = the updated residual stream. */
void dgo_oproj_residual(const float *attn, int rows, int k, const float *Wo, int h,
                        const float *w, double eps, double scale, const float *resid, double *out)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)rows * k);
    double *y = (double *)malloc(sizeof(double) * (size_t)rows * h);
    for (size_t i = 0; i < (size_t)rows * k; ++i) a[i] = (double)attn[i];
    dgo_linear(a, rows, k, Wo, h, y);
    for (int r = 0; r < rows; ++r) {
        const double *yr = y + (size_t)r * h;
        double ss = 0.0;
        for (int i = 0; i < h; ++i) ss += yr[i] * yr[i];
        double inv = 1.0 / sqrt(ss / (double)h + eps);
        for (int i = 0; i < h; ++i) {
            double v = yr[i] * inv;
            if (w) v *= (double)w[i];
            out[(size_t)r * h + i] = ((double)resid[(size_t)r * h + i] + v) * scale;
        }
    }
    free(a);
    free(y);
}

/* Thread control for the timed CPU baseline (1 when built without OpenMP). */
int dgo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
