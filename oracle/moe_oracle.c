/*
 * moe_oracle.c -- the CPU oracle of the sparse MoE FFN sublayer (see
 * moe_oracle.h for the equations and the passages they follow).
 *
 * TEST INFRASTRUCTURE ONLY: the product library never calls it.  Written for
 * clarity: plain loops, double accumulation, no blocking or fusion.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- reading stored values ------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load(const void *p, int dtype, size_t i)
{
    if (dtype == ORC_BF16)
        return bf16_to_double(((const uint16_t *)p)[i]);
    return (double)((const float *)p)[i];
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
static double silu(double z) { return z * sigmoid(z); }

/* y[r] = sum_i W[r][i] * x[i] for a [rows][cols] block starting at element
 * `base` of W. */
static void matvec(const void *W, int dtype, size_t base, int rows, int cols,
                   const double *x, double *y)
{
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        size_t row = base + (size_t)r * (size_t)cols;
        for (int i = 0; i < cols; ++i)
            acc += load(W, dtype, row + (size_t)i) * x[i];
        y[r] = acc;
    }
}

/* ---- configuration -------------------------------------------------------- */

int orc_check_config(const orc_config *c)
{
    if (!c) return -1;
    if (c->hidden < 1 || c->n_expert < 1 || c->expert_ff < 1) return -1;
    if (c->top_k < 1 || c->top_k > c->n_expert) return -1;
    if (c->shared_ff < 0) return -1;
    if (c->router_mode != ORC_ROUTER_SOFTMAX_TOPK && c->router_mode != ORC_ROUTER_TOPK_SOFTMAX) return -1;
    if (c->act != ORC_ACT_SWIGLU && c->act != ORC_ACT_CLAMP_GLU) return -1;
    if (c->w_dtype != ORC_F32 && c->w_dtype != ORC_BF16) return -1;
    if (c->x_dtype != ORC_F32 && c->x_dtype != ORC_BF16) return -1;
    return 0;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- step 1: router ------------------------------------------------------- */

static void router_row(const orc_config *c, const orc_weights *w, const double *xr,
                       double *logits_row, double *sh_logit)
{
    const int H = c->hidden, E = c->n_expert;
    matvec(w->router_w, c->w_dtype, 0, E, H, xr, logits_row);
    if (c->has_bias)
        for (int e = 0; e < E; ++e)
            logits_row[e] += load(w->router_b, c->w_dtype, (size_t)e);
    if (sh_logit && c->shared_ff > 0) {
        double s = 0.0;
        for (int i = 0; i < H; ++i)
            s += load(w->sh_gate_inp, c->w_dtype, (size_t)i) * xr[i];
        *sh_logit = s;
    }
}

static void load_row(const orc_config *c, const void *x, int t, double *xr)
{
    for (int i = 0; i < c->hidden; ++i)
        xr[i] = load(x, c->x_dtype, (size_t)t * (size_t)c->hidden + (size_t)i);
}

int orc_router_logits(const orc_config *c, const orc_weights *w, const void *x,
                      int n_tokens, double *logits, double *sh_logit)
{
    if (orc_check_config(c) || !w || !x || !logits || n_tokens < 0) return -1;
    double *xr = (double *)malloc(sizeof(double) * (size_t)c->hidden);
    if (!xr) return -3;
    for (int t = 0; t < n_tokens; ++t) {
        load_row(c, x, t, xr);
        router_row(c, w, xr, logits + (size_t)t * c->n_expert, sh_logit ? sh_logit + t : NULL);
    }
    free(xr);
    return 0;
}

/* ---- step 2: selection ---------------------------------------------------- */

/* The k largest entries of v[n] in descending order; among equal values the
 * lower index comes first (a strict '>' scan from index 0). */
static void top_k_desc(const double *v, int n, int k, int *idx)
{
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < n; ++e) {
            int taken = 0;
            for (int q = 0; q < j; ++q)
                if (idx[q] == e) { taken = 1; break; }
            if (taken) continue;
            if (best < 0 || v[e] > v[best]) best = e;
        }
        idx[j] = best;
    }
}

int orc_weights_for_selection(const orc_config *c, const double *l,
                              const int *idx, double *wt)
{
    const int E = c->n_expert, k = c->top_k;
    if (c->router_mode == ORC_ROUTER_SOFTMAX_TOPK) {
        /* softmax over all E experts, then keep the selected probabilities */
        double m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - m);
        double sel = 0.0;
        for (int j = 0; j < k; ++j) {
            wt[j] = exp(l[idx[j]] - m) / z;
            sel += wt[j];
        }
        if (c->norm_topk_prob)
            for (int j = 0; j < k; ++j) wt[j] /= sel;
        for (int j = 0; j < k; ++j) wt[j] *= c->weights_scale;
    } else {
        /* softmax over the k selected logits only */
        double m = l[idx[0]];
        for (int j = 1; j < k; ++j) if (l[idx[j]] > m) m = l[idx[j]];
        double z = 0.0;
        for (int j = 0; j < k; ++j) z += exp(l[idx[j]] - m);
        for (int j = 0; j < k; ++j) wt[j] = exp(l[idx[j]] - m) / z;
    }
    return 0;
}

int orc_select(const orc_config *c, const double *l, int *idx, double *wt)
{
    const int E = c->n_expert, k = c->top_k;
    if (c->router_mode == ORC_ROUTER_SOFTMAX_TOPK) {
        /* the selection is taken on the probabilities, as the pages order it */
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        if (!p) return -3;
        double m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - m); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;
        top_k_desc(p, E, k, idx);
        free(p);
    } else {
        top_k_desc(l, E, k, idx);
    }
    return orc_weights_for_selection(c, l, idx, wt);
}

/* ---- step 3: experts ------------------------------------------------------ */

static double activation(const orc_config *c, double gate, double up)
{
    if (c->act == ORC_ACT_SWIGLU)
        return silu(gate) * up;
    /* gpt-oss: gate clamped from above only, up on both sides, (up + 1) */
    double g = gate < c->act_limit ? gate : c->act_limit;
    double u = up;
    if (u < -c->act_limit) u = -c->act_limit;
    if (u > c->act_limit) u = c->act_limit;
    return (u + 1.0) * g * sigmoid(c->act_alpha * g);
}

int orc_expert(const orc_config *c, const orc_weights *w, int e,
               const double *xr, double *h, double *y)
{
    const int H = c->hidden, F = c->expert_ff;
    if (e < 0 || e >= c->n_expert) return -1;
    double *gate = (double *)malloc(sizeof(double) * (size_t)F);
    double *up = (double *)malloc(sizeof(double) * (size_t)F);
    if (!gate || !up) { free(gate); free(up); return -3; }

    if (c->gate_up_interleaved) {
        double *z = (double *)malloc(sizeof(double) * 2 * (size_t)F);
        if (!z) { free(gate); free(up); return -3; }
        matvec(w->gate_up_w, c->w_dtype, (size_t)e * 2 * F * H, 2 * F, H, xr, z);
        if (c->has_bias)
            for (int r = 0; r < 2 * F; ++r)
                z[r] += load(w->gate_up_b, c->w_dtype, (size_t)e * 2 * F + r);
        for (int j = 0; j < F; ++j) { gate[j] = z[2 * j]; up[j] = z[2 * j + 1]; }
        free(z);
    } else {
        matvec(w->gate_w, c->w_dtype, (size_t)e * F * H, F, H, xr, gate);
        matvec(w->up_w, c->w_dtype, (size_t)e * F * H, F, H, xr, up);
        if (c->has_bias)
            for (int j = 0; j < F; ++j) {
                gate[j] += load(w->gate_up_b, c->w_dtype, (size_t)e * 2 * F + j);
                up[j] += load(w->gate_up_b, c->w_dtype, (size_t)e * 2 * F + F + j);
            }
    }
    for (int j = 0; j < F; ++j) h[j] = activation(c, gate[j], up[j]);
    matvec(w->down_w, c->w_dtype, (size_t)e * H * F, H, F, h, y);
    if (c->has_bias)
        for (int i = 0; i < H; ++i)
            y[i] += load(w->down_b, c->w_dtype, (size_t)e * H + i);
    free(gate);
    free(up);
    return 0;
}

int orc_shared(const orc_config *c, const orc_weights *w, const double *xr,
               double *h, double *y, double *gate_out)
{
    const int H = c->hidden, Fs = c->shared_ff;
    if (Fs <= 0) return -1;
    double *g = (double *)malloc(sizeof(double) * (size_t)Fs);
    double *u = (double *)malloc(sizeof(double) * (size_t)Fs);
    if (!g || !u) { free(g); free(u); return -3; }
    matvec(w->sh_gate_w, c->w_dtype, 0, Fs, H, xr, g);
    matvec(w->sh_up_w, c->w_dtype, 0, Fs, H, xr, u);
    for (int j = 0; j < Fs; ++j) h[j] = silu(g[j]) * u[j];
    matvec(w->sh_down_w, c->w_dtype, 0, H, Fs, h, y);
    double s = 0.0;
    for (int i = 0; i < H; ++i) s += load(w->sh_gate_inp, c->w_dtype, (size_t)i) * xr[i];
    *gate_out = sigmoid(s);
    free(g);
    free(u);
    return 0;
}

/* ---- steps 4 and 5: combine ----------------------------------------------- */

int orc_token_output(const orc_config *c, const orc_weights *w, const double *xr,
                     const int *idx, const double *wt, double *out)
{
    const int H = c->hidden, F = c->expert_ff, k = c->top_k;
    int Fmax = F > c->shared_ff ? F : c->shared_ff;
    double *h = (double *)malloc(sizeof(double) * (size_t)Fmax);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    int rc = 0;
    if (!h || !y) { rc = -3; goto done; }
    for (int i = 0; i < H; ++i) out[i] = 0.0;
    for (int j = 0; j < k; ++j) {
        rc = orc_expert(c, w, idx[j], xr, h, y);
        if (rc) goto done;
        for (int i = 0; i < H; ++i) out[i] += wt[j] * y[i];
    }
    if (c->shared_ff > 0) {
        double gate;
        rc = orc_shared(c, w, xr, h, y, &gate);
        if (rc) goto done;
        for (int i = 0; i < H; ++i) out[i] += gate * y[i];
    }
done:
    free(h);
    free(y);
    return rc;
}

int orc_forward(const orc_config *c, const orc_weights *w, const void *x,
                int n_tokens, const int *rows, int n_rows, double *out,
                int *idx, double *wt, int n_threads)
{
    if (orc_check_config(c) || !w || !x || !out || n_tokens < 0) return -1;
    if (!rows) n_rows = n_tokens;
    if (n_rows < 0) return -1;
    if (rows)
        for (int r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= n_tokens) return -1;
    const int H = c->hidden, E = c->n_expert, k = c->top_k;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads) reduction(| : failed)
#endif
    for (int r = 0; r < n_rows; ++r) {
        int t = rows ? rows[r] : r;
        double *xr = (double *)malloc(sizeof(double) * (size_t)H);
        double *l = (double *)malloc(sizeof(double) * (size_t)E);
        int *ti = (int *)malloc(sizeof(int) * (size_t)k);
        double *tw = (double *)malloc(sizeof(double) * (size_t)k);
        if (!xr || !l || !ti || !tw) {
            failed = 1;
        } else {
            load_row(c, x, t, xr);
            router_row(c, w, xr, l, NULL);
            if (orc_select(c, l, ti, tw) ||
                orc_token_output(c, w, xr, ti, tw, out + (size_t)r * H))
                failed = 1;
            for (int j = 0; j < k; ++j) {
                if (idx) idx[(size_t)r * k + j] = ti[j];
                if (wt) wt[(size_t)r * k + j] = tw[j];
            }
        }
        free(xr);
        free(l);
        free(ti);
        free(tw);
    }
    (void)n_threads;
    return failed ? -3 : 0;
}

/* ---- MXFP4 expert weights (see moe_oracle.h) ---- */
double orc_e2m1_value(unsigned code)
{
    const unsigned sign = (code >> 3) & 1u, ex = (code >> 1) & 3u, man = code & 1u;
    const double mag = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, (int)ex - 1);
    return sign ? -mag : mag;
}

double orc_e8m0_scale(unsigned e8m0)
{
    return e8m0 == 255u ? NAN : ldexp(1.0, (int)e8m0 - 127);
}

int orc_mxfp4_dequant(const uint8_t *blocks, const uint8_t *scales, int64_t rows, int cols, float *out)
{
    if (!blocks || !scales || !out || rows < 0 || cols <= 0 || cols % 32) return -1;
    const int nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            const double sc = orc_e8m0_scale(scales[r * nb + b]);
            const uint8_t *blk = blocks + (r * nb + b) * 16;
            for (int j = 0; j < 32; ++j) {
                const unsigned byte = blk[j / 2];
                const unsigned code = (j & 1) ? (byte >> 4) : (byte & 15u);
                out[r * cols + b * 32 + j] = (float)(orc_e2m1_value(code) * sc);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Q4 records ("Engine" (cherenkov), section "Prefill": Q4 GEMMs with half
 * weights and float accumulation; "Qwen3.5-MoE Model Implementation", KV
 * Cache: ggml-Q4_0 rows).  A row is cols/32 blocks of 18 bytes: a half
 * (IEEE binary16, little-endian) scale d, then 16 bytes of codes, byte j
 * holding element j in its low nibble and element j + 16 in its high
 * nibble; element = (code - 8) * d.
 * ---------------------------------------------------------------------- */
double orc_fp16_value(unsigned h)
{
    const int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                 /* zero and subnormals */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

int orc_q4_dequant(const uint8_t *blocks, int64_t rows, int cols, float *out)
{
    if (!blocks || !out || rows < 0 || cols <= 0 || cols % 32) return -1;
    const int nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = blocks + (r * nb + b) * 18;
            const double d = orc_fp16_value((unsigned)blk[0] | ((unsigned)blk[1] << 8));
            for (int j = 0; j < 32; ++j) {
                const unsigned byte = blk[2 + (j & 15)];
                const unsigned code = j < 16 ? (byte & 15u) : (byte >> 4);
                out[r * cols + b * 32 + j] = (float)(((double)code - 8.0) * d);  /* exact in float */
            }
        }
    }
    return 0;
}
