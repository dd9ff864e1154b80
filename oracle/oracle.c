/*
 * oracle.c -- plain, slow CPU reference of MTP speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg. Nothing here is shared with the CUDA path.
 * Sources are named in oracle.h ([P1], [P4], [P5]).
 *
 * Every function follows the plain definition of the operation: no blocking,
 * fusion or reordering. Dot products run in index order in double precision;
 * output rows are independent, so the OpenMP split over rows does not change
 * any result.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

double or_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an IEEE binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double or_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, mant = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-14 / 1024 */
    else if (e == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp(1.0 + mant / 1024.0, e - 15);
    return sign ? -v : v;
}

/* The cache keeps K/V in the model's KV dtype. A value computed in double is
 * rounded to binary32 and, for a bf16 cache, then to bf16 (round to nearest,
 * ties to even), i.e. the cast an fp32 activation receives when stored. */
float or_round_kv(double x, int kv_dtype)
{
    float f = (float)x;
    if (kv_dtype != OR_BF16)
        return f;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) != 0x7f800000u) { /* finite */
        u += 0x7fffu + ((u >> 16) & 1u);
        u &= 0xffff0000u;
    }
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------ */
/* weights                                                             */
/* ------------------------------------------------------------------ */

/* Row n of a [N][K] matrix, dequantised exactly. Q4_0 per [P5 "Step 1"]:
 * 32-value blocks, one scale each, 4-bit codes; value = scale * (code - 8). */
void or_dequant_row(const or_w *w, int K, int64_t n, double *out)
{
    if (w->dtype == OR_F32) {
        const float *p = (const float *)w->data + n * (int64_t)K;
        for (int k = 0; k < K; ++k)
            out[k] = p[k];
    } else if (w->dtype == OR_BF16) {
        const uint16_t *p = (const uint16_t *)w->data + n * (int64_t)K;
        for (int k = 0; k < K; ++k)
            out[k] = or_bf16_to_double(p[k]);
    } else {
        const uint8_t *c = (const uint8_t *)w->data + n * (int64_t)(K / 2);
        const uint16_t *s = w->scales + n * (int64_t)(K / 32);
        for (int b = 0; b < K / 32; ++b) {
            double scale = or_f16_to_double(s[b]);
            for (int i = 0; i < 32; ++i) {
                uint8_t byte = c[b * 16 + (i & 15)];
                int code = i < 16 ? (byte & 0xf) : (byte >> 4);
                out[b * 32 + i] = scale * (double)(code - 8);
            }
        }
    }
}

/* The l-th [N][K] matrix of a stack of L matrices. */
static or_w layer_slice(const or_w *w, int l, int N, int K)
{
    or_w r = *w;
    int64_t elems = (int64_t)l * N * K;
    if (w->dtype == OR_F32)
        r.data = (const float *)w->data + elems;
    else if (w->dtype == OR_BF16)
        r.data = (const uint16_t *)w->data + elems;
    else {
        r.data = (const uint8_t *)w->data + elems / 2;
        r.scales = w->scales + elems / 32;
    }
    return r;
}

/* y[m][n] = sum_k x[m][k] * W[n][k] for M input rows. */
void or_linear(const or_w *w, int N, int K, const double *x, int M, double *y)
{
#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            or_dequant_row(w, K, n, row);
            for (int m = 0; m < M; ++m) {
                const double *xm = x + (int64_t)m * K;
                double acc = 0.0;
                for (int k = 0; k < K; ++k)
                    acc += xm[k] * row[k];
                y[(int64_t)m * N + n] = acc;
            }
        }
        free(row);
    }
}

/* ------------------------------------------------------------------ */
/* elementwise operations                                              */
/* ------------------------------------------------------------------ */

/* RMSNorm: x / sqrt(mean(x^2) + eps) * g. */
void or_rmsnorm(const double *x, int d, const float *g, double eps, double *out)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / d + eps);
    for (int i = 0; i < d; ++i)
        out[i] = x[i] * inv * (double)g[i];
}

/* Rotary embedding, rotate-half pairing: element i and i + hd/2 rotate by the
 * angle pos * theta^(-2i/hd). */
void or_rope(double *v, int hd, int64_t pos, double theta)
{
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double ang = (double)pos * pow(theta, -2.0 * i / hd);
        double c = cos(ang), s = sin(ang);
        double x0 = v[i], x1 = v[i + half];
        v[i] = x0 * c - x1 * s;
        v[i + half] = x1 * c + x0 * s;
    }
}

/* GELU, exact form x * Phi(x). */
double or_gelu(double x)
{
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

/* softmax(q K^T / sqrt(hd)) V over n_keys keys stored [n][hd]. */
void or_attend(const double *q, const float *K, const float *V, int n_keys,
               int hd, double *o)
{
    for (int i = 0; i < hd; ++i)
        o[i] = 0.0;
    if (n_keys <= 0)
        return;
    double *p = (double *)malloc(sizeof(double) * (size_t)n_keys);
    double scale = 1.0 / sqrt((double)hd), mx = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
        double s = 0.0;
        for (int i = 0; i < hd; ++i)
            s += q[i] * (double)K[(int64_t)j * hd + i];
        p[j] = s * scale;
        if (p[j] > mx)
            mx = p[j];
    }
    double sum = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        p[j] = exp(p[j] - mx);
        sum += p[j];
    }
    for (int j = 0; j < n_keys; ++j) {
        double wj = p[j] / sum;
        for (int i = 0; i < hd; ++i)
            o[i] += wj * (double)V[(int64_t)j * hd + i];
    }
    free(p);
}

/* Greedy choice. The decision is taken on the logits rounded to binary32
 * (the precision the GPU kernels compare in); ties go to the lowest index.
 * margin (optional) = top-1 minus top-2 logit, in double. */
int or_argmax_f32(const double *logits, int n, double *margin)
{
    int best = 0;
    float bv = (float)logits[0];
    for (int i = 1; i < n; ++i) {
        float v = (float)logits[i];
        if (v > bv) {
            bv = v;
            best = i;
        }
    }
    if (margin) {
        double second = -INFINITY;
        for (int i = 0; i < n; ++i)
            if (i != best && logits[i] > second)
                second = logits[i];
        *margin = n > 1 ? logits[best] - second : INFINITY;
    }
    return best;
}

void or_topk_f32(const double *scores, int n, int k, int32_t *idx, double *gap)
{
    char *taken = (char *)calloc((size_t)n, 1);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int i = 0; i < n; ++i)
            if (!taken[i] && (best < 0 || (float)scores[i] > (float)scores[best]))
                best = i;
        taken[best] = 1;
        idx[j] = best;
    }
    if (gap) {
        double lo_in = INFINITY, hi_out = -INFINITY;
        for (int i = 0; i < n; ++i) {
            if (taken[i] && scores[i] < lo_in)
                lo_in = scores[i];
            if (!taken[i] && scores[i] > hi_out)
                hi_out = scores[i];
        }
        *gap = lo_in - hi_out;
    }
    free(taken);
}

/* Mixture-of-experts FFN of one row ([P1 "MTP drafter internal
 * optimisations"]: a 26B mixture-of-experts target, whose routing makes batch
 * 1 the hard case; the pages give no layer definition). Reading: router
 * scores z = W_r . xn; the top_k experts by binary32 score (ties to the lower
 * id); weights = softmax of their scores; each expert is the gated-GELU FFN
 * of the dense layer with its own width ff_e. */
void or_moe_ffn(const or_model *m, int l, const double *xn, double *y)
{
    const int d = m->d, E = m->n_experts, K = m->top_k, ff = m->ff_e;
    double *z = (double *)malloc(sizeof(double) * (size_t)E);
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
    double *gu = (double *)malloc(sizeof(double) * (size_t)2 * ff);
    double *act = (double *)malloc(sizeof(double) * (size_t)ff);
    double *out = (double *)malloc(sizeof(double) * (size_t)d);
    or_w r = layer_slice(&m->router, l, E, d);
    or_linear(&r, E, d, xn, 1, z);
    or_topk_f32(z, E, K, sel, NULL);
    double mx = -INFINITY, tot = 0.0;
    for (int j = 0; j < K; ++j)
        if (z[sel[j]] > mx)
            mx = z[sel[j]];
    for (int j = 0; j < K; ++j)
        tot += exp(z[sel[j]] - mx);
    for (int i = 0; i < d; ++i)
        y[i] = 0.0;
    for (int j = 0; j < K; ++j) {
        const int e = sel[j];
        const double wgt = exp(z[e] - mx) / tot;
        or_w g = layer_slice(&m->wgu_e, l * E + e, 2 * ff, d);
        or_linear(&g, 2 * ff, d, xn, 1, gu);
        for (int i = 0; i < ff; ++i)
            act[i] = or_gelu(gu[i]) * gu[ff + i];
        or_w dn = layer_slice(&m->wdown_e, l * E + e, d, ff);
        or_linear(&dn, d, ff, act, 1, out);
        for (int i = 0; i < d; ++i)
            y[i] += wgt * out[i];
    }
    free(z); free(sel); free(gu); free(act); free(out);
}

/* ------------------------------------------------------------------ */
/* target model                                                        */
/* ------------------------------------------------------------------ */

static float *kv_at(const or_model *m, const or_seq *s, int l, int which, int h)
{
    int64_t plane = (((int64_t)l * 2 + which) * m->nkv + h) * s->cap;
    return s->kv + plane * m->hd;
}

/* Forward pass of R new rows at positions len..len+R-1: the target verifies
 * all drafted positions in one pass ([P5 "How does speculative decoding
 * work?"], [P1 "How MTP works"]). Pre-norm decoder layer:
 *   x += Wo . Attn(RoPE(Wq . N(x)), cache);  x += Wd . (GELU(Wg . N(x)) * (Wu . N(x)))
 * then logits = E . N_f(x) with the LM head tied to the embedding. */
int or_forward(const or_model *m, or_seq *s, const int32_t *tokens, int R,
               double *logits, int32_t *argmax, double *margin, double *hid)
{
    return or_forward_resid(m, s, tokens, R, logits, argmax, margin, hid, NULL);
}

/* or_forward that also hands out the residual stream x of every row after the
 * last layer, before the final RMSNorm (resid [R][d], optional). */
int or_forward_resid(const or_model *m, or_seq *s, const int32_t *tokens, int R,
                     double *logits, int32_t *argmax, double *margin, double *hid,
                     double *resid)
{
    if (R <= 0 || s->len + R > s->cap)
        return -1;
    const int d = m->d, hd = m->hd, qd = m->nq * hd, kd = m->nkv * hd;
    const int nqkv = qd + 2 * kd, ff = m->ff, grp = m->nq / m->nkv;
    double *x = (double *)calloc((size_t)R * d, sizeof(double));
    double *xn = (double *)calloc((size_t)R * d, sizeof(double));
    double *tmp = (double *)calloc((size_t)R * d, sizeof(double));
    double *qkv = (double *)calloc((size_t)R * nqkv, sizeof(double));
    double *att = (double *)calloc((size_t)R * qd, sizeof(double));
    double *gu = (double *)calloc((size_t)R * 2 * ff, sizeof(double));
    double *act = (double *)calloc((size_t)R * ff, sizeof(double));

    for (int r = 0; r < R; ++r)
        or_dequant_row(&m->embed, d, tokens[r], x + (int64_t)r * d);

    for (int l = 0; l < m->L; ++l) {
        for (int r = 0; r < R; ++r)
            or_rmsnorm(x + (int64_t)r * d, d, m->g_attn + (int64_t)l * d, m->eps,
                       xn + (int64_t)r * d);
        or_w w = layer_slice(&m->wqkv, l, nqkv, d);
        or_linear(&w, nqkv, d, xn, R, qkv);
        /* RoPE on q and k at the absolute position; K/V of every new row go
         * into the cache before any row attends (row r sees keys 0..len+r). */
        for (int r = 0; r < R; ++r) {
            int64_t pos = s->len + r;
            double *row = qkv + (int64_t)r * nqkv;
            for (int h = 0; h < m->nq; ++h)
                or_rope(row + h * hd, hd, pos, m->theta);
            for (int h = 0; h < m->nkv; ++h) {
                or_rope(row + qd + h * hd, hd, pos, m->theta);
                float *kc = kv_at(m, s, l, 0, h) + pos * hd;
                float *vc = kv_at(m, s, l, 1, h) + pos * hd;
                for (int i = 0; i < hd; ++i) {
                    kc[i] = or_round_kv(row[qd + h * hd + i], m->kv_dtype);
                    vc[i] = or_round_kv(row[qd + kd + h * hd + i], m->kv_dtype);
                }
            }
        }
        for (int r = 0; r < R; ++r)
            for (int h = 0; h < m->nq; ++h)
                or_attend(qkv + (int64_t)r * nqkv + h * hd, kv_at(m, s, l, 0, h / grp),
                          kv_at(m, s, l, 1, h / grp), s->len + r + 1, hd,
                          att + (int64_t)r * qd + h * hd);
        w = layer_slice(&m->wo, l, d, qd);
        or_linear(&w, d, qd, att, R, tmp);
        for (int64_t i = 0; i < (int64_t)R * d; ++i)
            x[i] += tmp[i];

        for (int r = 0; r < R; ++r)
            or_rmsnorm(x + (int64_t)r * d, d, m->g_ffn + (int64_t)l * d, m->eps,
                       xn + (int64_t)r * d);
        if (m->n_experts > 0) {
            for (int r = 0; r < R; ++r) {
                or_moe_ffn(m, l, xn + (int64_t)r * d, tmp + (int64_t)r * d);
                for (int i = 0; i < d; ++i)
                    x[(int64_t)r * d + i] += tmp[(int64_t)r * d + i];
            }
            continue;
        }
        w = layer_slice(&m->wgu, l, 2 * ff, d);
        or_linear(&w, 2 * ff, d, xn, R, gu);
        for (int r = 0; r < R; ++r)
            for (int j = 0; j < ff; ++j)
                act[(int64_t)r * ff + j] = or_gelu(gu[(int64_t)r * 2 * ff + j]) *
                                           gu[(int64_t)r * 2 * ff + ff + j];
        w = layer_slice(&m->wdown, l, d, ff);
        or_linear(&w, d, ff, act, R, tmp);
        for (int64_t i = 0; i < (int64_t)R * d; ++i)
            x[i] += tmp[i];
    }

    if (resid)
        memcpy(resid, x, sizeof(double) * (size_t)R * d);
    for (int r = 0; r < R; ++r)
        or_rmsnorm(x + (int64_t)r * d, d, m->g_final, m->eps, xn + (int64_t)r * d);
    if (hid)
        memcpy(hid, xn, sizeof(double) * (size_t)R * d);
    double *lg = logits ? logits : (double *)malloc(sizeof(double) * (size_t)R * m->V);
    or_linear(&m->embed, m->V, d, xn, R, lg);
    for (int r = 0; r < R; ++r) {
        int t = or_argmax_f32(lg + (int64_t)r * m->V, m->V, margin ? margin + r : NULL);
        if (argmax)
            argmax[r] = t;
    }
    if (!logits)
        free(lg);
    free(x); free(xn); free(tmp); free(qkv); free(att); free(gu); free(act);
    return 0;
}

int or_prefill(const or_model *m, or_seq *s, const int32_t *tokens, int R,
               double *margin_last)
{
    int32_t *t = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    double *mg = (double *)malloc(sizeof(double) * (size_t)R);
    double *hid = (double *)malloc(sizeof(double) * (size_t)R * m->d);
    int rc = or_forward(m, s, tokens, R, NULL, t, mg, hid);
    if (rc == 0) {
        s->len += R;
        s->pending = t[R - 1];
        memcpy(s->hid, hid + (int64_t)(R - 1) * m->d, sizeof(double) * m->d);
        if (margin_last)
            *margin_last = mg[R - 1];
    }
    free(t); free(mg); free(hid);
    return rc;
}

/* Greedy accept ([P5 "How does speculative decoding work?"]; [P4 "The
 * late-exit strategy"]): keep drafts up to the first one that differs from the
 * target's own choice at that position. drafts[j] is d_{j+1}; t[j] is the
 * target's choice after row j. A = largest j <= k with d_i == t_{i-1} for all
 * i <= j. */
int or_accept(int k, const int32_t *drafts, const int32_t *t)
{
    int A = 0;
    while (A < k && drafts[A] == t[A])
        ++A;
    return A;
}

/* One verify step. The step emits d_1..d_A followed by the target's own token
 * t_A (between 1 and k+1 tokens); since d_i == t_{i-1} for i <= A the emitted
 * tokens are t_0..t_A. The cache keeps rows 0..A (pending and the accepted
 * drafts); the rejected rows are dropped by rolling len back. */
int or_verify(const or_model *m, or_seq *s, int k, const int32_t *drafts,
              int32_t *out_tokens, int32_t *n_emitted, double *margins)
{
    int R = k + 1;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    int32_t *t = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    double *hid = (double *)malloc(sizeof(double) * (size_t)R * m->d);
    rows[0] = s->pending;
    for (int j = 0; j < k; ++j)
        rows[j + 1] = drafts[j];
    int rc = or_forward(m, s, rows, R, NULL, t, margins, hid);
    if (rc == 0) {
        int A = or_accept(k, drafts, t);
        for (int j = 0; j <= A; ++j)
            out_tokens[j] = t[j];
        *n_emitted = A + 1;
        s->len += A + 1;
        s->pending = t[A];
        memcpy(s->hid, hid + (int64_t)A * m->d, sizeof(double) * m->d);
    }
    free(rows); free(t); free(hid);
    return rc;
}

/* Rank of token `tok` among n binary32-rounded logits: the number of tokens
 * ordered before it (a higher logit, or the same logit and a lower index). */
int or_rank_f32(const double *logits, int n, int tok)
{
    float ft = (float)logits[tok];
    int r = 0;
    for (int i = 0; i < n; ++i) {
        float f = (float)logits[i];
        if (f > ft || (f == ft && i < tok))
            ++r;
    }
    return r;
}

/* Lenient verify ([P4 "Future directions"]: the strict token match between
 * draft and verification is relaxed for some uses; the pages give no rule).
 * Reading: draft d_j is accepted while it ranks among the target's top_m
 * tokens of row j-1 (or_rank_f32 < top_m), every earlier draft having been
 * accepted; the step emits the accepted drafts followed by the target's own
 * choice t_A at row A, and keeps rows 0..A in the cache. top_m = 1 is the
 * greedy accept of or_verify. decision (optional, [k]) receives, per draft,
 * the logit distance between the draft and the rank boundary it was judged
 * against (how far the accept decision is from flipping); margins [k+1] the
 * rows' top-1 minus top-2 gaps. */
int or_verify_topm(const or_model *m, or_seq *s, int k, const int32_t *drafts, int top_m,
                   int32_t *out_tokens, int32_t *n_emitted, double *margins, double *decision)
{
    int R = k + 1;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    int32_t *t = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    double *hid = (double *)malloc(sizeof(double) * (size_t)R * m->d);
    double *lg = (double *)malloc(sizeof(double) * (size_t)R * m->V);
    float *sorted = (float *)malloc(sizeof(float) * (size_t)m->V);
    rows[0] = s->pending;
    for (int j = 0; j < k; ++j)
        rows[j + 1] = drafts[j];
    int rc = or_forward(m, s, rows, R, lg, t, margins, hid);
    if (rc == 0) {
        int A = 0;
        for (int j = 0; j < k; ++j) {
            const double *row = lg + (int64_t)j * m->V;
            int d = drafts[j];
            int ok = d >= 0 && d < m->V && or_rank_f32(row, m->V, d) < top_m;
            if (decision) {
                /* the top_m-th and (top_m+1)-th largest binary32 logits */
                for (int i = 0; i < m->V; ++i)
                    sorted[i] = (float)row[i];
                double inside = -INFINITY, outside = -INFINITY;
                for (int r = 0; r <= top_m && r < m->V; ++r) {
                    int best = -1;
                    for (int i = 0; i < m->V; ++i)
                        if (sorted[i] != -INFINITY && (best < 0 || sorted[i] > sorted[best]))
                            best = i;
                    if (best < 0)
                        break;
                    if (r == top_m - 1)
                        inside = sorted[best];
                    if (r == top_m)
                        outside = sorted[best];
                    sorted[best] = -INFINITY;
                }
                double fd = d >= 0 && d < m->V ? (double)(float)row[d] : -INFINITY;
                decision[j] = ok ? fd - outside : inside - fd;
            }
            if (!ok)
                break;
            ++A;
        }
        if (decision)
            for (int j = A + 1; j < k; ++j)
                decision[j] = INFINITY;  /* never judged */
        for (int j = 0; j < A; ++j)
            out_tokens[j] = drafts[j];
        out_tokens[A] = t[A];
        *n_emitted = A + 1;
        s->len += A + 1;
        s->pending = t[A];
        memcpy(s->hid, hid + (int64_t)A * m->d, sizeof(double) * m->d);
    }
    free(rows); free(t); free(hid); free(lg); free(sorted);
    return rc;
}

/* Tree verify ([P4 "Future directions"]: exploring branching possibilities
 * in parallel to raise the chance of accepting a long sequence; the pages give
 * no algorithm). Reading: n draft nodes with tokens[i] and parents[i] (-1: a
 * child of the pending token, the root; else an earlier node). The target's
 * choice at a node is its greedy token after the root path to that node (the
 * committed context, the pending token, the ancestors' tokens, the node's
 * token); here each node's choice comes from a forward pass over exactly that
 * path. Greedy accept walks from the root: the lowest-index child whose token
 * equals the target's choice at the current node is accepted, and so on; the
 * step emits the accepted tokens followed by the target's choice at the last
 * accepted node, and the cache keeps the root and the accepted path at
 * consecutive positions. A chain (parents[i] = i - 1) is or_verify. */
int or_verify_tree(const or_model *m, or_seq *s, int n, const int32_t *tokens, const int32_t *parents,
                   int32_t *out_tokens, int32_t *n_emitted, double *margins)
{
    int32_t *choice = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    double *mg = (double *)malloc(sizeof(double) * (size_t)(n + 1));
    int32_t *path = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 2));
    int32_t *am = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 2));
    double *mm = (double *)malloc(sizeof(double) * (size_t)(n + 2));
    double *hid = (double *)malloc(sizeof(double) * (size_t)(n + 2) * m->d);
    or_seq tmp = *s;
    float *kv_save = NULL;
    int rc = 0;
    /* node r (r = 0: the root; r = i + 1: draft node i): its root path */
    for (int r = 0; r <= n && rc == 0; ++r) {
        int len = 0;
        for (int x = r - 1; x >= 0; x = parents[x]) {
            if (parents[x] >= x) {
                rc = -1;
                break;
            }
            path[len++] = tokens[x];
        }
        if (rc)
            break;
        path[len++] = s->pending;
        for (int i = 0; i < len / 2; ++i) { /* root first */
            int t = path[i];
            path[i] = path[len - 1 - i];
            path[len - 1 - i] = t;
        }
        tmp.len = s->len;
        rc = or_forward(m, &tmp, path, len, NULL, am, mm, NULL);
        choice[r] = am[len - 1];
        mg[r] = mm[len - 1];
    }
    if (rc == 0) {
        /* walk the tree from the root */
        int cur = 0, A = 0;
        for (;;) {
            int next = -1;
            for (int i = 0; i < n; ++i)
                if (parents[i] + 1 == cur && tokens[i] == choice[cur]) {
                    next = i + 1;
                    break;
                }
            if (next < 0)
                break;
            out_tokens[A++] = tokens[next - 1];
            cur = next;
        }
        out_tokens[A] = choice[cur];
        *n_emitted = A + 1;
        if (margins)
            for (int r = 0; r <= n; ++r)
                margins[r] = mg[r];
        /* the committed rows: the root and the accepted path, written again by
         * one forward over them at their final positions */
        path[0] = s->pending;
        for (int j = 0; j < A; ++j)
            path[j + 1] = out_tokens[j];
        rc = or_forward(m, s, path, A + 1, NULL, am, mm, hid);
        if (rc == 0) {
            s->len += A + 1;
            s->pending = choice[cur];
            memcpy(s->hid, hid + (int64_t)A * m->d, sizeof(double) * m->d);
        }
    }
    free(choice); free(mg); free(path); free(am); free(mm); free(hid); free(kv_save);
    return rc;
}

/* Plain greedy decoding: one token per target pass. */
int or_greedy(const or_model *m, or_seq *s, int n, int32_t *out, double *margins)
{
    for (int i = 0; i < n; ++i) {
        int32_t ne;
        int rc = or_verify(m, s, 0, NULL, out + i, &ne, margins ? margins + i : NULL);
        if (rc)
            return rc;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* drafter                                                             */
/* ------------------------------------------------------------------ */

/* Order used for the top-C cluster choice: higher binary32 score first, then
 * lower cluster id. */
typedef struct {
    float key;
    int id;
} or_scored;

static int cmp_scored(const void *a, const void *b)
{
    const or_scored *x = (const or_scored *)a, *y = (const or_scored *)b;
    if (x->key != y->key)
        return x->key > y->key ? -1 : 1;
    return x->id - y->id;
}

/* Output head of the drafter. Full head: argmax over the vocabulary table.
 * Clustered shortcut ([P5 "What is different about Gemma 4's drafter?"]:
 * num_centroids 2048; [P1 "MTP drafter internal optimisations"]: clustering in
 * the embedder so the final logits are cheaper): score every centroid, keep the
 * top_c clusters, score only their member rows, argmax with ties to the lower
 * token id. margin = smallest of the cluster-boundary gap and the final top-1
 * minus top-2 gap. */
int or_draft_head(const or_drafter *dr, const double *u_bar, double *margin)
{
    const int h = dr->h;
    if (!dr->clustered) {
        double *lg = (double *)malloc(sizeof(double) * (size_t)dr->V);
        or_linear(&dr->vocab, dr->V, h, u_bar, 1, lg);
        int t = or_argmax_f32(lg, dr->V, margin);
        free(lg);
        return t;
    }
    const int C = dr->n_centroids, cs = dr->cluster_size;
    double *sc = (double *)malloc(sizeof(double) * (size_t)C);
    or_linear(&dr->centroids, C, h, u_bar, 1, sc);
    or_scored *ord = (or_scored *)malloc(sizeof(or_scored) * (size_t)C);
    for (int c = 0; c < C; ++c) {
        ord[c].key = (float)sc[c];
        ord[c].id = c;
    }
    qsort(ord, (size_t)C, sizeof(or_scored), cmp_scored);
    double cgap = INFINITY;
    if (dr->top_c < C)
        cgap = sc[ord[dr->top_c - 1].id] - sc[ord[dr->top_c].id];

    double *row = (double *)malloc(sizeof(double) * (size_t)h);
    int best_tok = -1;
    float best_v = 0.f;
    double best_d = -INFINITY, second_d = -INFINITY;
    for (int i = 0; i < dr->top_c; ++i) {
        int c = ord[i].id;
        for (int p = c * cs; p < (c + 1) * cs; ++p) {
            or_dequant_row(&dr->vocab, h, p, row);
            double acc = 0.0;
            for (int k = 0; k < h; ++k)
                acc += u_bar[k] * row[k];
            int tok = dr->perm[p];
            float v = (float)acc;
            if (best_tok < 0 || v > best_v || (v == best_v && tok < best_tok)) {
                if (best_tok >= 0 && best_d > second_d)
                    second_d = best_d;
                best_tok = tok;
                best_v = v;
                best_d = acc;
            } else if (acc > second_d) {
                second_d = acc;
            }
        }
    }
    if (margin) {
        double fgap = best_d - second_d;
        *margin = fgap < cgap ? fgap : cgap;
    }
    free(row); free(ord); free(sc);
    return best_tok;
}

/* Draft k tokens. The drafter is a light transformer head on the target's last
 * layer ([P4 "The late-exit strategy"]): it starts from the target's final
 * hidden state and predicts autoregressively; it keeps no cache of its own and
 * cross-attends the target's KV cache directly ([P4 "Zero-copy
 * architecture"]; [P5 "What is different about Gemma 4's drafter?"]: 4 layers
 * of width 256 reading the backbone_hidden_size-wide target state). Step j:
 *   u = W_in . [N(h_{j-1}); N(E[tok_{j-1}])]
 *   per layer: u += Wo' . CrossAttn(RoPE(Wq' . N(u), len+j-1), target last-layer K/V[0, len))
 *              u += Wd' . (GELU(Wg' . N(u)) * (Wu' . N(u)))
 *   h_j = W_out . u;  d_j = head(N_out(u))
 * with h_0 = the target's final-normed hidden of the row that produced the
 * pending token and tok_0 = pending. */
int or_draft(const or_model *m, const or_drafter *dr, const or_seq *s, int k,
             int32_t *drafts, double *margins)
{
    return or_draft_states(m, dr, s, k, drafts, margins, NULL, NULL);
}

/* or_draft that also hands out, per step j, the normalised drafter state the
 * head reads (u_bar [k][h]) and the next hidden state h_j (h_next [k][bh]);
 * both optional. */
int or_draft_states(const or_model *m, const or_drafter *dr, const or_seq *s, int k,
                    int32_t *drafts, double *margins, double *u_bar, double *h_next)
{
    const int h = dr->h, bh = dr->bh, hd = dr->hd, qd = dr->nq * hd, ff = dr->ff;
    const int grp = dr->nq / dr->nkv;
    if (bh != m->d || hd != m->hd || dr->nkv != m->nkv)
        return -1;
    double *hprev = (double *)malloc(sizeof(double) * (size_t)bh);
    double *cat = (double *)malloc(sizeof(double) * (size_t)2 * bh);
    double *e = (double *)malloc(sizeof(double) * (size_t)bh);
    double *u = (double *)malloc(sizeof(double) * (size_t)h);
    double *un = (double *)malloc(sizeof(double) * (size_t)h);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)h);
    double *q = (double *)malloc(sizeof(double) * (size_t)qd);
    double *att = (double *)malloc(sizeof(double) * (size_t)qd);
    double *gu = (double *)malloc(sizeof(double) * (size_t)2 * ff);
    double *act = (double *)malloc(sizeof(double) * (size_t)ff);
    memcpy(hprev, s->hid, sizeof(double) * bh);
    int tok = s->pending;
    const int last = m->L - 1;

    for (int j = 1; j <= k; ++j) {
        or_rmsnorm(hprev, bh, dr->g_in_h, m->eps, cat);
        or_dequant_row(&m->embed, bh, tok, e);
        or_rmsnorm(e, bh, dr->g_in_e, m->eps, cat + bh);
        or_linear(&dr->w_in, h, 2 * bh, cat, 1, u);
        int64_t pos = s->len + j - 1;
        for (int l = 0; l < dr->L; ++l) {
            or_rmsnorm(u, h, dr->g_attn + (int64_t)l * h, m->eps, un);
            or_w w = layer_slice(&dr->wq, l, qd, h);
            or_linear(&w, qd, h, un, 1, q);
            for (int hh = 0; hh < dr->nq; ++hh) {
                or_rope(q + hh * hd, hd, pos, m->theta);
                or_attend(q + hh * hd, kv_at(m, s, last, 0, hh / grp),
                          kv_at(m, s, last, 1, hh / grp), s->len, hd, att + hh * hd);
            }
            w = layer_slice(&dr->wo, l, h, qd);
            or_linear(&w, h, qd, att, 1, tmp);
            for (int i = 0; i < h; ++i)
                u[i] += tmp[i];
            or_rmsnorm(u, h, dr->g_ffn + (int64_t)l * h, m->eps, un);
            w = layer_slice(&dr->wgu, l, 2 * ff, h);
            or_linear(&w, 2 * ff, h, un, 1, gu);
            for (int i = 0; i < ff; ++i)
                act[i] = or_gelu(gu[i]) * gu[ff + i];
            w = layer_slice(&dr->wdown, l, h, ff);
            or_linear(&w, h, ff, act, 1, tmp);
            for (int i = 0; i < h; ++i)
                u[i] += tmp[i];
        }
        or_linear(&dr->w_out, bh, h, u, 1, hprev);
        or_rmsnorm(u, h, dr->g_out, m->eps, un);
        if (u_bar)
            memcpy(u_bar + (int64_t)(j - 1) * h, un, sizeof(double) * h);
        if (h_next)
            memcpy(h_next + (int64_t)(j - 1) * bh, hprev, sizeof(double) * bh);
        tok = or_draft_head(dr, un, margins ? margins + (j - 1) : NULL);
        drafts[j - 1] = tok;
    }
    free(hprev); free(cat); free(e); free(u); free(un); free(tmp);
    free(q); free(att); free(gu); free(act);
    return 0;
}
