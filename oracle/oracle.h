/*
 * oracle.h -- plain, slow CPU reference of MTP speculative decoding.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product path (the CUDA library
 * under speculative_decoding_spec_gb300/) never calls it and shares no code,
 * header, table or helper with it.
 *
 * Arithmetic: every weight is dequantised exactly to double, every product is
 * accumulated in double, activations are double. The KV cache is stored in the
 * model's KV dtype (fp32 or bf16) because that is the state the method keeps;
 * values are held here as float after rounding to that dtype.
 *
 * Sources (page title and section):
 *  [P1] "Gemma 4 acceleration: faster inference with multi-token prediction
 *       drafters" (cafe.daangn.com), sections "How MTP works" and
 *       "MTP drafter internal optimisations".
 *  [P4] "Accelerating Gemini Nano on Pixel with frozen multi-token prediction"
 *       (ai-news-spoon), sections "The late-exit strategy", "Advantages of a
 *       frozen backbone", "Zero-copy architecture".
 *  [P5] "Gemma 4's MTP drafter explained: speculative decoding and ..."
 *       (molayo1419.me), sections "Why is generating one token at a time
 *       slow?", "How does speculative decoding work?", "What is different
 *       about Gemma 4's drafter?", "Step 1 - repacking the QAT drafter",
 *       "Step 3 - serving the target with the drafter".
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_Q4_0 = 2 };

/* A weight matrix [N][K] stored row-major in one of three formats.
 * OR_F32 / OR_BF16: data = N*K elements.
 * OR_Q4_0: data = codes, N rows of K/2 bytes; scales = N rows of K/32 fp16.
 *          Block b of a row holds elements 32b..32b+31; element i of a block is
 *          the low nibble of byte i (i < 16) or the high nibble of byte i-16;
 *          value = scale_b * (code - 8).  [P5 "Step 1"]: blocks of 32 values,
 *          at most 16 distinct values per block, one scale per block. */
typedef struct {
    int dtype;
    const void *data;
    const uint16_t *scales;
} or_w;

typedef struct {
    int L, d, nq, nkv, hd, ff, V;
    int kv_dtype;            /* OR_F32 or OR_BF16 */
    double eps, theta;       /* RMSNorm epsilon, RoPE base */
    or_w embed;              /* [V][d], also the (tied) LM head */
    or_w wqkv;               /* L x [(nq+2nkv)*hd][d]: q rows, then k rows, then v rows */
    or_w wo;                 /* L x [d][nq*hd] */
    or_w wgu;                /* L x [2*ff][d]: gate rows then up rows */
    or_w wdown;              /* L x [d][ff] */
    const float *g_attn;     /* [L][d] */
    const float *g_ffn;      /* [L][d] */
    const float *g_final;    /* [d] */
    /* mixture of experts (n_experts = 0: the dense FFN above) */
    int n_experts, top_k, ff_e;
    or_w router;             /* L x [n_experts][d] */
    or_w wgu_e;              /* L x n_experts x [2*ff_e][d]: gate rows then up rows */
    or_w wdown_e;            /* L x n_experts x [d][ff_e] */
} or_model;

typedef struct {
    int L, h, bh, ff, nq, hd, nkv;
    int clustered;           /* 0: full-vocabulary head, 1: centroid shortcut */
    int n_centroids, top_c, cluster_size, V;
    or_w w_in;               /* [h][2*bh] */
    const float *g_in_h;     /* [bh] */
    const float *g_in_e;     /* [bh] */
    or_w wq;                 /* L x [nq*hd][h] */
    or_w wo;                 /* L x [h][nq*hd] */
    or_w wgu;                /* L x [2*ff][h] */
    or_w wdown;              /* L x [h][ff] */
    const float *g_attn;     /* [L][h] */
    const float *g_ffn;      /* [L][h] */
    const float *g_out;      /* [h] */
    or_w w_out;              /* [bh][h] */
    or_w vocab;              /* [V][h]; cluster-sorted rows when clustered */
    or_w centroids;          /* [n_centroids][h] */
    const int32_t *perm;     /* [V] token id of sorted row p (clustered only) */
} or_drafter;

/* One sequence: its KV cache and decoding state.
 * kv: float [L][2][nkv][cap][hd] (K then V), values rounded to kv_dtype.
 * len: committed positions; pending: emitted token not yet in the cache;
 * hid: final-normed hidden state of the row that produced `pending`. */
typedef struct {
    float *kv;
    int cap;
    int len;
    int pending;
    double *hid;             /* [d] */
} or_seq;

/* ---- single operations (exposed so the tests can pin each one) ---- */
double or_bf16_to_double(uint16_t b);
double or_f16_to_double(uint16_t h);
float  or_round_kv(double x, int kv_dtype);
void   or_dequant_row(const or_w *w, int K, int64_t n, double *out);
void   or_linear(const or_w *w, int N, int K, const double *x, int M, double *y);
void   or_rmsnorm(const double *x, int d, const float *g, double eps, double *out);
void   or_rope(double *v, int hd, int64_t pos, double theta);
double or_gelu(double x);
void   or_attend(const double *q, const float *K, const float *V, int n_keys,
                 int hd, double *o);
int    or_argmax_f32(const double *logits, int n, double *margin);
/* The k largest of n binary32-rounded scores (ties: lower index first), in
 * order; gap (optional) = smallest distance between a chosen and an unchosen
 * score. */
void   or_topk_f32(const double *scores, int n, int k, int32_t *idx, double *gap);
/* One row through a mixture-of-experts FFN layer l: y = sum over the row's
 * top_k experts (router scores on xn) of softmax-weight * expert FFN(xn). */
void   or_moe_ffn(const or_model *m, int l, const double *xn, double *y);

/* ---- target model ---- */
/* Forward R rows of one sequence at positions len..len+R-1 (causal). Writes
 * the rows' K/V into the cache (len is NOT advanced). Outputs are optional. */
int or_forward(const or_model *m, or_seq *s, const int32_t *tokens, int R,
               double *logits, int32_t *argmax, double *margin, double *hid);
/* or_forward plus the residual stream of every row after the last layer,
 * before the final RMSNorm (resid [R][d], optional). */
int or_forward_resid(const or_model *m, or_seq *s, const int32_t *tokens, int R,
                     double *logits, int32_t *argmax, double *margin, double *hid,
                     double *resid);
/* Prompt processing: forward, commit all R rows, pending = argmax of the last
 * row, hid = its hidden. */
int or_prefill(const or_model *m, or_seq *s, const int32_t *tokens, int R,
               double *margin_last);
/* Greedy accept of one verify pass. t[0..k] are the target's argmax tokens of
 * rows [pending, d_1..d_k]; returns A = accepted drafts. */
int or_accept(int k, const int32_t *drafts, const int32_t *t);
/* One verify step: rows [pending, drafts], accept, emit, roll back. */
int or_verify(const or_model *m, or_seq *s, int k, const int32_t *drafts,
              int32_t *out_tokens, int32_t *n_emitted, double *margins);
/* Rank of token tok among n logits rounded to binary32: how many tokens come
 * before it (higher logit, or equal logit and lower index). */
int or_rank_f32(const double *logits, int n, int tok);
/* Lenient verify: accept drafts while each ranks among the target's top_m
 * tokens at its row; emit the accepted drafts then the target's own choice.
 * top_m = 1 is or_verify. decision [k] (optional): per draft, the logit
 * distance to the rank boundary it was judged against (INFINITY if not
 * judged). */
int or_verify_topm(const or_model *m, or_seq *s, int k, const int32_t *drafts, int top_m,
                   int32_t *out_tokens, int32_t *n_emitted, double *margins, double *decision);
/* Tree verify: n draft nodes (tokens, parents: -1 = child of the pending
 * token, else an earlier node); each node's target choice after its root
 * path; accept the lowest-index matching child from the root down; emit the
 * accepted tokens then the target's choice at the last accepted node; keep the
 * root and the accepted path in the cache. margins [n+1]: per node (root
 * first) the top-1 minus top-2 gap of its choice. */
int or_verify_tree(const or_model *m, or_seq *s, int n, const int32_t *tokens, const int32_t *parents,
                   int32_t *out_tokens, int32_t *n_emitted, double *margins);
/* n plain greedy steps (verify with k = 0); out[i] = emitted token i. */
int or_greedy(const or_model *m, or_seq *s, int n, int32_t *out, double *margins);

/* ---- drafter ---- */
int or_draft(const or_model *m, const or_drafter *dr, const or_seq *s, int k,
             int32_t *drafts, double *margins);
/* or_draft plus, per step j, the normalised state the head reads
 * (u_bar [k][h]) and the next hidden state h_j = W_out . u (h_next [k][bh]). */
int or_draft_states(const or_model *m, const or_drafter *dr, const or_seq *s, int k,
                    int32_t *drafts, double *margins, double *u_bar, double *h_next);
/* The drafter's output head on one normalised drafter state u_bar [h]. */
int or_draft_head(const or_drafter *dr, const double *u_bar, double *margin);

#ifdef __cplusplus
}
#endif
#endif
