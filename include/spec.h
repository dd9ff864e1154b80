/*
 * spec.h -- C ABI of the GB300 MTP speculative-decoding hot path.
 *
 * One step of the method, as the pages state it:
 *   draft  -- a light drafter head reads the target's last hidden state and
 *             cross-attends the target's own KV cache (no cache of its own) to
 *             propose k tokens ("Accelerating Gemini Nano on Pixel with frozen
 *             multi-token prediction" (ai-news-spoon), sections "The late-exit
 *             strategy" and "Zero-copy architecture");
 *   verify -- the target runs ONE forward pass over the k drafted positions
 *             plus its own next position ("Gemma 4's MTP drafter explained"
 *             (molayo1419.me), section "How does speculative decoding work?");
 *   accept -- keep the drafts up to the first disagreement, drop the rest, and
 *             append the target's own token, so a step emits between 1 and k+1
 *             tokens and the output equals plain greedy decoding of the target
 *             (same section; "Gemma 4 acceleration with MTP drafters"
 *             (cafe.daangn.com), section "How MTP works").
 *
 * Conventions for every entry point:
 *  - All device memory (weights, KV pool, block table, sequence state,
 *    workspace, inputs and outputs) is allocated by the caller and borrowed.
 *    The library allocates no device memory; spec_destroy frees host objects
 *    and captured CUDA graphs only.
 *  - Pointers marked "device" must point to device memory of the current
 *    device; "host" pointers are read before the call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    is the legacy default stream, on which graph capture is disabled).
 *  - Arguments are validated on the host before any launch; an invalid call
 *    returns SPEC_EINVAL and leaves all state unchanged. Kernels never trap:
 *    a capacity or page-table violation found on the device sets an error
 *    word, skips the offending access and leaves the sequence state as it was;
 *    spec_sync() reports it as SPEC_ECAPACITY.
 *  - Alignment: every tensor 16-byte aligned; weights and KV pages 128-byte
 *    aligned.
 *  - Nothing is thrown across the ABI.
 */
#ifndef SPEC_GB300_H
#define SPEC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = 1,      /* bad argument (null pointer, shape, range)           */
    SPEC_ECAPACITY = 2,   /* a sequence would run past its pages / the workspace */
    SPEC_ESTATE = 3,      /* call order violated (e.g. verify before prefill)    */
    SPEC_ECUDA = 4,       /* a CUDA runtime call failed                          */
    SPEC_ETIMEOUT = 5,    /* a bounded device wait gave up                        */
    SPEC_EUNSUPPORTED = 6 /* shape or dtype combination not built                 */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1, SPEC_Q4_0 = 2 } spec_dtype;

/* A stack of L row-major weight matrices [N][K] ("device").
 *  SPEC_F32 / SPEC_BF16: data holds L*N*K elements; scales = NULL.
 *  SPEC_Q4_0: 32-value blocks with one fp16 scale and 4-bit codes, value =
 *    scale * (code - 8) ("Gemma 4's MTP drafter explained", section "Step 1 -
 *    repacking the QAT drafter": every 32-value block holds at most 16
 *    distinct values, the Q4_0 layout). Stored as two planes: data = codes,
 *    L*N*K/2 bytes, element i of a block in the low nibble of byte i (i < 16)
 *    or the high nibble of byte i-16; scales = L*N*K/32 fp16. K % 32 == 0. */
typedef struct {
    int32_t dtype;
    const void *data;
    const void *scales;
} spec_matrix;

/* Target decoder: pre-norm layers of RMSNorm -> QKV -> RoPE -> causal GQA
 * attention -> O (+residual), RMSNorm -> gate/up -> GELU(gate)*up -> down
 * (+residual); final RMSNorm; LM head tied to the embedding.
 * Mixture of experts (n_experts > 0; "Gemma 4 acceleration: faster inference
 * with multi-token prediction drafters" (cafe.daangn.com), section "MTP drafter
 * internal optimisations" names a 26B mixture-of-experts target without its
 * layer): the FFN becomes router scores W_r . xn over n_experts experts, each
 * row's top_k experts by score (ties to the lower id), softmax weights over
 * the chosen scores, and a gated-GELU FFN of width d_ff_expert per expert,
 * y = sum of weight * expert(xn). top_k <= 8, n_experts <= 256; f32 or bf16
 * weights. */
typedef struct {
    int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ff, vocab;
    int32_t w_dtype;     /* spec_dtype of every matrix, embedding included  */
    int32_t kv_dtype;    /* SPEC_F32 or SPEC_BF16                           */
    float rms_eps;       /* 1e-6                                            */
    float rope_theta;    /* 10000, rotate-half pairing                      */
    int32_t n_experts;   /* 0: dense FFN                                    */
    int32_t top_k;       /* experts per row (mixture of experts)            */
    int32_t d_ff_expert; /* width of one expert's FFN                       */
} spec_model_desc;

typedef struct {
    spec_matrix embed;   /* [vocab][d_model], also the LM head               */
    spec_matrix wqkv;    /* n_layers x [(nq+2nkv)*hd][d_model]: q, k, v rows  */
    spec_matrix wo;      /* n_layers x [d_model][nq*hd]                      */
    spec_matrix wgu;     /* n_layers x [2*d_ff][d_model]: gate rows, up rows  */
    spec_matrix wdown;   /* n_layers x [d_model][d_ff]                       */
    const float *g_attn; /* [n_layers][d_model] RMSNorm gains                */
    const float *g_ffn;  /* [n_layers][d_model]                              */
    const float *g_final;/* [d_model]                                        */
    spec_matrix router;  /* mixture of experts: n_layers x [n_experts][d_model] */
    spec_matrix wgu_e;   /* (n_layers * n_experts) x [2*d_ff_expert][d_model]: gate rows, up rows */
    spec_matrix wdown_e; /* (n_layers * n_experts) x [d_model][d_ff_expert]  */
} spec_weights;

/* Drafter head ("Gemma 4's MTP drafter explained", section "What is different
 * about Gemma 4's drafter?": 4 layers, hidden 256, reads the target's
 * backbone-width hidden state, clustered output with 2048 centroids). Query
 * heads use the target's head_dim and map onto the target's KV heads. */
typedef struct {
    int32_t n_layers, hidden, d_ff, n_q_heads;
    int32_t clustered;     /* 0: full-vocabulary head; 1: centroid shortcut   */
    int32_t n_centroids;   /* 2048                                           */
    int32_t top_c;         /* clusters kept (32)                              */
    int32_t w_dtype;
} spec_drafter_desc;

typedef struct {
    spec_matrix w_in;      /* [hidden][2*d_model] over [N(h); N(E[tok])]      */
    const float *g_in_h, *g_in_e;    /* [d_model]                             */
    spec_matrix wq;        /* n_layers x [nq*hd][hidden]                      */
    spec_matrix wo;        /* n_layers x [hidden][nq*hd]                      */
    spec_matrix wgu;       /* n_layers x [2*d_ff][hidden]                     */
    spec_matrix wdown;     /* n_layers x [hidden][d_ff]                       */
    const float *g_attn, *g_ffn;     /* [n_layers][hidden]                    */
    const float *g_out;    /* [hidden]                                        */
    spec_matrix w_out;     /* [d_model][hidden]: next hidden state             */
    spec_matrix vocab;     /* [vocab][hidden], rows in cluster order if clustered */
    spec_matrix centroids; /* [n_centroids][hidden] (clustered only)          */
    const int32_t *perm;   /* [vocab] token id of row p (clustered only)      */
} spec_drafter_weights;

/* Paged KV cache ("device"). pool: [n_layers][n_pages][2][n_kv_heads][64][head_dim]
 * in kv_dtype (K plane then V plane per page). block_table: int32
 * [n_slots][max_pages_per_seq]; position p of slot s lives in page
 * block_table[s][p/64], row p%64. Keys are stored after RoPE. */
typedef struct {
    void *pool;
    int32_t n_pages;
    int32_t page_size;            /* must be 64 */
    const int32_t *block_table;
    int32_t max_pages_per_seq;
    int32_t n_slots;
} spec_kv_desc;

/* Per-slot decoding state ("device"; caller-owned, so it can be saved and
 * restored). seq_len: committed cache positions; pending: the last emitted
 * token, not yet in the cache; hid: final-normed target hidden state of the row
 * that produced `pending` (seeds the drafter); stats: passes, drafted,
 * accepted, emitted. */
typedef struct {
    int32_t *seq_len;   /* [n_slots] */
    int32_t *pending;   /* [n_slots] */
    float *hid;         /* [n_slots][d_model] */
    int64_t *stats;     /* [n_slots][4] */
} spec_state;

typedef struct {
    int64_t passes, drafted, accepted, emitted;
    double tokens_per_pass; /* emitted / passes = 1 + accepted / passes */
} spec_stats_t;

typedef struct spec_ctx spec_ctx;

/* Bytes of workspace needed for batches of up to B_max sequences, prompts of
 * up to rows_max tokens per sequence (>= k_max + 1) and sequences of up to
 * max_pages_per_seq KV pages. A target pass takes at most
 * P = min(rows_max, 64, 128 / (n_q_heads / n_kv_heads)) rows per sequence;
 * longer prompts run as consecutive passes of P rows, and k_max + 1 <= P.
 * Returns 0 on invalid descriptors. */
size_t spec_workspace_bytes(const spec_model_desc *m, const spec_drafter_desc *d,
                            int32_t B_max, int32_t rows_max, int32_t max_pages_per_seq);

/* Validate descriptors and pointers and bind them to a new context. The
 * descriptors and weight structs are copied; the device buffers they point to
 * must outlive the context. `drafter`/`dweights` may be NULL (no spec_draft).
 * `workspace` ("device", ws_bytes >= spec_workspace_bytes(...)) is zeroed on
 * `stream` here and owned by the context until spec_destroy. */
spec_status spec_init(const spec_model_desc *model, const spec_weights *weights,
                      const spec_drafter_desc *drafter, const spec_drafter_weights *dweights,
                      const spec_kv_desc *kv, const spec_state *state, int32_t B_max,
                      int32_t rows_max, void *workspace, size_t ws_bytes, void *stream,
                      spec_ctx **out);

/* Prompt processing: feed R tokens per sequence (tokens "device" int32 [B][R])
 * at positions seq_len..seq_len+R-1, commit them all, set pending to the
 * target's choice after the last one and hid to its hidden state. The target
 * processes the whole context before drafting starts; the drafter has no
 * prefill of its own ("Accelerating Gemini Nano on Pixel with frozen
 * multi-token prediction" (ai-news-spoon), section "Zero-copy architecture").
 * R <= rows_max; prompts longer than a pass (see spec_workspace_bytes) run as
 * consecutive causal passes within the call. seq_ids ("device" int32 [B])
 * name distinct slots. A caller that filled the cache itself sets seq_len
 * first and feeds the last prompt token with R = 1. */
spec_status spec_prefill(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t R,
                         const int32_t *tokens, void *stream);

/* Draft k tokens per sequence into drafts ("device" int32 [B][k]). Reads the
 * slot state and the target's last-layer KV pages; writes nothing else. */
spec_status spec_draft(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t k,
                       int32_t *drafts, void *stream);

/* Verify: rows [pending, d_1..d_k] per sequence in one target pass, greedy
 * accept, KV-length rollback. out_tokens ("device" int32 [B][k+1]) gets the
 * emitted tokens t_0..t_A followed by -1; n_emitted ("device" int32 [B]) gets
 * A+1 in [1, k+1]. logits_dbg ("device" float [B*(k+1)][vocab]) may be NULL;
 * when given it receives every row's logits. k in [0, P-1], P the rows of a
 * pass (see spec_workspace_bytes). */
spec_status spec_verify(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t k,
                        const int32_t *drafts, int32_t *out_tokens, int32_t *n_emitted,
                        float *logits_dbg, void *stream);

/* Lenient verify ("Accelerating Gemini Nano on Pixel with frozen multi-token
 * prediction" (ai-news-spoon), section "Future directions": relaxing the strict
 * token match between draft and verification for some uses; the pages give no
 * rule). Here draft d_j is accepted while every earlier draft was and d_j ranks
 * among the target's top_m tokens of row j-1 (rank = tokens with a higher
 * binary32 logit, or an equal one and a lower index); the step emits the
 * accepted drafts followed by the target's own choice at the next row, commits
 * those rows and rolls the rest back, as spec_verify does. top_m = 1 is
 * spec_verify's greedy accept; larger values no longer reproduce plain greedy
 * decoding. k in [1, P-1] (P as for spec_verify), top_m >= 1. The rows' logits go to
 * logits_dbg when given, else to the workspace. */
spec_status spec_verify_topm(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t k,
                             const int32_t *drafts, int32_t top_m, int32_t *out_tokens,
                             int32_t *n_emitted, float *logits_dbg, void *stream);

/* Tree verify ("Accelerating Gemini Nano on Pixel with frozen multi-token
 * prediction" (ai-news-spoon), section "Future directions": exploring branching
 * possibilities in parallel so that long sequences are accepted more often;
 * the pages give no algorithm). Per sequence, n draft nodes: tokens ("device"
 * int32 [B][n]) and parents ("device" int32 [B][n]; -1: a child of the pending
 * token, the root; else an earlier node index). One target pass verifies the
 * root and every node: node i sits at position seq_len + depth(i) and sees the
 * committed keys, the root and its own ancestors. Greedy accept walks from the
 * root: the lowest-index child whose token equals the target's choice at the
 * current node is accepted, and so on. out_tokens ([B][n+1]) gets the accepted
 * tokens followed by the target's choice at the last accepted node, then -1;
 * n_emitted in [1, depth + 1]. The root and the accepted nodes stay in the
 * cache at consecutive positions (their keys and values are moved there), the
 * other nodes are dropped. A chain (parents[i] = i - 1) is spec_verify.
 * n in [1, P-1] (P as for spec_verify), at most 16. */
spec_status spec_verify_tree(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t n,
                             const int32_t *tokens, const int32_t *parents, int32_t *out_tokens,
                             int32_t *n_emitted, float *logits_dbg, void *stream);

/* spec_draft followed by spec_verify on the context's own draft buffer. */
spec_status spec_step(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t k,
                      int32_t *out_tokens, int32_t *n_emitted, void *stream);

/* Plain greedy decoding: one target token per sequence (spec_verify, k = 0). */
spec_status spec_decode(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t *out_tok,
                        void *stream);

/* Acceptance-rate injection for measurements (not part of the method): draft j
 * of sequence b is replaced by ref[slot][seq_len + j] when draws[b*k + j-1] <
 * alpha, else by (ref[...] + offsets[b*k + j-1]) mod vocab. ref ("device"
 * int32 [n_slots][ref_len]) holds the target's greedy token for every absolute
 * position; draws ("device" float) and offsets ("device" int32, in
 * [1, vocab-1]) hold B*k values. */
spec_status spec_inject_drafts(spec_ctx *ctx, int32_t B, const int32_t *seq_ids, int32_t k,
                               int32_t *drafts, const int32_t *ref, int32_t ref_len,
                               float alpha, const float *draws, const int32_t *offsets,
                               void *stream);

/* One weight-streaming projection, the kernel every linear layer of the pass
 * runs: y[m][n] = sum_k xn[m][k] * W[n][k] for m < M, n < N, where xn = x, or
 * RMSNorm(x) * gain when gain is not NULL. w points to one [N][K] matrix
 * ("device"; for Q4_0 both planes). x ("device" float [M][K]), gain ("device"
 * float [K] or NULL), y ("device" float [M][N]). 1 <= M <= 64. workspace
 * ("device", ws_bytes >= spec_linear_workspace_bytes(N, K, M)) holds split-tile
 * partials and arrival counters; it must be zeroed before its first use and
 * the kernel leaves it zeroed. Calls sharing a workspace must not overlap.
 * Exposed for kernel-level checks and timing; the passes above call the same
 * kernel. */
size_t spec_linear_workspace_bytes(int32_t N, int32_t K, int32_t M);
spec_status spec_linear(const spec_matrix *w, int32_t N, int32_t K, const float *x, int32_t M,
                        const float *gain, float eps, float *y, void *workspace, size_t ws_bytes,
                        void *stream);

/* spec_linear without a caller workspace, for callers that cannot allocate
 * device memory (a host application that owns the whole device-memory budget,
 * a plugin whose framework allocator must see every allocation, code that must
 * not reach cudaMalloc because it can synchronise the device). The pages have
 * no counterpart of this call: it only moves spec_linear's scratch (split-tile
 * partials and arrival counters) into a fixed 512 KiB array in the library's
 * device image, held by every GPU that loads the library until the process
 * exits. Same arguments and results as spec_linear otherwise, with one
 * difference in how the work runs: M > 8 rows run as passes of 8 rows on the
 * register-fragment kernel, each pass streaming W again (spec_linear runs 9-64
 * rows in one tcgen05 pass, whose activation planes would not fit the array).
 *  - N may be at most SPEC_LINEAR_NOALLOC_MAX_ROWS; larger N returns
 *    SPEC_ECAPACITY without launching anything.
 *  - The first call on a device looks up the array's address with that device
 *    current; make it before any stream capture.
 *  - All calls share the array: calls that overlap on the GPU (other streams,
 *    other host threads) race on it and must be serialised by the caller.
 *  - The counters are cleared on `stream` at the start of every call.
 * Allocates nothing (no cudaMalloc / cudaFree, no allocating library call). */
#define SPEC_LINEAR_NOALLOC_MAX_ROWS 523776
spec_status spec_linear_noalloc(const spec_matrix *w, int32_t N, int32_t K, const float *x, int32_t M,
                                const float *gain, float eps, float *y, void *stream);

/* One attention launch over the paged cache, the kernels every pass runs (a
 * kernel-level entry for checks and timing; the passes call the same code).
 * Causal attention of the verified rows ("Gemma 4's MTP drafter explained"
 * (molayo1419.me), section "How does speculative decoding work?": the target
 * checks every drafted position in one pass): with key_extra = 1, row i of
 * sequence b sits at position seq_len[seq_ids[b]] + i, its key and value are
 * already in the cache, and it attends keys [0, seq_len + i]; with key_extra =
 * 0 every row of sequence b attends [0, seq_len) (the drafter's
 * cross-attention into the target's cache, "Accelerating Gemini Nano on Pixel
 * with frozen multi-token prediction" (ai-news-spoon), "Zero-copy
 * architecture"). Scores are q.k / sqrt(head_dim), softmax in fp32.
 *  m: head_dim, n_kv_heads, kv_dtype and n_layers describe the cache (other
 *     fields must be valid but are unused); kv: the cache; layer: which layer.
 *  seq_ids ("device" int32 [B]) and seq_len ("device" int32 [n_slots]).
 *  q ("device" float [B*R][n_q_heads*head_dim], row b*R+i, head h at column
 *     h*head_dim, already rotated); query head h reads KV head
 *     h / (n_q_heads / n_kv_heads). out ("device" float, same shape).
 *  workspace ("device", ws_bytes >= spec_attention_workspace_bytes(m, B, R,
 *     n_q_heads, kv->max_pages_per_seq)): zeroed before its first use; the
 *     kernels leave it zeroed except the split partials.
 * B <= 64, R <= 64, R * n_q_heads / n_kv_heads <= 128. A page id out of range
 * is skipped and recorded in the workspace's first int (SPEC_ECAPACITY's
 * device code 2). Asynchronous on `stream`. */
size_t spec_attention_workspace_bytes(const spec_model_desc *m, int32_t B, int32_t R, int32_t n_q_heads,
                                      int32_t max_pages_per_seq);
spec_status spec_attention(const spec_model_desc *m, const spec_kv_desc *kv, int32_t layer, int32_t B,
                           const int32_t *seq_ids, const int32_t *seq_len, int32_t R, int32_t n_q_heads,
                           int32_t key_extra, const float *q, float *out, void *workspace, size_t ws_bytes,
                           void *stream);

/* Copy one slot's counters to the host (synchronises `stream`). */
spec_status spec_stats(spec_ctx *ctx, int32_t slot, spec_stats_t *out, void *stream);

/* Wait for `stream` and report (then clear) the device error word. */
spec_status spec_sync(spec_ctx *ctx, void *stream);

/* Capture each distinct call shape in a CUDA graph and replay it (default on
 * for non-NULL streams). */
spec_status spec_set_graphs(spec_ctx *ctx, int32_t enable);

/* Execution options:
 *  SPEC_OPT_GRAPHS      (default 1) capture each call shape in a CUDA graph
 *                       and replay it;
 *  SPEC_OPT_PREFETCH    (default 0) each projection CTA first pulls its share
 *                       of the weights towards L2 (bulk L2 prefetch).
 * Changing an option drops the captured graphs. */
#define SPEC_OPT_GRAPHS 1
#define SPEC_OPT_PREFETCH 4
/*  SPEC_OPT_TEST_ATTN_WAIT (default 0; for failure-detection tests only) 1:
 *                       the split merge of the tensor-core attention waits for
 *                       one more arrival than there are splits, so its bounded
 *                       wait (about one second) runs out: the launch records
 *                       a timeout, skips the merge and returns, and the pass
 *                       commits nothing; spec_sync then reports SPEC_ETIMEOUT
 *                       and later passes run normally once the option is 0. */
#define SPEC_OPT_TEST_ATTN_WAIT 8
/*  SPEC_OPT_WIDE_TRACE  value = a device pointer to a zeroed uint64 buffer of at
 *                       least 256 * n_SMs * 16 entries, or 0: the next 256
 *                       enqueued projections record per-CTA globaltimer stamps.
 *                       A register-fragment launch (at most 8 rows, bf16 or
 *                       Q4_0) uses slots 2 entry, 3 past the launch dependency,
 *                       0 activations staged, 1 main loop done, 4 done. A
 *                       tcgen05 launch (passes of more than 8 rows) records
 *                       (ns) in 16 slots: 0 entry, 1 setup done, 2 producer past
 *                       the launch dependency, 3 first stage consumed, 4 last
 *                       MMA issued, 5 last accumulator ready, 6 epilogue done,
 *                       7 tensor memory freed, 8 last split-tile partial
 *                       written, 9 its arrival counted, 10 partials summed (the
 *                       tile's last CTA), 11 that tile finished, 12 first
 *                       accumulator ready, 13 first tile done; slots a CTA does
 *                       not reach stay as they were. Launch i uses entries
 *                       [i * n_SMs * 16, (i + 1) * n_SMs * 16). Stamps are taken
 *                       when a launch runs; with graphs on, the launches of a
 *                       captured shape keep the slots of their capture. */
#define SPEC_OPT_WIDE_TRACE 7
spec_status spec_set_option(spec_ctx *ctx, int32_t option, int64_t value);

/* Number of kernels the library launched (or replayed inside graphs) since the
 * context was created. */
int64_t spec_kernel_launches(const spec_ctx *ctx);

const char *spec_status_str(spec_status s);
void spec_destroy(spec_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif
