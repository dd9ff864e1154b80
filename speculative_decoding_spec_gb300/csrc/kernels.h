// kernels.h -- internal interface between the C-ABI controller and the
// sm_103a kernels. Plain types only; every launcher enqueues on `st` and
// returns the number of kernels it launched (negative on a launch error).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

enum { DT_F32 = 0, DT_BF16 = 1, DT_Q4_0 = 2 };

// Device error word values (first error wins).
enum { SPEC_ERR_NONE = 0, SPEC_ERR_TOKEN = 1, SPEC_ERR_CAPACITY = 2, SPEC_ERR_REF = 3, SPEC_ERR_TIMEOUT = 4 };

// One row-major matrix [N][K] (a layer of a stack, offset already applied).
struct Mat {
  int dtype;
  const void* data;
  const void* scales;  // Q4_0 only: fp16 [N][K/32]
};

// Byte offset of layer l of a stack of [N][K] matrices.
__host__ __device__ inline Mat mat_layer(Mat m, int l, int N, int K) {
  long long e = (long long)l * N * K;
  if (m.dtype == DT_F32) m.data = (const char*)m.data + e * 4;
  else if (m.dtype == DT_BF16) m.data = (const char*)m.data + e * 2;
  else {
    m.data = (const char*)m.data + e / 2;
    m.scales = (const char*)m.scales + (e / 32) * 2;
  }
  return m;
}

enum Epi { EPI_STORE = 0, EPI_ADD = 1, EPI_GEGLU = 2, EPI_ARGMAX = 3, EPI_ROPE = 4 };

// EPI_ROPE: the QKV projection's epilogue rotates q and k heads (rotate-half
// RoPE with the pass's cos/sin table), writes rotated q to Y and k, v to the
// paged cache at each row's position.
struct RopeEpi {
  int nq, nkv, hd, R;
  const float* rope_cs;      // [M][hd/2][2]
  const int32_t* pos;        // [M]
  const int32_t* seq_ids;    // [B]
  void* pool;                // bf16 pool
  long long layer_off;       // elements to this layer
  int n_pages, max_pages;
  const int32_t* block_table;
  int* err;
};
enum Tail { TAIL_NONE = 0, TAIL_VERIFY = 1, TAIL_PREFILL = 2, TAIL_DRAFT = 3, TAIL_TREE = 4 };

// Tree verify: whether pass row i of a sequence sees key `key`: every committed
// key (key < L0) and, of the pass's own rows (stored at L0 + row), those set in
// the row's ancestor mask (bit r: row r is the row itself or an ancestor).
// mask_i = ~0u outside tree verify (the causal limit alone decides).
__host__ __device__ inline bool tree_visible(unsigned int mask_i, int L0, int key) {
  const int r = key - L0;
  return r < 0 || r >= 32 || ((mask_i >> r) & 1u);
}

// What the last CTA of an argmax launch does once every row's argmax is known.
struct TailArgs {
  int mode;
  int B, R, k;
  const int32_t* seq_ids;   // [B]
  const int32_t* drafts;    // VERIFY: [B][k]
  int32_t* out_tokens;      // VERIFY: [B][k+1]
  int32_t* n_emitted;       // VERIFY: [B]
  int32_t* seq_len;         // state [slots]
  int32_t* pending;         // state [slots]
  int64_t* stats;           // state [slots][4]
  int32_t* sel_row;         // [B] pass row whose hidden seeds the drafter
  int32_t* draft_out;       // DRAFT: [B][draft_ld]
  int draft_ld, draft_j;
  const int32_t* parents;   // TREE: [B][k] parent node of each draft node (-1: the root)
  int32_t* path;            // TREE: [B][path_ld] rows of the accepted path (root first)
  int path_ld;
  const int32_t* token_of;  // optional row -> token id map (clustered head)
  unsigned long long* best_all;  // every pass row's packed argmax, zeroed by the last CTA
  unsigned int* counter;    // arrival counter, reset by the last CTA
  int* err;
};

// Scratch of the tcgen05 projection for 9..64 rows (gemm_wide.cu); all null:
// that path is not used and more rows run as passes of 8.
struct WideScratch {
  uint16_t* xs;             // [2][64][kmax] bf16 activation planes (hi, lo)
  float* rms;               // [64][16] per-row sums of squares of 1024-column blocks (RMSNorm)
  float* fix;               // gemv_wide_fix_bytes(): split-tile partial sums
  int kmax;                 // largest K the planes hold
  int* err;                 // device error word (timeouts), may be null
  unsigned long long* trace;  // optional [grid][16] globaltimer stamps of this launch
  // Planes written by the kernel that produced this launch's input, with no
  // RMSNorm on it (the attention before O, the gated GELU before down):
  // `ready` = 1, no preparation kernel, 1/rms = 1.
  int ready;
  // EPI_ADD producer: split tiles only publish their partial sums (`defer`),
  // and the next projection's preparation adds them up, in CTA order, into the
  // residual rows (fix_*: the producer's partials and unit split).
  int defer;
  const float* fix_src;
  int fix_U, fix_grid, fix_C, fix_T;
  // This launch's EPI_GEGLU output as the next projection's planes:
  // out_xs [2][MP][N'] (N' = the output width), fp16 when out_f16 (a Q4_0
  // consumer), or null.
  uint16_t* out_xs;
  int out_f16;
};

struct GemvArgs {
  const float* X;           // [M][ldx] fp32 activations
  int ldx, M, N, K;
  Mat W;
  const float* gain;        // RMSNorm prologue gain [K] (nullptr: none)
  float eps;
  int epi;
  float* Y;                 // output [M][ldy] (STORE / ADD / GEGLU; ARGMAX: optional logits)
  int ldy;
  int geglu_half;           // GEGLU: rows j and j+half pair; Y has `half` columns
  unsigned long long* best; // ARGMAX: [M] packed (score, row) keys, zero before the launch
  TailArgs tail;
  RopeEpi rope;
  int m_base;               // absolute index of row 0 of X (row tables of EPI_ROPE)
  float* tc_fix;            // tensor-core kernel: split-tile partials (gemv_tc_fixup_bytes())
  unsigned int* tc_cnt;     // tensor-core kernel: per-tile arrival counters, zero between launches
  int pdl;                  // launch with programmatic dependent launch
  int prefetch;             // tensor-core kernel: pull the CTA's weight slice to L2 first
  WideScratch wide;         // tcgen05 path for more than 8 rows (bf16 weights)
  unsigned long long* tc_trace;  // optional [grid][16] globaltimer stamps of a register-fragment launch
};
int gemv(const GemvArgs& a, cudaStream_t st);
// True when gemv() runs this projection on the tcgen05 kernel (one launch
// for up to 64 rows).
bool gemv_goes_wide(const GemvArgs& a);

// Per-pass row setup: tokens, positions and RoPE cos/sin for M = B*R rows.
struct RowsArgs {
  int B, R, mode;           // mode: TAIL_VERIFY (rows = [pending, drafts]) or TAIL_PREFILL
  const int32_t* seq_ids;
  const int32_t* tokens;    // PREFILL: [B][tok_ld], this pass's R from column 0; VERIFY: drafts [B][R-1]
  int tok_ld;               // PREFILL: row stride of tokens (the whole prompt's length)
  const int32_t* parents;   // tree verify: [B][R-1] parent node of each draft node (-1: the root); else null
  unsigned int* tree_mask;  // tree verify: [M] ancestor mask of each row (out)
  const int32_t* pending;
  const int32_t* seq_len;
  Mat embed;
  int d, hd;
  float theta;
  float* x;                 // [M][d] embedding rows (fp32)
  int32_t* pos;             // [M]
  float* rope_cs;           // [M][hd/2][2]
  int* err;
  int vocab;
};
int embed_rows(const RowsArgs& a, cudaStream_t st);

struct RopeAppendArgs {
  float* qkv;               // [M][nqkv] in/out: q and k rotated in place
  int M, R, nq, nkv, hd;
  const float* rope_cs;
  const int32_t* pos;       // [M]
  const int32_t* seq_ids;
  void* pool;
  int kv_dtype;
  long long layer_elems;    // elements per layer of the pool
  int layer, n_pages, max_pages;
  const int32_t* block_table;
  int* err;
};
int rope_append(const RopeAppendArgs& a, cudaStream_t st);

struct AttnArgs {
  const float* q;           // [M][ldq]; head h at column h*hd
  int ldq;
  int B, R, nq, nkv, hd;
  int key_extra;            // keys of row i: [0, seq_len + i + key_extra)
  const void* pool;
  int kv_dtype;
  long long layer_elems;
  int layer, n_pages, max_pages;
  const int32_t* block_table;
  const int32_t* seq_ids;
  const int32_t* seq_len;
  const float* rope_cs;     // when non-null, q is rotated on load with [M][hd/2][2]
  const unsigned int* tree_mask;  // tree verify: [B*R] ancestor mask of each row (tree_visible); else null
  int n_split, pages_per_split;
  float* part_o;            // [M][nq][n_split][hd]
  float* part_ml;           // [M][nq][n_split][2]
  float* out;               // [M][nq*hd] merged output
  int* err;
  int standalone;           // 1: launched outside the library's kernel chain (no programmatic launch)
  // tcgen05 kernel only: the merged rows also as the next projection's
  // activation planes, hi at planes[m][c], lo at planes[planes_mp + m][c]
  // (c < nq*hd; fp16 when planes_f16), or null
  uint16_t* planes;
  int planes_mp, planes_f16;
};
int attention(const AttnArgs& a, cudaStream_t st);

// Lenient accept (accept_topm.cu): drafts kept while each ranks among the
// target's top_m tokens of its row; the pass's LM head wrote every row's logits
// and its packed argmax (best, consumed and zeroed here).
struct TopmArgs {
  int B, k, top_m, V, S;       // S: vocabulary parts per draft (set by the launcher)
  const int32_t* seq_ids;      // [B]
  const int32_t* drafts;       // [B][k]
  const float* logits;         // [B*(k+1)][V]
  unsigned long long* best;    // [B*(k+1)]
  unsigned int* rank;          // [B*k] counts, zero between launches
  unsigned int* counter;       // arrival counter, zero between launches
  int32_t *out_tokens, *n_emitted, *seq_len, *pending, *sel_row;
  int64_t* stats;
  int* err;
};
int topm_accept(const TopmArgs& a, cudaStream_t st);

// Tree verify: the accepted path's K/V rows (all layers) moved from their
// pass slots (seq_len_old + row) to consecutive positions (seq_len_old + j).
// Skipped when the device error word is set (nothing was committed).
struct TreeMoveArgs {
  int B, R, L, nkv, hd, kv_bytes;   // kv_bytes: 2 (bf16) or 4 (fp32)
  const int32_t* seq_ids;
  const int32_t* seq_len;           // already advanced by A + 1
  const int32_t* n_emitted;         // [B] A + 1
  const int32_t* path;              // [B][path_ld]
  int path_ld;
  void* pool;
  long long layer_elems;
  int max_pages;
  const int32_t* block_table;
  int n_pages;
  const int* err;
};
int tree_move(const TreeMoveArgs& a, cudaStream_t st);

// Mixture-of-experts FFN (moe.cu) of M pass rows: routing of the router scores
// z, grouped expert projections over the rows routed to each expert, and the
// weighted combine into the residual x.
struct MoeArgs {
  int M, E, K, d, ff;          // rows, experts, experts per row, width, expert FFN width
  const float* xn;             // [M][d] normalised rows (FFN gain applied)
  const float* z;              // [M][E] router scores
  int32_t* sel;                // [M][K] chosen experts
  float* wts;                  // [M][K] their softmax weights
  int32_t* cnt;                // [E] rows per expert
  int32_t* list;               // [E][M] selections (row * K + slot) per expert, row order
  float* act;                  // [M*K][ff] expert intermediates per selection
  float* out;                  // [M*K][d] expert outputs per selection
  float* x;                    // [M][d] residual (in/out)
};
void setup_moe_attributes();
size_t moe_smem(int d, int ff);
int moe_ffn(const MoeArgs& a, const void* wgu_layer, const void* wdown_layer, int wdtype, cudaStream_t st);
int rmsnorm_rows(const float* x, int M, int d, const float* g, float eps, float* xn, cudaStream_t st);

// Final-normed hidden state of the row chosen by the accept step -> slot state.
// Skipped when the device error word `err` is set (the pass commits nothing).
int commit_hidden(int B, const int32_t* seq_ids, const int32_t* sel_row, const float* x, int d,
                  const float* g_final, float eps, float* hid_state, const int* err, cudaStream_t st);

// Drafter step input: cat[b] = [N(h); N(E[tok])], RoPE table at the draft position.
struct DraftInArgs {
  int B, j, k, d, hd;
  const int32_t* seq_ids;
  const float* h_prev;      // j == 1: slot state hid[slot]; else [B][d]
  int h_from_state;
  const int32_t* pending;
  const int32_t* drafts;    // [B][k] (token of step j-1 when j > 1)
  const int32_t* seq_len;
  Mat embed;
  const float* g_h;
  const float* g_e;
  float eps, theta;
  float* cat;               // [B][2d]
  float* rope_cs;           // [B][hd/2][2]
};
int draft_input(const DraftInArgs& a, cudaStream_t st);

// Clustered head: top-C clusters per row, then member scoring + argmax.
struct ClusterArgs {
  int B, C, top_c, cs, h;
  const float* scores;      // [B][C] centroid scores
  int32_t* chosen;          // [B][top_c]
  const float* u;           // [B][h] raw drafter state (normalised here)
  const float* g_out;
  float eps;
  Mat vocab;                // [V][h] cluster-sorted rows
  const int32_t* perm;
  unsigned long long* best; // [B]
  TailArgs tail;
};
int cluster_head(const ClusterArgs& a, cudaStream_t st);

int inject_drafts(int B, int k, const int32_t* seq_ids, const int32_t* seq_len, int32_t* drafts,
                  const int32_t* ref, int ref_len, float alpha, const float* draws,
                  const int32_t* offsets, int vocab, int* err, cudaStream_t st);

// Set the dynamic shared-memory limits of every kernel (call once, outside
// stream capture).
void setup_gemv_attributes();
void setup_gemv_tc_attributes();
int gemv_tc(const GemvArgs& a, float* fix, unsigned int* cnt, cudaStream_t st);
size_t gemv_tc_fixup_bytes();
void setup_gemv_wide_attributes();
bool gemv_wide_ok(const GemvArgs& a);
// The unit split a tcgen05 launch of `a` uses (tile-major units of C 64-column
// chunks over T tiles, balanced over `grid` CTAs), and whether its split tiles
// can be left to the next projection's preparation (balanced ranges, at most
// 16 CTAs on a tile, at most 128 tiles).
struct WideSplit {
  int U, grid, C, T;
  bool deferrable;
};
WideSplit gemv_wide_split(const GemvArgs& a);
// bf16 matrices of at least this many elements (64 MB) take the tcgen05 path at
// any row count: they stream at about 70-90% of the HBM rate there, the
// register-fragment kernel reaches about half of it on long rows.
constexpr long long WIDE_MIN_ELEMS = 1ll << 25;
// ... and rows of at least this many columns (shorter rows stream well on the
// register-fragment kernel: a 262144 x 1536 LM head reaches about 88% of the
// copy bandwidth there)
constexpr int WIDE_MIN_K = 4096;
int gemv_wide(const GemvArgs& a, cudaStream_t st);
size_t gemv_wide_fix_bytes();
// bytes of WideScratch for activation planes of up to kmax columns (0 when kmax == 0)
inline size_t gemv_wide_xs_bytes(int kmax) { return (size_t)2 * 64 * kmax * 2; }
void setup_attn_attributes();
void setup_draft_attributes();

constexpr int MAX_DEVICES = 64;
int num_sms();
// Sets every kernel's dynamic shared-memory limit on the current device, once
// per device (function attributes are per device). Call outside stream capture.
void setup_device_attributes();

// tensor-core attention for bf16 caches (head_dim 64 or 128)
size_t attention_tc_smem(int hd, int qn, int r);
size_t attention_tc_smem_slots(int hd, int qn, int r, int pw);
void setup_attn_tc_attributes();
int attention_tc_splits(int B, int nkv, int max_pages, int* pps, int qn);
int attention_tc(const AttnArgs& a, unsigned int* counters, int pps, cudaStream_t st);
size_t attention_smem(int hd, int qn);
// tcgen05 attention (attn_flash.cu): bf16 cache, head_dim 128, at most 32
// query rows (R x GQA group) per (sequence, KV head). counters: 2 x B x nkv
// words, zero between launches. wait_extra > 0 makes the split merge's
// bounded wait run out (failure-detection tests only). Returns 1, -2 when the
// shape is not covered, -1 on a launch error.
void setup_attn_flash_attributes();
// The tcgen05 attention's partials are CTA-major: CTA c writes query rows
// [c*32, c*32 + 32) of part_o / part_ml (a compact block the pair's CTAs read
// back), so the partial buffers hold at least this many rows on top of the
// pair-major layout of the other attention kernels.
constexpr int ATTN_FLASH_PART_ROWS = 256 * 32;
bool attention_flash_ok(const AttnArgs& a);
int attention_flash(const AttnArgs& a, unsigned int* counters, int wait_extra, cudaStream_t st);

}  // namespace spec
