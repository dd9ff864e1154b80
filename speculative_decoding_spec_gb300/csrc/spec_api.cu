// spec_api.cu -- the C ABI (include/spec.h): host-side validation, workspace
// layout, the draft / verify / accept pass as a kernel sequence on one stream,
// and a cache of CUDA graphs keyed by call shape.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/spec.h"
#include "kernels.h"

using namespace spec;

namespace {

struct Buf {
  size_t off = 0;
  template <typename T>
  T* take(char* base, size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

struct Work {
  // target pass
  float *x, *qkv, *att, *act, *part_o, *part_ml, *rope_cs;
  int32_t *pos, *sel_row, *n_emit1;
  unsigned long long* best;
  unsigned int* counter;
  unsigned int* attn_count;
  float* lg;                // [M][V] row logits (lenient accept)
  MoeArgs moe;              // mixture-of-experts buffers (null fields for a dense target)
  unsigned int* tmask;      // [M] tree verify: ancestor mask per row
  int32_t* path;            // [B_max][KMAX + 1] tree verify: accepted path rows
  unsigned int *rank, *rank_cnt;
  float* tc_fix;
  unsigned int* tc_cnt;
  WideScratch wide;         // tcgen05 projection scratch (null when passes have <= 8 rows)
  uint16_t* xs_alt;         // second activation-plane buffer (planes written by a producer kernel)
  int* err;
  // drafter
  float *d_cat, *d_u, *d_q, *d_att, *d_act, *d_h, *d_scores, *d_rope, *d_part_o, *d_part_ml;
  int32_t *d_chosen, *d_drafts;
  unsigned long long* d_best;
  unsigned int* d_counter;
  size_t bytes;
};

constexpr int KMAX = 16;
constexpr int WTRACE_LAUNCHES = 256;

// Arrival counters of the tensor-core projection: one per 8 output rows of
// the widest matrix the passes project with.
size_t tc_counters(const spec_model_desc& m, const spec_drafter_desc* d) {
  size_t n = std::max<size_t>({(size_t)m.vocab, (size_t)2 * m.d_ff,
                               (size_t)(m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim, (size_t)m.d_model});
  if (d) n = std::max<size_t>({n, (size_t)2 * d->d_ff, (size_t)d->n_q_heads * m.head_dim,
                               (size_t)std::max(d->n_centroids, 1)});
  return n / 8 + 64;
}

// Rows of one target pass per sequence: at most 64, and at most 128 query rows
// (rows x GQA group) per (sequence, KV head) for the attention. A longer
// prompt runs as consecutive passes of this many rows.
int pass_rows(const spec_model_desc& m, int rows_max) {
  const int G = m.n_q_heads / m.n_kv_heads;
  return std::max(1, std::min({rows_max, 64, 128 / G}));
}

Work carve(char* base, const spec_model_desc& m, const spec_drafter_desc* d, int B_max, int rows_max,
           int max_pages) {
  Work w = {};
  Buf b;
  const size_t M = (size_t)B_max * pass_rows(m, rows_max);
  const int nqkv = (m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim, qd = m.n_q_heads * m.head_dim;
  w.x = b.take<float>(base, M * m.d_model);
  w.qkv = b.take<float>(base, M * nqkv);
  w.att = b.take<float>(base, M * qd);
  w.act = b.take<float>(base, M * m.d_ff);
  w.part_o = b.take<float>(base, (M * m.n_q_heads * (size_t)max_pages + ATTN_FLASH_PART_ROWS) * m.head_dim);
  w.part_ml = b.take<float>(base, (M * m.n_q_heads * (size_t)max_pages + ATTN_FLASH_PART_ROWS) * 2);
  w.rope_cs = b.take<float>(base, M * m.head_dim);
  w.pos = b.take<int32_t>(base, M);
  w.sel_row = b.take<int32_t>(base, B_max);
  w.n_emit1 = b.take<int32_t>(base, B_max);
  w.best = b.take<unsigned long long>(base, M);
  w.counter = b.take<unsigned int>(base, 4);
  w.attn_count = b.take<unsigned int>(base, (size_t)2 * B_max * m.n_kv_heads);
  w.lg = b.take<float>(base, M * m.vocab);
  w.rank = b.take<unsigned int>(base, (size_t)B_max * KMAX);
  w.rank_cnt = b.take<unsigned int>(base, 4);
  w.tmask = b.take<unsigned int>(base, M);
  if (m.n_experts > 0) {
    const int E = m.n_experts, K = m.top_k, ff = m.d_ff_expert;
    w.moe.E = E; w.moe.K = K; w.moe.d = m.d_model; w.moe.ff = ff;
    w.moe.xn = b.take<float>(base, M * m.d_model);
    w.moe.z = b.take<float>(base, M * E);
    w.moe.sel = b.take<int32_t>(base, M * K);
    w.moe.wts = b.take<float>(base, M * K);
    w.moe.cnt = b.take<int32_t>(base, E);
    w.moe.list = b.take<int32_t>(base, (size_t)E * M);
    w.moe.act = b.take<float>(base, M * K * ff);
    w.moe.out = b.take<float>(base, M * K * m.d_model);
  }
  w.path = b.take<int32_t>(base, (size_t)B_max * (KMAX + 1));
  w.tc_fix = b.take<float>(base, gemv_tc_fixup_bytes() / sizeof(float));
  w.tc_cnt = b.take<unsigned int>(base, tc_counters(m, d));
  w.err = b.take<int>(base, 4);
  // a matrix taking the tcgen05 path at any row count (large and long rows)
  const int qd_ = m.n_q_heads * m.head_dim;
  const bool big = (m.d_model >= WIDE_MIN_K && ((long long)m.vocab * m.d_model >= WIDE_MIN_ELEMS ||
                                                2ll * m.d_ff * m.d_model >= WIDE_MIN_ELEMS)) ||
                   (qd_ >= WIDE_MIN_K && (long long)m.d_model * qd_ >= WIDE_MIN_ELEMS) ||
                   (m.d_ff >= WIDE_MIN_K && (long long)m.d_model * m.d_ff >= WIDE_MIN_ELEMS);
  if (M > 8 || (m.w_dtype == SPEC_BF16 && big)) {
    // widest reduction of any projection: target d, q heads, FFN; drafter input [h; e], width, heads, FFN
    int kmax = std::max({2 * m.d_model, m.n_q_heads * m.head_dim, m.d_ff});
    if (d) kmax = std::max({kmax, d->hidden, d->n_q_heads * m.head_dim, d->d_ff});
    w.wide.kmax = kmax;
    w.wide.xs = b.take<uint16_t>(base, gemv_wide_xs_bytes(kmax) / 2);
    w.wide.rms = b.take<float>(base, 64 * 16);  // [64 rows][16 column blocks] sums of squares
    w.wide.fix = b.take<float>(base, gemv_wide_fix_bytes() / sizeof(float));
    w.wide.err = w.err;
    w.xs_alt = b.take<uint16_t>(base, gemv_wide_xs_bytes(kmax) / 2);
  }
  if (d) {
    const int dq = d->n_q_heads * m.head_dim;
    w.d_cat = b.take<float>(base, (size_t)B_max * 2 * m.d_model);
    w.d_u = b.take<float>(base, (size_t)B_max * d->hidden);
    w.d_q = b.take<float>(base, (size_t)B_max * dq);
    w.d_att = b.take<float>(base, (size_t)B_max * dq);
    w.d_act = b.take<float>(base, (size_t)B_max * d->d_ff);
    w.d_h = b.take<float>(base, (size_t)B_max * m.d_model);
    w.d_scores = b.take<float>(base, (size_t)B_max * std::max(d->n_centroids, 1));
    w.d_rope = b.take<float>(base, (size_t)B_max * m.head_dim);
    w.d_part_o = b.take<float>(base, ((size_t)B_max * d->n_q_heads * max_pages + ATTN_FLASH_PART_ROWS) * m.head_dim);
    w.d_part_ml = b.take<float>(base, ((size_t)B_max * d->n_q_heads * max_pages + ATTN_FLASH_PART_ROWS) * 2);
    w.d_chosen = b.take<int32_t>(base, (size_t)B_max * std::max(d->top_c, 1));
    w.d_drafts = b.take<int32_t>(base, (size_t)B_max * KMAX);
    w.d_best = b.take<unsigned long long>(base, B_max);
    w.d_counter = b.take<unsigned int>(base, 4);
  }
  w.bytes = (b.off + 255) & ~size_t(255);
  return w;
}

bool mat_ok(const spec_matrix& mm, int K) {
  if (!mm.data) return false;
  if (mm.dtype == SPEC_Q4_0) return mm.scales && K % 32 == 0;
  if (mm.dtype == SPEC_F32 || mm.dtype == SPEC_BF16) return K % 8 == 0;
  return false;
}

Mat M_(const spec_matrix& m) { return Mat{m.dtype, m.data, m.scales}; }

bool model_ok(const spec_model_desc& m) {
  if (m.n_experts < 0 || (m.n_experts > 0 && (m.n_experts > 256 || m.top_k < 1 || m.top_k > 8 ||
                                               m.top_k > m.n_experts || m.d_ff_expert <= 0 ||
                                               m.d_ff_expert % 8 || m.w_dtype == SPEC_Q4_0)))
    return false;
  return m.n_layers > 0 && m.d_model > 0 && m.n_q_heads > 0 && m.n_kv_heads > 0 && m.head_dim > 0 &&
         m.head_dim % 2 == 0 && m.head_dim <= 256 && m.n_q_heads % m.n_kv_heads == 0 && m.d_ff > 0 &&
         m.vocab > 1 && (m.kv_dtype == SPEC_F32 || m.kv_dtype == SPEC_BF16) && m.d_model % 8 == 0 &&
         m.d_ff % 8 == 0 && (m.w_dtype != SPEC_Q4_0 || (m.d_model % 32 == 0 && m.d_ff % 32 == 0 &&
                                                     (m.n_q_heads * m.head_dim) % 32 == 0));
}

bool drafter_ok(const spec_model_desc& m, const spec_drafter_desc& d) {
  if (d.n_layers <= 0 || d.hidden <= 0 || d.d_ff <= 0 || d.n_q_heads <= 0) return false;
  if (d.n_q_heads % m.n_kv_heads) return false;
  if (d.hidden % 8 || d.d_ff % 8) return false;
  if (d.w_dtype == SPEC_Q4_0 && (d.hidden % 32 || d.d_ff % 32)) return false;
  if (d.clustered) {
    if (d.n_centroids <= 0 || d.n_centroids > 8192 || m.vocab % d.n_centroids) return false;
    if (d.top_c <= 0 || d.top_c > d.n_centroids) return false;
  }
  return true;
}

}  // namespace

struct spec_ctx {
  spec_model_desc m;
  spec_weights w;
  bool has_drafter = false;
  spec_drafter_desc dd;
  spec_drafter_weights dw;
  spec_kv_desc kv;
  spec_state state;
  int B_max, rows_max, pass_rows;
  long long layer_elems;
  Work wk;
  bool graphs = true;
  bool fused_rope = false;
  bool prefetch = false;
  int test_attn_wait = 0;   // SPEC_OPT_TEST_ATTN_WAIT
  unsigned long long* wtrace = nullptr;  // tcgen05 projection timelines (SPEC_OPT_WIDE_TRACE)
  int wtrace_n = 0;
  long long launches = 0;
  struct Entry {
    cudaGraphExec_t exec;
    int kernels;
  };
  std::map<std::string, Entry> cache;
  std::mutex mu;
};

namespace {

// Where a tcgen05 projection takes its activation planes from, and whether it
// writes the next projection's planes (see enqueue_pass).
struct PlaneCfg {
  uint16_t* in_xs = nullptr;
  int ready = 0;
  uint16_t* out_xs = nullptr;
  int out_f16 = 0;
  int defer = 0;                 // EPI_ADD producer leaves its split tiles to the next preparation
  WideSplit fix = {};            // consumer: the deferring producer's split (fix.U > 0: add its partials)
};
int run_gemv(spec_ctx* c, GemvArgs g, cudaStream_t st, const PlaneCfg* pc = nullptr);

int kv_dt(const spec_ctx* c) { return c->m.kv_dtype == SPEC_F32 ? DT_F32 : DT_BF16; }

// Tensor-core attention for bf16 caches with head_dim 64/128; the CUDA-core
// kernels otherwise (fp32 caches). `counters` [B][nkv] are zero between
// launches; the partial buffers of `at` hold max_pages splits per row and head.
int launch_attention(int kv_dtype, AttnArgs at, unsigned int* counters, int wait_extra, cudaStream_t st,
                     bool* flash = nullptr) {
  if (flash) *flash = false;
  if (kv_dtype == SPEC_BF16 && attention_flash_ok(at)) {
    const int r = attention_flash(at, counters, wait_extra, st);
    if (r != -2) {
      if (flash) *flash = r > 0;
      return r;
    }
  }
  at.planes = nullptr;  // only the tcgen05 kernel writes planes
  if (kv_dtype == SPEC_BF16 && (at.hd == 64 || at.hd == 128)) {
    int pps = 1;
    at.n_split = attention_tc_splits(at.B, at.nkv, at.max_pages, &pps, at.R * (at.nq / at.nkv));
    at.pages_per_split = pps;
    const int r = attention_tc(at, counters, pps, st);
    if (r != -2) return r;
    at.n_split = at.max_pages;  // the CUDA-core kernel's split: one page each
    at.pages_per_split = 1;
  }
  return attention(at, st);
}

int run_attention(spec_ctx* c, AttnArgs at, cudaStream_t st, bool* flash = nullptr) {
  return launch_attention(c->m.kv_dtype, at, c->wk.attn_count, c->test_attn_wait, st, flash);
}

}  // namespace

void spec::setup_device_attributes() {
  static std::mutex mu;
  static bool done[MAX_DEVICES];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) dev = 0;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev]) return;
  setup_gemv_attributes();
  setup_attn_attributes();
  setup_attn_tc_attributes();
  setup_draft_attributes();
  setup_attn_flash_attributes();
  setup_moe_attributes();
  done[dev] = true;
}

namespace {

// Workspace of spec_attention: error word, arrival counters, split partials.
struct AttnWork {
  int* err;
  unsigned int* counters;
  float *part_o, *part_ml;
  size_t bytes;
};
AttnWork carve_attention(char* base, int B, int R, int nq, int nkv, int hd, int max_pages) {
  AttnWork w = {};
  Buf b;
  const size_t M = (size_t)B * R;
  w.err = b.take<int>(base, 4);
  w.counters = b.take<unsigned int>(base, (size_t)2 * B * nkv);
  w.part_o = b.take<float>(base, (M * nq * (size_t)max_pages + ATTN_FLASH_PART_ROWS) * hd);
  w.part_ml = b.take<float>(base, (M * nq * (size_t)max_pages + ATTN_FLASH_PART_ROWS) * 2);
  w.bytes = (b.off + 255) & ~size_t(255);
  return w;
}

// ---- the target pass: rows -> layers -> LM head + argmax + accept -----------
int enqueue_pass(spec_ctx* c, int B, const int32_t* seq_ids, int R, int mode, const int32_t* tokens,
                 int32_t* out_tokens, int32_t* n_emitted, float* logits, cudaStream_t st, int top_m = 0,
                 int tok_ld = 0, const int32_t* parents = nullptr) {
  const spec_model_desc& m = c->m;
  const Work& w = c->wk;
  const int M = B * R, d = m.d_model, hd = m.head_dim, nq = m.n_q_heads, nkv = m.n_kv_heads;
  const int nqkv = (nq + 2 * nkv) * hd, qd = nq * hd, ff = m.d_ff;
  int n = 0, r;
#define LAUNCH(expr)        \
  do {                      \
    r = (expr);             \
    if (r < 0) return -1;   \
    n += r;                 \
  } while (0)

  RowsArgs ra = {};
  ra.B = B; ra.R = R; ra.mode = mode; ra.seq_ids = seq_ids; ra.tokens = tokens;
  ra.pending = c->state.pending; ra.seq_len = c->state.seq_len; ra.embed = M_(c->w.embed);
  ra.d = d; ra.hd = hd; ra.theta = m.rope_theta; ra.x = w.x; ra.pos = w.pos; ra.rope_cs = w.rope_cs;
  ra.err = w.err; ra.vocab = m.vocab; ra.tok_ld = tok_ld > 0 ? tok_ld : R;
  ra.parents = parents; ra.tree_mask = parents ? w.tmask : nullptr;
  LAUNCH(embed_rows(ra, st));

  // Activation planes written by the producer. Where the tcgen05 attention
  // feeds O, or a tcgen05 gate/up projection feeds down, the producer also
  // writes the consumer's bf16 (fp16 for Q4_0) hi + lo planes into the plane
  // buffer it does not read itself, and the consumer has no preparation
  // kernel. (These links have no RMSNorm; folding the norm into a residual
  // add's epilogue cost that epilogue about as much as it saved.) The two
  // buffers alternate; a producer writes after its dependency wait, when
  // every earlier reader has finished.
  const bool fuse = w.wide.xs && w.xs_alt && M <= 64;
  uint16_t* bufs[2] = {w.wide.xs, w.xs_alt};
  const int f16 = m.w_dtype == SPEC_Q4_0 ? 1 : 0;
  int rd = -1;          // buffer holding the next projection's planes
  int in_idx = 0;       // buffer the latest tcgen05 projection read
  // A residual-add projection on the tcgen05 kernel whose consumer prepares
  // its planes (O -> gate/up, down -> the next QKV or the LM head) leaves its
  // split tiles' partial sums to that preparation, which adds them into the
  // residual rows in CTA order (the sum the producer's last CTA would make):
  // the producer's CTAs exit after their last tile instead of waiting for
  // the arrivals and finishing tiles one by one.
  WideSplit pending_fix = {};
  auto defer = [&](PlaneCfg& pc, const GemvArgs& prod, bool prod_wide, bool cons_wide) {
    if (!fuse || !prod_wide || !cons_wide || d % 128) return;
    GemvArgs t = prod;
    t.wide = w.wide;
    t.tc_cnt = w.tc_cnt;
    const WideSplit sp = gemv_wide_split(t);
    if (!sp.deferrable) return;
    pc.defer = 1;
    pending_fix = sp;
  };
  auto fixup = [&](PlaneCfg& pc) {
    pc.fix = pending_fix;
    pending_fix = WideSplit{};
  };
  auto wide_of = [&](const GemvArgs& g) {
    GemvArgs t = g;
    t.wide = w.wide;
    t.tc_cnt = w.tc_cnt;
    return fuse && gemv_goes_wide(t);
  };
  // consumer side of projection g (wide: g runs on the tcgen05 kernel)
  auto take = [&](PlaneCfg& pc, bool wide) {
    if (wide && rd >= 0) {
      pc.in_xs = bufs[rd];
      pc.ready = 1;
      in_idx = rd;
    } else if (wide) {
      pc.in_xs = bufs[0];
      in_idx = 0;
    }
    rd = -1;
  };
  // the projections after the attention, built ahead so that their routes are known
  auto o_args = [&](int l) {
    GemvArgs g = {};
    g.X = w.att; g.ldx = qd; g.M = M; g.N = d; g.K = qd;
    g.W = mat_layer(M_(c->w.wo), l, d, qd);
    g.epi = EPI_ADD; g.Y = w.x; g.ldy = d; g.pdl = 1;
    return g;
  };
  auto gu_args = [&](int l) {
    GemvArgs g = {};
    g.X = w.x; g.ldx = d; g.M = M; g.N = 2 * ff; g.K = d;
    g.W = mat_layer(M_(c->w.wgu), l, 2 * ff, d);
    g.gain = c->w.g_ffn + (size_t)l * d; g.eps = m.rms_eps;
    g.epi = EPI_GEGLU; g.geglu_half = ff; g.Y = w.act; g.ldy = ff; g.pdl = 1;
    return g;
  };
  auto down_args = [&](int l) {
    GemvArgs g = {};
    g.X = w.act; g.ldx = ff; g.M = M; g.N = d; g.K = ff;
    g.W = mat_layer(M_(c->w.wdown), l, d, ff);
    g.epi = EPI_ADD; g.Y = w.x; g.ldy = d; g.pdl = 1;
    return g;
  };
  auto qkv_args = [&](int l) {
    GemvArgs g = {};
    g.X = w.x; g.ldx = d; g.M = M; g.N = nqkv; g.K = d;
    g.W = mat_layer(M_(c->w.wqkv), l, nqkv, d);
    g.gain = c->w.g_attn + (size_t)l * d; g.eps = m.rms_eps;
    g.epi = EPI_STORE; g.Y = w.qkv; g.ldy = nqkv; g.pdl = 1;
    return g;
  };
  auto head_args = [&]() {
    GemvArgs g = {};
    g.X = w.x; g.ldx = d; g.M = M; g.N = m.vocab; g.K = d;
    g.W = M_(c->w.embed);
    g.gain = c->w.g_final; g.eps = m.rms_eps;
    g.epi = EPI_ARGMAX; g.Y = logits; g.ldy = m.vocab; g.best = w.best; g.pdl = 1;
    return g;
  };

  const bool fused_rope = c->fused_rope;
  for (int l = 0; l < m.n_layers; ++l) {
    GemvArgs g = qkv_args(l);
    PlaneCfg pq;
    take(pq, wide_of(g));
    fixup(pq);
    if (fused_rope) {
      g.epi = EPI_ROPE;
      RopeEpi& e = g.rope;
      e.nq = nq; e.nkv = nkv; e.hd = hd; e.R = R; e.rope_cs = w.rope_cs; e.pos = w.pos; e.seq_ids = seq_ids;
      e.pool = c->kv.pool; e.layer_off = (long long)l * c->layer_elems; e.n_pages = c->kv.n_pages;
      e.max_pages = c->kv.max_pages_per_seq; e.block_table = c->kv.block_table; e.err = w.err;
    }
    LAUNCH(run_gemv(c, g, st, &pq));

    if (!fused_rope) {
    RopeAppendArgs rp = {};
    rp.qkv = w.qkv; rp.M = M; rp.R = R; rp.nq = nq; rp.nkv = nkv; rp.hd = hd; rp.rope_cs = w.rope_cs;
    rp.pos = w.pos; rp.seq_ids = seq_ids; rp.pool = c->kv.pool; rp.kv_dtype = kv_dt(c);
    rp.layer_elems = c->layer_elems; rp.layer = l; rp.n_pages = c->kv.n_pages;
    rp.max_pages = c->kv.max_pages_per_seq; rp.block_table = c->kv.block_table; rp.err = w.err;
    LAUNCH(rope_append(rp, st));
    }

    AttnArgs at = {};
    at.q = w.qkv; at.ldq = nqkv; at.B = B; at.R = R; at.nq = nq; at.nkv = nkv; at.hd = hd;
    at.key_extra = 1; at.pool = c->kv.pool; at.kv_dtype = kv_dt(c); at.layer_elems = c->layer_elems;
    at.layer = l; at.n_pages = c->kv.n_pages; at.max_pages = c->kv.max_pages_per_seq;
    at.block_table = c->kv.block_table; at.seq_ids = seq_ids; at.seq_len = c->state.seq_len;
    at.rope_cs = nullptr; at.n_split = c->kv.max_pages_per_seq; at.pages_per_split = 1;
    at.part_o = w.part_o; at.part_ml = w.part_ml; at.out = w.att; at.err = w.err;
    at.tree_mask = parents ? w.tmask : nullptr;
    g = o_args(l);
    const bool o_wide = wide_of(g);
    if (o_wide) {
      at.planes = bufs[1 - in_idx];
      at.planes_mp = (M + 15) / 16 * 16;
      at.planes_f16 = f16;
    }
    bool flash = false;
    LAUNCH(run_attention(c, at, st, &flash));
    if (o_wide && flash) rd = 1 - in_idx;

    PlaneCfg po;
    take(po, o_wide);
    if (m.n_experts == 0) defer(po, g, o_wide, wide_of(gu_args(l)));
    LAUNCH(run_gemv(c, g, st, &po));

    if (m.n_experts > 0) {
      // mixture of experts: normalised rows, router scores, routing, grouped
      // experts, weighted combine into the residual
      const int E = m.n_experts, ffe = m.d_ff_expert;
      MoeArgs ma = w.moe;
      ma.M = M; ma.x = w.x;
      LAUNCH(rmsnorm_rows(w.x, M, d, c->w.g_ffn + (size_t)l * d, m.rms_eps, const_cast<float*>(ma.xn), st));
      g = GemvArgs{};
      g.X = ma.xn; g.ldx = d; g.M = M; g.N = E; g.K = d;
      g.W = mat_layer(M_(c->w.router), l, E, d);
      g.epi = EPI_STORE; g.Y = const_cast<float*>(ma.z); g.ldy = E; g.pdl = 1;
      LAUNCH(run_gemv(c, g, st));
      const Mat gu = mat_layer(M_(c->w.wgu_e), l * E, 2 * ffe, d);
      const Mat dn = mat_layer(M_(c->w.wdown_e), l * E, d, ffe);
      LAUNCH(moe_ffn(ma, gu.data, dn.data, m.w_dtype == SPEC_F32 ? DT_F32 : DT_BF16, st));
      continue;
    }
    g = gu_args(l);
    const bool gu_wide = wide_of(g);
    PlaneCfg pg;
    take(pg, gu_wide);
    fixup(pg);
    const GemvArgs gd = down_args(l);
    const bool dn_wide = wide_of(gd);
    if (gu_wide && dn_wide) {
      pg.out_xs = bufs[1 - in_idx];
      pg.out_f16 = f16;
    }
    LAUNCH(run_gemv(c, g, st, &pg));
    if (pg.out_xs) rd = 1 - in_idx;

    PlaneCfg pd;
    take(pd, dn_wide);
    defer(pd, gd, dn_wide, wide_of(l + 1 == m.n_layers ? head_args() : qkv_args(l + 1)));
    LAUNCH(run_gemv(c, gd, st, &pd));
  }

  GemvArgs g = head_args();
  PlaneCfg ph;
  take(ph, wide_of(g));
  fixup(ph);
  TailArgs& t = g.tail;
  t.mode = mode; t.B = B; t.R = R; t.k = R - 1; t.seq_ids = seq_ids; t.drafts = tokens;
  t.out_tokens = out_tokens; t.n_emitted = n_emitted; t.seq_len = c->state.seq_len;
  t.pending = c->state.pending; t.stats = c->state.stats; t.sel_row = w.sel_row;
  t.best_all = w.best; t.counter = w.counter; t.err = w.err;
  if (parents) {
    t.mode = TAIL_TREE;
    t.parents = parents;
    t.path = w.path;
    t.path_ld = KMAX + 1;
  }
  if (top_m > 0) {
    // lenient accept: every row's logits kept, the accept runs in its own kernel
    if (!g.Y) g.Y = w.lg;
    t.mode = TAIL_NONE;
  }
  LAUNCH(run_gemv(c, g, st, &ph));
  if (top_m > 0) {
    TopmArgs ta = {};
    ta.B = B; ta.k = R - 1; ta.top_m = top_m; ta.V = m.vocab; ta.seq_ids = seq_ids; ta.drafts = tokens;
    ta.logits = g.Y; ta.best = w.best; ta.rank = w.rank; ta.counter = w.rank_cnt; ta.out_tokens = out_tokens;
    ta.n_emitted = n_emitted; ta.seq_len = c->state.seq_len; ta.pending = c->state.pending; ta.sel_row = w.sel_row;
    ta.stats = c->state.stats; ta.err = w.err;
    LAUNCH(topm_accept(ta, st));
  }
  LAUNCH(commit_hidden(B, seq_ids, w.sel_row, w.x, d, c->w.g_final, m.rms_eps, c->state.hid, w.err, st));
  if (parents) {
    TreeMoveArgs tm = {};
    tm.B = B; tm.R = R; tm.L = m.n_layers; tm.nkv = nkv; tm.hd = hd; tm.kv_bytes = m.kv_dtype == SPEC_F32 ? 4 : 2;
    tm.seq_ids = seq_ids; tm.seq_len = c->state.seq_len; tm.n_emitted = n_emitted; tm.path = w.path;
    tm.path_ld = KMAX + 1; tm.pool = c->kv.pool; tm.layer_elems = c->layer_elems;
    tm.max_pages = c->kv.max_pages_per_seq; tm.block_table = c->kv.block_table; tm.n_pages = c->kv.n_pages;
    tm.err = w.err;
    LAUNCH(tree_move(tm, st));
  }
  return n;
}

// ---- the drafter: k autoregressive steps on the target's last hidden state ---
int enqueue_draft(spec_ctx* c, int B, const int32_t* seq_ids, int k, int32_t* drafts, cudaStream_t st) {
  const spec_model_desc& m = c->m;
  const spec_drafter_desc& dd = c->dd;
  const spec_drafter_weights& dw = c->dw;
  const Work& w = c->wk;
  const int d = m.d_model, h = dd.hidden, hd = m.head_dim, dq = dd.n_q_heads * hd, ff = dd.d_ff;
  int n = 0, r;
  for (int j = 1; j <= k; ++j) {
    DraftInArgs di = {};
    di.B = B; di.j = j; di.k = k; di.d = d; di.hd = hd; di.seq_ids = seq_ids;
    di.h_prev = j == 1 ? c->state.hid : w.d_h; di.h_from_state = j == 1;
    di.pending = c->state.pending; di.drafts = drafts; di.seq_len = c->state.seq_len;
    di.embed = M_(c->w.embed); di.g_h = dw.g_in_h; di.g_e = dw.g_in_e; di.eps = m.rms_eps;
    di.theta = m.rope_theta; di.cat = w.d_cat; di.rope_cs = w.d_rope;
    LAUNCH(draft_input(di, st));

    GemvArgs g = {};
    g.X = w.d_cat; g.ldx = 2 * d; g.M = B; g.N = h; g.K = 2 * d; g.W = M_(dw.w_in);
    g.epi = EPI_STORE; g.Y = w.d_u; g.ldy = h; g.pdl = 1;
    LAUNCH(run_gemv(c, g, st));

    for (int l = 0; l < dd.n_layers; ++l) {
      g = GemvArgs{};
      g.X = w.d_u; g.ldx = h; g.M = B; g.N = dq; g.K = h; g.W = mat_layer(M_(dw.wq), l, dq, h);
      g.gain = dw.g_attn + (size_t)l * h; g.eps = m.rms_eps;
      g.epi = EPI_STORE; g.Y = w.d_q; g.ldy = dq; g.pdl = 1;
      LAUNCH(run_gemv(c, g, st));

      AttnArgs at = {};
      at.q = w.d_q; at.ldq = dq; at.B = B; at.R = 1; at.nq = dd.n_q_heads; at.nkv = m.n_kv_heads;
      at.hd = hd; at.key_extra = 0; at.pool = c->kv.pool; at.kv_dtype = kv_dt(c);
      at.layer_elems = c->layer_elems; at.layer = m.n_layers - 1; at.n_pages = c->kv.n_pages;
      at.max_pages = c->kv.max_pages_per_seq; at.block_table = c->kv.block_table; at.seq_ids = seq_ids;
      at.seq_len = c->state.seq_len; at.rope_cs = w.d_rope; at.n_split = c->kv.max_pages_per_seq;
      at.pages_per_split = 1; at.part_o = w.d_part_o; at.part_ml = w.d_part_ml; at.out = w.d_att;
      at.err = w.err;
      LAUNCH(run_attention(c, at, st));

      g = GemvArgs{};
      g.X = w.d_att; g.ldx = dq; g.M = B; g.N = h; g.K = dq; g.W = mat_layer(M_(dw.wo), l, h, dq);
      g.epi = EPI_ADD; g.Y = w.d_u; g.ldy = h; g.pdl = 1;
      LAUNCH(run_gemv(c, g, st));

      g = GemvArgs{};
      g.X = w.d_u; g.ldx = h; g.M = B; g.N = 2 * ff; g.K = h; g.W = mat_layer(M_(dw.wgu), l, 2 * ff, h);
      g.gain = dw.g_ffn + (size_t)l * h; g.eps = m.rms_eps;
      g.epi = EPI_GEGLU; g.geglu_half = ff; g.Y = w.d_act; g.ldy = ff; g.pdl = 1;
      LAUNCH(run_gemv(c, g, st));

      g = GemvArgs{};
      g.X = w.d_act; g.ldx = ff; g.M = B; g.N = h; g.K = ff; g.W = mat_layer(M_(dw.wdown), l, h, ff);
      g.epi = EPI_ADD; g.Y = w.d_u; g.ldy = h; g.pdl = 1;
      LAUNCH(run_gemv(c, g, st));
    }

    // next hidden state h_j = W_out . u
    g = GemvArgs{};
    g.X = w.d_u; g.ldx = h; g.M = B; g.N = d; g.K = h; g.W = M_(dw.w_out);
    g.epi = EPI_STORE; g.Y = w.d_h; g.ldy = d; g.pdl = 1;
    LAUNCH(run_gemv(c, g, st));

    if (!dd.clustered) {
      g = GemvArgs{};
      g.X = w.d_u; g.ldx = h; g.M = B; g.N = m.vocab; g.K = h; g.W = M_(dw.vocab);
      g.gain = dw.g_out; g.eps = m.rms_eps; g.epi = EPI_ARGMAX; g.best = w.d_best; g.pdl = 1;
      TailArgs& t = g.tail;
      t.mode = TAIL_DRAFT; t.B = B; t.R = 1; t.k = k; t.seq_ids = seq_ids; t.draft_out = drafts;
      t.draft_ld = k; t.draft_j = j - 1; t.best_all = w.d_best; t.counter = w.d_counter; t.err = w.err;
      LAUNCH(run_gemv(c, g, st));
    } else {
      g = GemvArgs{};
      g.X = w.d_u; g.ldx = h; g.M = B; g.N = dd.n_centroids; g.K = h; g.W = M_(dw.centroids);
      g.gain = dw.g_out; g.eps = m.rms_eps; g.epi = EPI_STORE; g.Y = w.d_scores; g.ldy = dd.n_centroids;
      g.pdl = 1;
      LAUNCH(run_gemv(c, g, st));
      ClusterArgs ca = {};
      ca.B = B; ca.C = dd.n_centroids; ca.top_c = dd.top_c; ca.cs = m.vocab / dd.n_centroids; ca.h = h;
      ca.scores = w.d_scores; ca.chosen = w.d_chosen; ca.u = w.d_u; ca.g_out = dw.g_out; ca.eps = m.rms_eps;
      ca.vocab = M_(dw.vocab); ca.perm = dw.perm; ca.best = w.d_best;
      ca.tail.mode = TAIL_DRAFT; ca.tail.B = B; ca.tail.draft_out = drafts; ca.tail.draft_ld = k;
      ca.tail.draft_j = j - 1; ca.tail.counter = w.d_counter;
      LAUNCH(cluster_head(ca, st));
    }
  }
  return n;
#undef LAUNCH
}

int run_gemv(spec_ctx* c, GemvArgs g, cudaStream_t st, const PlaneCfg* pc) {
  g.tc_fix = c->wk.tc_fix;
  g.tc_cnt = c->wk.tc_cnt;
  g.wide = c->wk.wide;
  if (pc) {
    if (pc->in_xs) g.wide.xs = pc->in_xs;
    g.wide.ready = pc->ready;
    g.wide.out_xs = pc->out_xs;
    g.wide.out_f16 = pc->out_f16;
    g.wide.defer = pc->defer;
    if (pc->fix.U > 0) {
      g.wide.fix_src = c->wk.wide.fix;
      g.wide.fix_U = pc->fix.U;
      g.wide.fix_grid = pc->fix.grid;
      g.wide.fix_C = pc->fix.C;
      g.wide.fix_T = pc->fix.T;
    }
  }
  if (c->wtrace && c->wtrace_n < WTRACE_LAUNCHES) {
    unsigned long long* slot = c->wtrace + (size_t)(c->wtrace_n++) * num_sms() * 16;
    g.wide.trace = slot;  // whichever projection kernel runs records into the slot
    g.tc_trace = slot;
  }
  g.prefetch = c->prefetch ? 1 : 0;
  return gemv(g, st);
}

// Run `fn` eagerly, or through a cached CUDA graph keyed by `key`.
template <typename F>
spec_status run_graph(spec_ctx* c, const std::string& key, cudaStream_t st, F fn) {
  if (!c->graphs || st == nullptr) {
    const int n = fn(st);
    if (n < 0) return SPEC_ECUDA;
    c->launches += n;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
  }
  std::lock_guard<std::mutex> lk(c->mu);
  auto it = c->cache.find(key);
  if (it == c->cache.end()) {
    cudaGraph_t graph;
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return SPEC_ECUDA;
    const int n = fn(st);
    const cudaError_t e = cudaStreamEndCapture(st, &graph);
    if (n < 0 || e != cudaSuccess) {
      if (e == cudaSuccess) cudaGraphDestroy(graph);
      cudaGetLastError();
      return SPEC_ECUDA;
    }
    cudaGraphExec_t exec;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return SPEC_ECUDA;
    it = c->cache.emplace(key, spec_ctx::Entry{exec, n}).first;
  }
  if (cudaGraphLaunch(it->second.exec, st) != cudaSuccess) return SPEC_ECUDA;
  c->launches += it->second.kernels;
  return SPEC_OK;
}

std::string key_of(const char* op, std::initializer_list<long long> v) {
  std::string s(op);
  char buf[32];
  for (long long x : v) {
    snprintf(buf, sizeof buf, ":%llx", x);
    s += buf;
  }
  return s;
}

bool batch_ok(const spec_ctx* c, int B, const int32_t* seq_ids) {
  return c && B > 0 && B <= c->B_max && seq_ids;
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(const spec_model_desc* m, const spec_drafter_desc* d, int32_t B_max, int32_t rows_max,
                            int32_t max_pages_per_seq) {
  if (!m || !model_ok(*m) || B_max <= 0 || rows_max <= 0 || max_pages_per_seq <= 0) return 0;
  if (d && !drafter_ok(*m, *d)) return 0;
  return carve(nullptr, *m, d, B_max, rows_max, max_pages_per_seq).bytes;
}

spec_status spec_init(const spec_model_desc* model, const spec_weights* weights, const spec_drafter_desc* drafter,
                      const spec_drafter_weights* dweights, const spec_kv_desc* kv, const spec_state* state,
                      int32_t B_max, int32_t rows_max, void* workspace, size_t ws_bytes, void* stream,
                      spec_ctx** out) {
  if (!out || !model || !weights || !kv || !state || !workspace) return SPEC_EINVAL;
  *out = nullptr;
  const spec_model_desc& m = *model;
  if (!model_ok(m)) return SPEC_EINVAL;
  if (B_max <= 0 || rows_max <= 0) return SPEC_EINVAL;
  if (kv->page_size != 64 || !kv->pool || !kv->block_table || kv->n_pages <= 0 || kv->max_pages_per_seq <= 0 ||
      kv->n_slots < B_max)
    return SPEC_EINVAL;
  if (!state->seq_len || !state->pending || !state->hid || !state->stats) return SPEC_EINVAL;
  const int nqkv = (m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim, qd = m.n_q_heads * m.head_dim;
  const spec_weights& w = *weights;
  if (!mat_ok(w.embed, m.d_model) || !mat_ok(w.wqkv, m.d_model) || !mat_ok(w.wo, qd) || !w.g_attn || !w.g_ffn ||
      !w.g_final)
    return SPEC_EINVAL;
  if (m.n_experts == 0 && (!mat_ok(w.wgu, m.d_model) || !mat_ok(w.wdown, m.d_ff))) return SPEC_EINVAL;
  if (m.n_experts > 0 && (!mat_ok(w.router, m.d_model) || !mat_ok(w.wgu_e, m.d_model) ||
                          !mat_ok(w.wdown_e, m.d_ff_expert) || w.router.dtype != m.w_dtype ||
                          w.wgu_e.dtype != m.w_dtype || w.wdown_e.dtype != m.w_dtype))
    return SPEC_EINVAL;
  for (const spec_matrix* mm : {&w.embed, &w.wqkv, &w.wo})
    if (mm->dtype != m.w_dtype) return SPEC_EINVAL;
  (void)nqkv;
  const int G = m.n_q_heads / m.n_kv_heads;
  if (G > 128 || attention_smem(m.head_dim, pass_rows(m, rows_max) * G) > 200 * 1024) return SPEC_EUNSUPPORTED;
  if (drafter) {
    if (!dweights || !drafter_ok(m, *drafter)) return SPEC_EINVAL;
    const spec_drafter_weights& dw = *dweights;
    const int h = drafter->hidden, dq = drafter->n_q_heads * m.head_dim;
    if (!mat_ok(dw.w_in, 2 * m.d_model) || !mat_ok(dw.wq, h) || !mat_ok(dw.wo, dq) || !mat_ok(dw.wgu, h) ||
        !mat_ok(dw.wdown, drafter->d_ff) || !mat_ok(dw.w_out, h) || !mat_ok(dw.vocab, h) || !dw.g_in_h ||
        !dw.g_in_e || !dw.g_attn || !dw.g_ffn || !dw.g_out)
      return SPEC_EINVAL;
    if (drafter->clustered && (!mat_ok(dw.centroids, h) || !dw.perm)) return SPEC_EINVAL;
    if (attention_smem(m.head_dim, drafter->n_q_heads / m.n_kv_heads) > 200 * 1024) return SPEC_EUNSUPPORTED;
  }
  const Work need = carve(nullptr, m, drafter, B_max, rows_max, kv->max_pages_per_seq);
  if (ws_bytes < need.bytes) return SPEC_ECAPACITY;

  spec_ctx* c = new spec_ctx();
  c->m = m;
  c->w = w;
  c->has_drafter = drafter != nullptr;
  if (drafter) {
    c->dd = *drafter;
    c->dw = *dweights;
  }
  c->kv = *kv;
  c->state = *state;
  c->B_max = B_max;
  c->rows_max = rows_max;
  c->pass_rows = pass_rows(m, rows_max);
  c->layer_elems = (long long)kv->n_pages * 2 * m.n_kv_heads * 64 * m.head_dim;
  c->wk = carve((char*)workspace, m, drafter, B_max, rows_max, kv->max_pages_per_seq);
  setup_device_attributes();
  // RoPE and the KV append run in the QKV projection's epilogue when that
  // projection is the tensor-core kernel (bf16 or Q4_0) writing a bf16 cache
  c->fused_rope = ((m.w_dtype == SPEC_BF16 && m.d_model % 32 == 0) ||
                   (m.w_dtype == SPEC_Q4_0 && m.d_model % 128 == 0)) &&
                  m.kv_dtype == SPEC_BF16 && m.head_dim % 16 == 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, need.bytes, st) != cudaSuccess) {
    delete c;
    return SPEC_ECUDA;
  }
  *out = c;
  return SPEC_OK;
}

spec_status spec_prefill(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t R, const int32_t* tokens,
                         void* stream) {
  if (!batch_ok(c, B, seq_ids) || R <= 0 || R > c->rows_max || !tokens) return SPEC_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  // passes of at most pass_rows rows; each commits its rows, so the next one's
  // rows attend to them as cached keys
  return run_graph(c, key_of("prefill", {B, R, (long long)seq_ids, (long long)tokens, (long long)st}), st,
                   [&](cudaStream_t s) {
                     int n = 0;
                     for (int r0 = 0; r0 < R; r0 += c->pass_rows) {
                       const int r = std::min(c->pass_rows, R - r0);
                       const int k = enqueue_pass(c, B, seq_ids, r, TAIL_PREFILL, tokens + r0, nullptr, nullptr,
                                                  nullptr, s, 0, R);
                       if (k < 0) return -1;
                       n += k;
                     }
                     return n;
                   });
}

spec_status spec_verify(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t k, const int32_t* drafts,
                        int32_t* out_tokens, int32_t* n_emitted, float* logits_dbg, void* stream) {
  if (!batch_ok(c, B, seq_ids) || k < 0 || k > KMAX || k + 1 > c->pass_rows || !out_tokens || !n_emitted ||
      (k > 0 && !drafts))
    return SPEC_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  return run_graph(c,
                   key_of("verify", {B, k, (long long)seq_ids, (long long)drafts, (long long)out_tokens,
                                     (long long)n_emitted, (long long)logits_dbg, (long long)st}),
                   st, [&](cudaStream_t s) {
                     return enqueue_pass(c, B, seq_ids, k + 1, TAIL_VERIFY, drafts, out_tokens, n_emitted,
                                         logits_dbg, s);
                   });
}

spec_status spec_verify_topm(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t k, const int32_t* drafts,
                             int32_t top_m, int32_t* out_tokens, int32_t* n_emitted, float* logits_dbg,
                             void* stream) {
  if (!batch_ok(c, B, seq_ids) || k < 1 || k > KMAX || k + 1 > c->pass_rows || !out_tokens || !n_emitted ||
      !drafts || top_m < 1)
    return SPEC_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  return run_graph(c,
                   key_of("verify_topm", {B, k, top_m, (long long)seq_ids, (long long)drafts, (long long)out_tokens,
                                          (long long)n_emitted, (long long)logits_dbg, (long long)st}),
                   st, [&](cudaStream_t s) {
                     return enqueue_pass(c, B, seq_ids, k + 1, TAIL_VERIFY, drafts, out_tokens, n_emitted,
                                         logits_dbg, s, top_m);
                   });
}

spec_status spec_verify_tree(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t n, const int32_t* tokens,
                             const int32_t* parents, int32_t* out_tokens, int32_t* n_emitted, float* logits_dbg,
                             void* stream) {
  if (!batch_ok(c, B, seq_ids) || n < 1 || n > KMAX || n + 1 > c->pass_rows || !tokens || !parents || !out_tokens ||
      !n_emitted)
    return SPEC_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  return run_graph(c,
                   key_of("verify_tree", {B, n, (long long)seq_ids, (long long)tokens, (long long)parents,
                                          (long long)out_tokens, (long long)n_emitted, (long long)logits_dbg,
                                          (long long)st}),
                   st, [&](cudaStream_t s) {
                     return enqueue_pass(c, B, seq_ids, n + 1, TAIL_VERIFY, tokens, out_tokens, n_emitted,
                                         logits_dbg, s, 0, 0, parents);
                   });
}

spec_status spec_draft(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t k, int32_t* drafts, void* stream) {
  if (!batch_ok(c, B, seq_ids) || k <= 0 || k > KMAX || !drafts) return SPEC_EINVAL;
  if (!c->has_drafter) return SPEC_ESTATE;
  cudaStream_t st = (cudaStream_t)stream;
  return run_graph(c, key_of("draft", {B, k, (long long)seq_ids, (long long)drafts, (long long)st}), st,
                   [&](cudaStream_t s) { return enqueue_draft(c, B, seq_ids, k, drafts, s); });
}

spec_status spec_step(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t k, int32_t* out_tokens,
                      int32_t* n_emitted, void* stream) {
  if (!batch_ok(c, B, seq_ids)) return SPEC_EINVAL;
  spec_status s = spec_draft(c, B, seq_ids, k, c->wk.d_drafts, stream);
  if (s != SPEC_OK) return s;
  return spec_verify(c, B, seq_ids, k, c->wk.d_drafts, out_tokens, n_emitted, nullptr, stream);
}

spec_status spec_decode(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t* out_tok, void* stream) {
  if (!batch_ok(c, B, seq_ids) || !out_tok) return SPEC_EINVAL;
  // n_emitted is always 1 for k = 0; it lands in a workspace buffer
  return spec_verify(c, B, seq_ids, 0, nullptr, out_tok, c->wk.n_emit1, nullptr, stream);
}

spec_status spec_inject_drafts(spec_ctx* c, int32_t B, const int32_t* seq_ids, int32_t k, int32_t* drafts,
                               const int32_t* ref, int32_t ref_len, float alpha, const float* draws,
                               const int32_t* offsets, void* stream) {
  if (!batch_ok(c, B, seq_ids) || k <= 0 || k > KMAX || !drafts || !ref || ref_len <= 0 || !draws || !offsets)
    return SPEC_EINVAL;
  const int n = inject_drafts(B, k, seq_ids, c->state.seq_len, drafts, ref, ref_len, alpha, draws, offsets,
                              c->m.vocab, c->wk.err, (cudaStream_t)stream);
  if (n < 0) return SPEC_ECUDA;
  c->launches += n;
  return SPEC_OK;
}

size_t spec_linear_workspace_bytes(int32_t N, int32_t K, int32_t M) {
  if (N <= 0 || K <= 0 || M <= 0) return 0;
  size_t n = gemv_tc_fixup_bytes() + (((size_t)N / 8 + 64) * sizeof(unsigned int) + 255) / 256 * 256 + 256;
  if (M > 8 || ((long long)N * K >= WIDE_MIN_ELEMS && K >= WIDE_MIN_K))
    n += gemv_wide_fix_bytes() + gemv_wide_xs_bytes(K) + 64 * 16 * sizeof(float) + 3 * 256;
  return n;
}

spec_status spec_linear(const spec_matrix* w, int32_t N, int32_t K, const float* x, int32_t M, const float* gain,
                        float eps, float* y, void* workspace, size_t ws_bytes, void* stream) {
  if (!w || !x || !y || N <= 0 || K <= 0 || M <= 0 || M > 64 || !mat_ok(*w, K)) return SPEC_EINVAL;
  if (!workspace || ws_bytes < spec_linear_workspace_bytes(N, K, M)) return SPEC_ECAPACITY;
  GemvArgs g = {};
  g.X = x; g.ldx = K; g.M = M; g.N = N; g.K = K; g.W = M_(*w); g.gain = gain; g.eps = eps;
  g.epi = EPI_STORE; g.Y = y; g.ldy = N; g.pdl = 0; g.prefetch = 0;
  g.tc_fix = (float*)workspace;
  g.tc_cnt = (unsigned int*)((char*)workspace + gemv_tc_fixup_bytes());
  if (M > 8 || ((long long)N * K >= WIDE_MIN_ELEMS && K >= WIDE_MIN_K)) {
    char* p = (char*)workspace + gemv_tc_fixup_bytes() +
              (((size_t)N / 8 + 64) * sizeof(unsigned int) + 255) / 256 * 256 + 256;
    g.wide.fix = (float*)p;
    p += (gemv_wide_fix_bytes() + 255) / 256 * 256;
    g.wide.xs = (uint16_t*)p;
    p += (gemv_wide_xs_bytes(K) + 255) / 256 * 256;
    g.wide.rms = (float*)p;
    g.wide.kmax = K;
  }
  setup_device_attributes();
  if (gemv(g, (cudaStream_t)stream) < 0) return SPEC_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

size_t spec_attention_workspace_bytes(const spec_model_desc* m, int32_t B, int32_t R, int32_t n_q_heads,
                                      int32_t max_pages_per_seq) {
  if (!m || !model_ok(*m) || B <= 0 || R <= 0 || n_q_heads <= 0 || n_q_heads % m->n_kv_heads ||
      max_pages_per_seq <= 0)
    return 0;
  return carve_attention(nullptr, B, R, n_q_heads, m->n_kv_heads, m->head_dim, max_pages_per_seq).bytes;
}

spec_status spec_attention(const spec_model_desc* m, const spec_kv_desc* kv, int32_t layer, int32_t B,
                           const int32_t* seq_ids, const int32_t* seq_len, int32_t R, int32_t n_q_heads,
                           int32_t key_extra, const float* q, float* out, void* workspace, size_t ws_bytes,
                           void* stream) {
  if (!m || !model_ok(*m) || !kv || !kv->pool || !kv->block_table || kv->page_size != 64 || kv->n_pages <= 0 ||
      kv->max_pages_per_seq <= 0 || layer < 0 || layer >= m->n_layers || B <= 0 || B > 64 || !seq_ids ||
      !seq_len || R <= 0 || R > 64 || n_q_heads <= 0 || n_q_heads % m->n_kv_heads || (key_extra != 0 && key_extra != 1) ||
      !q || !out || !workspace)
    return SPEC_EINVAL;
  if (R * (n_q_heads / m->n_kv_heads) > 128) return SPEC_EUNSUPPORTED;
  const AttnWork w = carve_attention((char*)workspace, B, R, n_q_heads, m->n_kv_heads, m->head_dim,
                                     kv->max_pages_per_seq);
  if (ws_bytes < w.bytes) return SPEC_ECAPACITY;
  AttnArgs at = {};
  at.q = q; at.ldq = n_q_heads * m->head_dim; at.B = B; at.R = R; at.nq = n_q_heads; at.nkv = m->n_kv_heads;
  at.hd = m->head_dim; at.key_extra = key_extra; at.pool = kv->pool;
  at.kv_dtype = m->kv_dtype == SPEC_F32 ? DT_F32 : DT_BF16;
  at.layer_elems = (long long)kv->n_pages * 2 * m->n_kv_heads * 64 * m->head_dim;
  at.layer = layer; at.n_pages = kv->n_pages; at.max_pages = kv->max_pages_per_seq;
  at.block_table = kv->block_table; at.seq_ids = seq_ids; at.seq_len = seq_len; at.rope_cs = nullptr;
  at.n_split = kv->max_pages_per_seq; at.pages_per_split = 1; at.part_o = w.part_o; at.part_ml = w.part_ml;
  at.out = out; at.err = w.err; at.standalone = 1;
  setup_device_attributes();
  if (launch_attention(m->kv_dtype, at, w.counters, 0, (cudaStream_t)stream) < 0) return SPEC_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

spec_status spec_stats(spec_ctx* c, int32_t slot, spec_stats_t* out, void* stream) {
  if (!c || !out || slot < 0 || slot >= c->kv.n_slots) return SPEC_EINVAL;
  int64_t v[4];
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(v, c->state.stats + (size_t)slot * 4, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SPEC_ECUDA;
  out->passes = v[0];
  out->drafted = v[1];
  out->accepted = v[2];
  out->emitted = v[3];
  out->tokens_per_pass = v[0] ? (double)v[3] / (double)v[0] : 0.0;
  return SPEC_OK;
}

spec_status spec_sync(spec_ctx* c, void* stream) {
  if (!c) return SPEC_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ECUDA;
  int err = 0;
  if (cudaMemcpy(&err, c->wk.err, sizeof err, cudaMemcpyDeviceToHost) != cudaSuccess) return SPEC_ECUDA;
  if (err) {
    if (cudaMemset(c->wk.err, 0, sizeof(int)) != cudaSuccess) return SPEC_ECUDA;
    if (err == SPEC_ERR_TIMEOUT) return SPEC_ETIMEOUT;
    return err == SPEC_ERR_CAPACITY ? SPEC_ECAPACITY : SPEC_EINVAL;
  }
  return SPEC_OK;
}

spec_status spec_set_graphs(spec_ctx* c, int32_t enable) {
  if (!c) return SPEC_EINVAL;
  c->graphs = enable != 0;
  return SPEC_OK;
}

spec_status spec_set_option(spec_ctx* c, int32_t option, int64_t value) {
  if (!c) return SPEC_EINVAL;
  std::lock_guard<std::mutex> lk(c->mu);
  if (option == SPEC_OPT_GRAPHS) c->graphs = value != 0;
  else if (option == SPEC_OPT_PREFETCH) c->prefetch = value != 0;
  else if (option == SPEC_OPT_TEST_ATTN_WAIT) c->test_attn_wait = value > 0 ? 1 : 0;
  else if (option == SPEC_OPT_WIDE_TRACE) {
    c->wtrace = (unsigned long long*)(uintptr_t)value;
    c->wtrace_n = 0;
  }
  else return SPEC_EINVAL;
  for (auto& kv : c->cache) cudaGraphExecDestroy(kv.second.exec);
  c->cache.clear();
  return SPEC_OK;
}

int64_t spec_kernel_launches(const spec_ctx* c) { return c ? c->launches : 0; }

const char* spec_status_str(spec_status s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument";
    case SPEC_ECAPACITY: return "capacity exceeded";
    case SPEC_ESTATE: return "invalid state";
    case SPEC_ECUDA: return "CUDA error";
    case SPEC_ETIMEOUT: return "device wait timed out";
    case SPEC_EUNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

void spec_destroy(spec_ctx* c) {
  if (!c) return;
  for (auto& kv : c->cache) cudaGraphExecDestroy(kv.second.exec);
  delete c;
}

}  // extern "C"
