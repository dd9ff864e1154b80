// draft_cluster.cu -- all k drafter steps in one launch: one thread-block
// cluster per sequence.
//
// The drafter is a light head on the target's last layer: from the target's
// final hidden state it predicts the next tokens one after another
// ("Accelerating Gemini Nano on Pixel with frozen multi-token prediction"
// (ai-news-spoon), section "The late-exit strategy"), cross-attends the
// target's KV cache in place ("Zero-copy architecture"), and scores its output
// through 2048 centroids ("Gemma 4's MTP drafter explained" (molayo1419.me),
// section "What is different about Gemma 4's drafter?"). For one sequence, a
// step j is a chain of small dependent operations:
//   u   = W_in . [N(h_{j-1}) ; N(E[tok_{j-1}])]
//   per layer: u += Wo' . CrossAttn(RoPE(Wq' . N(u)), target last-layer K/V[0, seq_len))
//              u += Wd' . (GELU(Wg' . N(u)) * (Wu' . N(u)))
//   h_j = W_out . u ;  tok_j = clustered (or full) head of N_out(u)
// with the query at position seq_len + j - 1.
//
// Run as separate kernels, launch and ramp latency dominate (a few MB of
// weights per operation). Here the CTAs of one cluster (16 when the GPU allows,
// else 8) walk the chain together:
//  - every weight matrix is split by output rows across the CTAs; each CTA
//    streams its rows through a ring of shared-memory slots with bulk async
//    copies (cp.async.bulk + mbarrier). The copies run ahead of the
//    computation across operation boundaries: weights do not depend on
//    activations, so thread 0 refills the ring with the next operations' rows
//    between its arrival at a cluster barrier and the wait for the others;
//  - each warp reduces 32 rows at once: every lane accumulates its 8-element
//    slice of 32 dot products, and a transposing butterfly (31 shuffles)
//    leaves lane i with row i's sum;
//  - activation vectors are pushed into every CTA's shared memory with
//    distributed-shared-memory stores (st.shared::cluster), and a hardware
//    cluster barrier separates dependent operations;
//  - the cross-attention reads the target's last-layer pages in place with the
//    target's tensor-core paged attention: the CTAs of the cluster are
//    (kv head, page split) pairs and the last split of each kv head merges
//    (bf16 caches; an fp32 cache takes a CUDA-core path, one warp per
//    (kv head, page range)). The attention works in the ring's shared memory,
//    so the ring is drained before it and refilled after it.
// Dot products and reductions run in fp32 in a fixed order, so the drafts do
// not depend on timing. Every wait on an mbarrier is bounded: on a timeout the
// CTA sets the error word, stops computing and still passes every cluster
// barrier, so no CTA is left waiting.
#include <math.h>

#include <algorithm>
#include <type_traits>

#include "attn_tc.cuh"
#include "common.cuh"
#include "mbar.cuh"

#define SPEC_HD __host__ __device__ __forceinline__

namespace spec {

namespace {

constexpr int DW = 16;            // warps per CTA
constexpr int NTH = DW * 32;
constexpr int SLOT = 16384;       // bytes per ring slot
constexpr int NS_MAX = 16;        // ring slots
constexpr int GMAX = 8;           // q heads per kv head
constexpr int PAGE = 64;
constexpr int MAXSEG = 8;         // row segments of one operation in one CTA
constexpr int MAXC = 16;          // CTAs per cluster
constexpr int TOPC_MAX = 256;
constexpr unsigned SPIN_LIMIT = 1u << 26;

enum { PH_WIN, PH_WQ, PH_WO, PH_WGU, PH_WDOWN, PH_WOUT, PH_HEAD, PH_MEMB };

// ---- cluster primitives (mbarrier and bulk copies in mbar.cuh) -----------

SPEC_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
SPEC_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
SPEC_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
SPEC_DEV unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
SPEC_DEV unsigned cluster_ctas() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
SPEC_DEV uint32_t remote(const void* p, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(sa(p)), "r"(rank));
  return r;
}
SPEC_DEV void st_remote(const float* p, unsigned rank, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote(p, rank)), "f"(v) : "memory");
}
SPEC_DEV void st_remote4(const float* p, unsigned rank, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote(p, rank)), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
SPEC_DEV void st_remote_u64(const unsigned long long* p, unsigned rank, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote(p, rank)), "l"(v) : "memory");
}
// Bounded wait on an mbarrier phase; on a timeout the CTA aborts.
SPEC_DEV bool wait_phase(uint64_t* b, unsigned parity, volatile int* abort_s, int* err) {
  for (unsigned it = 0; it < SPIN_LIMIT; ++it) {
    if (mbar_test(b, parity)) return true;
    if (*abort_s) return false;
  }
  *abort_s = 1;
  set_error(err, SPEC_ERR_TIMEOUT);
  return false;
}

// ---- operations and their row chunks --------------------------------------

constexpr int MAX_OPS = 3 + 4 * 16 + 1;  // at most 16 drafter layers
constexpr int MAX_CH = 384;              // weight chunks of one step per CTA, members excluded
constexpr int MAX_MCH = 64;              // member chunks of one step per CTA

SPEC_HD int imin(int a, int b) { return a < b ? a : b; }

// One weight operation as seen by one CTA: its matrix, the logical outputs
// [o0, o0 + no) it computes, its local rows (2 * no for the gate/up pair),
// pieces per row and its chunks [c0, c0 + nc) in the step's table.
struct OpI {
  const void* data;
  const void* scales;
  int K, type, o0, no, rows, nkp, c0, nc;
};
// One chunk: matrix rows [row, row + nr) (local rows from lrow) and the k
// range [ka, ka + kw) of operation `op`.
struct ChE {
  int row, lrow, nr, ka, kw, op;
};

SPEC_HD int n_ops(int L, int clustered) { return 3 + 4 * L + (clustered ? 1 : 0); }

// Operation ph of a draft step (0: W_in; 1 + 4l + {0..3}: Wq, Wo, Wgu, Wdown
// of layer l; 1 + 4L: W_out; 2 + 4L: head; 3 + 4L: cluster members): its
// type, reduction width K and logical output count N.
SPEC_HD void op_dims(int ph, int L, int d, int h, int dq, int ff, int C, int V, int members, int clustered,
                     int& type, int& K, int& N) {
  if (ph == 0) { type = PH_WIN; K = 2 * d; N = h; }
  else if (ph <= 4 * L) {
    const int s = (ph - 1) & 3;
    if (s == 0) { type = PH_WQ; K = h; N = dq; }
    else if (s == 1) { type = PH_WO; K = dq; N = h; }
    else if (s == 2) { type = PH_WGU; K = h; N = ff; }
    else { type = PH_WDOWN; K = ff; N = h; }
  } else if (ph == 4 * L + 1) { type = PH_WOUT; K = h; N = d; }
  else if (ph == 4 * L + 2) { type = PH_HEAD; K = h; N = clustered ? C : V; }
  else { type = PH_MEMB; K = h; N = members; }
}

SPEC_DEV Mat op_matrix(const DraftDesc& D, int ph, int type) {
  const int h = D.h, dq = D.dnq * D.hd, l = ph >= 1 ? (ph - 1) >> 2 : 0;
  switch (type) {
    case PH_WIN: return D.w_in;
    case PH_WQ: return mat_layer(D.wq, l, dq, h);
    case PH_WO: return mat_layer(D.wo, l, h, dq);
    case PH_WGU: return mat_layer(D.wgu, l, 2 * D.ff, h);
    case PH_WDOWN: return mat_layer(D.wdown, l, h, D.ff);
    case PH_WOUT: return D.w_out;
    case PH_HEAD: return D.clustered ? D.centroids : D.vocab;
    default: return D.vocab;
  }
}

// Chunk geometry: k-width (the whole row when a row fits a slot) and rows per chunk.
struct Geo {
  int kw, rpc;
};
SPEC_HD Geo geometry(int K, int wt) {
  const int eb16 = wt == DT_F32 ? 64 : wt == DT_BF16 ? 32 : 9;  // bytes per 16 elements
  Geo g;
  if ((long long)K * eb16 <= (long long)SLOT * 16) g.kw = K;
  else g.kw = ((SLOT * 16 / eb16) / 256) * 256;
  const long long rb = (long long)g.kw * eb16 / 16;
  g.rpc = (int)(SLOT / rb);
  if (g.rpc < 1) g.rpc = 1;
  return g;
}
// Elements per dot-product piece: the largest of 256/128/64/32 dividing K.
SPEC_HD int piece_of(int K) {
  for (int p = 256; p >= 32; p >>= 1)
    if (K % p == 0) return p;
  return 0;
}

// Append (or, with t == nullptr, count) the chunks of matrix rows
// [row0, row0 + n), local rows from lrow.
SPEC_HD int add_chunks(ChE* t, int nt, int cap, int op, int row0, int lrow, int n, int K, Geo g) {
  for (int r = 0; r < n; r += g.rpc)
    for (int ka = 0; ka < K; ka += g.kw) {
      if (t && nt < cap) t[nt] = ChE{row0 + r, lrow + r, imin(g.rpc, n - r), ka, imin(g.kw, K - ka), op};
      ++nt;
    }
  return nt;
}

// The operation table and the chunks of every operation but the members
// (thread 0, once per launch). Returns the chunk count.
template <int WT>
SPEC_DEV int build_tables(const DraftDesc& D, unsigned rank, unsigned ncta, OpI* ops, ChE* ch) {
  int nt = 0;
  const int nop = n_ops(D.L, D.clustered), dq = D.dnq * D.hd;
  for (int ph = 0; ph < nop; ++ph) {
    int type, K, N;
    op_dims(ph, D.L, D.d, D.h, dq, D.ff, D.C, D.V, D.top_c * D.cs, D.clustered, type, K, N);
    const Mat W = op_matrix(D, ph, type);
    OpI o;
    o.data = W.data;
    o.scales = W.scales;
    o.K = K;
    o.type = type;
    o.o0 = (int)((long long)N * rank / ncta);
    o.no = (int)((long long)N * (rank + 1) / ncta) - o.o0;
    o.rows = type == PH_WGU ? 2 * o.no : o.no;
    o.nkp = K / piece_of(K);
    o.c0 = nt;
    if (type != PH_MEMB) {
      const Geo g = geometry(K, WT);
      nt = add_chunks(ch, nt, MAX_CH, ph, o.o0, 0, o.no, K, g);
      if (type == PH_WGU) nt = add_chunks(ch, nt, MAX_CH, ph, D.ff + o.o0, o.no, o.no, K, g);
    }
    o.nc = nt - o.c0;
    ops[ph] = o;
  }
  return nt;
}

// The member chunks of the kept clusters (thread 0, each step after the
// selection): member m of the kept clusters (in increasing cluster id) is row
// chosen[m / cs] * cs + m % cs of the cluster-sorted vocabulary.
template <int WT>
SPEC_DEV int build_members(const DraftDesc& D, const OpI& o, int ph, const int* chosen, ChE* mch, int* seg_row,
                           int* seg_lrow, int* nseg) {
  const Geo g = geometry(o.K, WT);
  int nt = 0, n = 0;
  for (int m = o.o0; m < o.o0 + o.no;) {
    const int c = m / D.cs, e = min(o.o0 + o.no, (c + 1) * D.cs);
    const int row0 = chosen[c] * D.cs + (m - c * D.cs);
    if (n < MAXSEG) {
      seg_row[n] = row0;
      seg_lrow[n] = m - o.o0;
    }
    ++n;
    nt = add_chunks(mch, nt, MAX_MCH, ph, row0, m - o.o0, e - m, o.K, g);
    m = e;
  }
  *nseg = n;
  return nt;
}

// ---- the ring filler (thread 0 of each CTA) --------------------------------

// Chunk stream position: step j, position in the step's stream (the table's
// chunks, then the members').
struct Filler {
  int j, pos;
  int issued;        // chunks issued so far
  int slot;          // ring slot of the next chunk (issued % ns)
  bool done;
};

// The tables both the filler and the consumers read (shared memory).
struct Tabs {
  const OpI* ops;
  const ChE* ch;
  const ChE* mch;
  int nch;
  const int* nm;        // member chunks of step *sel_step
  const int* sel_step;  // last step whose clusters are chosen
  const int* att_done;  // attentions finished in this launch (nullptr: no gate)
  int L;
};

// Attentions that must be finished before operation ph of step j may take
// ring slots (the attention of layer l uses the ring's shared memory between
// Wq of layer l and Wo of layer l).
SPEC_DEV int att_needed(int ph, int j, int L) {
  int n = ph >= 2 ? (ph - 2) / 4 + 1 : 0;
  n = n > L ? L : n;
  return (j - 1) * L + n;
}

template <int WT>
SPEC_DEV void issue_chunk(const OpI& P, const ChE& c, unsigned char* slot, uint64_t* full) {
  const int K = P.K;
  if (WT != DT_Q4_0) {
    const int eb = WT == DT_F32 ? 4 : 2;
    const char* src = (const char*)P.data + ((size_t)c.row * K + c.ka) * eb;
    const unsigned rb = (unsigned)c.kw * eb;
    mbar_expect_tx(full, rb * c.nr);
    if (c.kw == K) {
      bulk_load(slot, src, rb * c.nr, full);
    } else {
      for (int i = 0; i < c.nr; ++i) bulk_load(slot + (size_t)i * rb, src + (size_t)i * K * eb, rb, full);
    }
  } else {
    const char* codes = (const char*)P.data + (size_t)c.row * (K / 2) + c.ka / 2;
    const char* scales = (const char*)P.scales + ((size_t)c.row * (K / 32) + c.ka / 32) * 2;
    const unsigned cb = (unsigned)c.kw / 2, sb = (unsigned)c.kw / 16;
    mbar_expect_tx(full, (cb + sb) * c.nr);
    unsigned char* sdst = slot + (size_t)c.nr * cb;
    if (c.kw == K) {
      bulk_load(slot, codes, cb * c.nr, full);
      bulk_load(sdst, scales, sb * c.nr, full);
    } else {
      for (int i = 0; i < c.nr; ++i) {
        bulk_load(slot + (size_t)i * cb, codes + (size_t)i * (K / 2), cb, full);
        bulk_load(sdst + (size_t)i * sb, scales + (size_t)i * (K / 16), sb, full);
      }
    }
  }
}

// Issue chunks into free slots until the ring holds `ns` chunks past the
// `consumed` ones, the stream ends, or the next chunk is a member row of a step
// whose clusters are not chosen yet. Called only where every warp of the CTA
// is done with the consumed chunks (after a CTA barrier), so their slots are
// free without a per-slot release barrier.
template <int WT>
SPEC_DEV void fill(const DraftDesc& D, Filler& F, int consumed, const Tabs& T, unsigned char* ring,
                   uint64_t* full, volatile int* abort_s) {
  while (!F.done && !*abort_s && F.issued < consumed + D.ns) {
    const ChE* e = nullptr;
    if (F.pos < T.nch) {
      e = &T.ch[F.pos];
    } else if (D.clustered) {
      if (*T.sel_step < F.j) return;
      if (F.pos - T.nch < *T.nm) e = &T.mch[F.pos - T.nch];
    }
    if (!e) {
      F.pos = 0;
      if (++F.j > D.k) F.done = true;
      continue;
    }
    if (T.att_done && *T.att_done < att_needed(e->op, F.j, T.L)) return;
    issue_chunk<WT>(T.ops[e->op], *e, ring + (size_t)F.slot * SLOT, &full[F.slot]);
    ++F.issued;
    if (++F.slot == D.ns) F.slot = 0;
    ++F.pos;
  }
}

// ---- dot products of one chunk ---------------------------------------------

struct Chunk {
  long long row;   // first matrix row
  int lrow, nr;    // first local row, rows
  int ka, kw;      // k range [ka, ka + kw)
};

template <int WT>
SPEC_DEV void weights8(const unsigned char* slot, int kw, int nr, int r, int e0, float* w) {
  if (WT == DT_BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(slot + ((size_t)r * kw + e0) * 2);
    w[0] = bf16lo(v.x); w[1] = bf16hi(v.x); w[2] = bf16lo(v.y); w[3] = bf16hi(v.y);
    w[4] = bf16lo(v.z); w[5] = bf16hi(v.z); w[6] = bf16lo(v.w); w[7] = bf16hi(v.w);
  } else if (WT == DT_F32) {
    const float4 a = *reinterpret_cast<const float4*>(slot + ((size_t)r * kw + e0) * 4);
    const float4 b = *reinterpret_cast<const float4*>(slot + ((size_t)r * kw + e0) * 4 + 16);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else {
    // elements 8q .. 8q+7 of a 32-value block: bytes 8(q&1) .. +7, low nibble
    // for q < 2, high nibble for q >= 2
    const int blk = e0 >> 5, q = (e0 & 31) >> 3;
    const uint2 raw = *reinterpret_cast<const uint2*>(slot + (size_t)r * (kw / 2) + blk * 16 + 8 * (q & 1));
    const float s = __half2float(*reinterpret_cast<const __half*>(slot + (size_t)nr * (kw / 2) +
                                                                 (size_t)r * (kw / 16) + blk * 2));
    const uint32_t wv[2] = {raw.x, raw.y};
    const int sh = q < 2 ? 0 : 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = s * (float)((int)((wv[i >> 2] >> (8 * (i & 3) + sh)) & 15u) - 8);
  }
}

// part[lrow * nkp + k / KP] = dot(row piece, x piece) for every piece of the chunk.
template <int WT>
SPEC_DEV void dot_chunk(const unsigned char* slot, const Chunk& c, const float* x, int KP, int nkp, float* part,
                        int warp, int lane) {
  const int LP = KP / 8, PPW = 32 / LP;
  const int npk = c.kw / KP, np = c.nr * npk;
  const int sub = lane % LP, pi = lane / LP;
  for (int p0 = warp * PPW; p0 < np; p0 += DW * PPW) {
    const int p = p0 + pi;
    float acc = 0.f;
    int r = 0, kp = 0;
    if (p < np) {
      r = p / npk;
      kp = p - r * npk;
      const int e0 = kp * KP + sub * 8;
      float w[8];
      weights8<WT>(slot, c.kw, c.nr, r, e0, w);
      const float4 x0 = *reinterpret_cast<const float4*>(x + c.ka + e0);
      const float4 x1 = *reinterpret_cast<const float4*>(x + c.ka + e0 + 4);
      acc = w[0] * x0.x;
      acc = fmaf(w[1], x0.y, acc); acc = fmaf(w[2], x0.z, acc); acc = fmaf(w[3], x0.w, acc);
      acc = fmaf(w[4], x1.x, acc); acc = fmaf(w[5], x1.y, acc); acc = fmaf(w[6], x1.z, acc);
      acc = fmaf(w[7], x1.w, acc);
    }
    for (int o = LP >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
    if (p < np && sub == 0) part[(size_t)(c.lrow + r) * nkp + c.ka / KP + kp] = acc;
  }
}

// 32 pieces of 256 elements of chunk e, from piece p0 on. Lane l multiplies
// elements [8l, 8l + 8) of each piece; the transposing butterfly (31
// shuffles) then leaves piece p0 + i's sum in lane i, which stores it.
// Pieces past the chunk's end read its last row and are not stored.
template <int WT>
SPEC_DEV void tile256(const unsigned char* slot, const ChE& e, int p0, const float* x, int nkp, float* part,
                      int lane) {
  const int npk = e.kw >> 8, np = e.nr * npk, last = e.nr - 1;
  float v[32];
  if (npk == 1) {
    const float4 xa = *reinterpret_cast<const float4*>(x + e.ka + 8 * lane);
    const float4 xb = *reinterpret_cast<const float4*>(x + e.ka + 8 * lane + 4);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float w[8];
      weights8<WT>(slot, e.kw, e.nr, imin(p0 + i, last), 8 * lane, w);
      float a = w[0] * xa.x;
      a = fmaf(w[1], xa.y, a); a = fmaf(w[2], xa.z, a); a = fmaf(w[3], xa.w, a);
      a = fmaf(w[4], xb.x, a); a = fmaf(w[5], xb.y, a); a = fmaf(w[6], xb.z, a); a = fmaf(w[7], xb.w, a);
      v[i] = a;
    }
  } else {
    int r = p0 / npk, kp = p0 - r * npk;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float* xx = x + e.ka + kp * 256 + 8 * lane;
      const float4 xa = *reinterpret_cast<const float4*>(xx), xb = *reinterpret_cast<const float4*>(xx + 4);
      float w[8];
      weights8<WT>(slot, e.kw, e.nr, imin(r, last), kp * 256 + 8 * lane, w);
      float a = w[0] * xa.x;
      a = fmaf(w[1], xa.y, a); a = fmaf(w[2], xa.z, a); a = fmaf(w[3], xa.w, a);
      a = fmaf(w[4], xb.x, a); a = fmaf(w[5], xb.y, a); a = fmaf(w[6], xb.z, a); a = fmaf(w[7], xb.w, a);
      v[i] = a;
      ++kp;
      const bool wrap = kp == npk;
      kp = wrap ? 0 : kp;
      r += wrap ? 1 : 0;
    }
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? v[i] : v[i + s];
      const float keep = up ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, send, s);
    }
  }
  const int p = p0 + lane;
  if (p < np) {
    const int rr = p / npk, kk = p - rr * npk;
    part[(size_t)(e.lrow + rr) * nkp + (e.ka >> 8) + kk] = v[0];
  }
}

// ---- shared state of one CTA -----------------------------------------------

struct Cta {
  unsigned rank, ncta;
  int tid, lane, warp;
  unsigned char* ring;
  uint64_t* full;
  volatile int* abort_s;
  Tabs T;
  const int* seg_row;
  const int* seg_lrow;
  const int* nseg;
  float* part;
  float* y;
  unsigned long long* cta_best;
  int q;            // chunks consumed
  int qs;           // ring slot of the next chunk to consume (q % ns)
  unsigned qp;      // its mbarrier phase parity ((q / ns) & 1)
  bool rec;         // this thread records the phase trace
  int tn;           // trace entries written
};

// Timestamp of the current point of the walk (thread 0 of CTA 0 of sequence 0).
SPEC_DEV void mark(const DraftDesc& D, Cta& C) {
  if (C.rec) D.trace[C.tn++] = globaltimer();
}

SPEC_DEV float row_sum(const float* part, int lr, int nkp) {
  float s = 0.f;
  for (int i = 0; i < nkp; ++i) s += part[(size_t)lr * nkp + i];
  return s;
}

// Cluster barrier with the ring refill in its shadow: thread 0 issues the
// next chunks after its CTA has arrived and before it waits for the others.
template <int WT>
SPEC_DEV void barrier_fill(const DraftDesc& D, Cta& C, Filler& F) {
  cluster_arrive();
  if (C.tid == 0) fill<WT>(D, F, C.q, C.T, C.ring, C.full, C.abort_s);
  __syncwarp();
  cluster_wait();
}

enum { E_STORE, E_ADD, E_GEGLU, E_BEST, E_GLOBAL };

// Consume operation `ph` (x: its input vector in shared memory) and apply its
// epilogue. STORE / ADD / GEGLU push the CTA's outputs into `dst` of every CTA
// of the cluster; GLOBAL writes them to `dst` in global memory; BEST pushes
// the CTA's best (score, token) key into best_s[rank] of every CTA. The chunks are taken in groups of at most `ns`
// (one group unless a CTA's rows exceed the ring); the group's 32-piece tiles
// are dealt to the warps round-robin.
template <int WT>
SPEC_DEV void run_op(const DraftDesc& D, Cta& C, Filler& F, int ph, const float* x, int epi, float* dst,
                     unsigned long long* best_s) {
  const OpI o = C.T.ops[ph];
  // the members' chunks are a table of their own, rebuilt each step from 0
  const ChE* tab = o.type == PH_MEMB ? C.T.mch : C.T.ch + o.c0;
  const int nc = o.type == PH_MEMB ? *C.T.nm : o.nc;
  const int nkp = o.nkp, KP = o.K / nkp;
  if (C.tid == 0) *C.cta_best = 0ull;
  for (int g0 = 0; g0 < nc; g0 += D.ns) {
    const int n = imin(D.ns, nc - g0);
    // top the ring up first: the slots of every consumed chunk are free here
    if (C.tid == 0) fill<WT>(D, F, C.q, C.T, C.ring, C.full, C.abort_s);
    int ok = 1;
    if (C.lane == 0) {
      for (int i = 0; i < n && ok; ++i) {
        const bool wrap = C.qs + i >= D.ns;  // n <= ns: at most one wrap
        ok = wait_phase(&C.full[C.qs + i - (wrap ? D.ns : 0)], C.qp ^ (wrap ? 1u : 0u), C.abort_s, D.err) ? 1 : 0;
      }
    }
    ok = __shfl_sync(FULL, ok, 0);
    if (ok) {
      int tb = 0;
      for (int i = 0; i < n; ++i) {
        const ChE e = tab[g0 + i];
        const int si = C.qs + i >= D.ns ? C.qs + i - D.ns : C.qs + i;
        const unsigned char* slot = C.ring + (size_t)si * SLOT;
        if (KP == 256) {
          const int nt = (e.nr * (e.kw >> 8) + 31) >> 5;
          for (int t = tb + ((C.warp - tb % DW) + DW) % DW; t < tb + nt; t += DW)
            tile256<WT>(slot, e, (t - tb) * 32, x, nkp, C.part, C.lane);
          tb += nt;
        } else {
          const Chunk c{e.row, e.lrow, e.nr, e.ka, e.kw};
          dot_chunk<WT>(slot, c, x, KP, nkp, C.part, C.warp, C.lane);
        }
      }
    }
    C.q += n;
    C.qs += n;
    if (C.qs >= D.ns) {
      C.qs -= D.ns;
      C.qp ^= 1u;
    }
    __syncthreads();  // the group's slots are free again
  }
  if (nc == 0) __syncthreads();
  mark(D, C);
  if (epi == E_BEST) {
    unsigned long long best = 0ull;
    for (int lr = C.tid; lr < o.rows; lr += NTH) {
      const float v = row_sum(C.part, lr, nkp);
      int tok;
      if (o.type == PH_MEMB) {
        int sgi = 0;
        while (sgi + 1 < *C.nseg && lr >= C.seg_lrow[sgi + 1]) ++sgi;
        tok = D.perm[C.seg_row[sgi] + (lr - C.seg_lrow[sgi])];
      } else {
        tok = o.o0 + lr;
      }
      const unsigned long long key = pack_best(v, (uint32_t)tok);
      best = key > best ? key : best;
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
      const unsigned long long t = __shfl_xor_sync(FULL, best, s);
      best = t > best ? t : best;
    }
    if (C.lane == 0 && best) atomicMax(C.cta_best, best);
    __syncthreads();
    if (C.tid < (int)C.ncta) st_remote_u64(&best_s[C.rank], C.tid, *C.cta_best);
    return;
  }
  if (epi == E_GLOBAL) {
    // this CTA's outputs to global memory (read after the next cluster barrier)
    for (int i = C.tid; i < o.no; i += NTH) dst[o.o0 + i] = row_sum(C.part, i, nkp);
    __syncthreads();
    return;
  }
  for (int i = C.tid; i < o.no; i += NTH) {
    float v;
    if (epi == E_GEGLU) {
      const float gt = row_sum(C.part, i, nkp), up = row_sum(C.part, o.no + i, nkp);
      v = 0.5f * gt * (1.f + erff(gt * 0.70710678118654752f)) * up;
    } else {
      v = row_sum(C.part, i, nkp);
      if (epi == E_ADD) v += dst[o.o0 + i];
    }
    C.y[i] = v;
  }
  __syncthreads();
  for (int t = C.tid; t < o.no * (int)C.ncta; t += NTH) {
    const int i = t / C.ncta, r = t - i * C.ncta;
    st_remote(dst + o.o0 + i, r, C.y[i]);
  }
  __syncthreads();
}

// dst[k] = src[k] / rms(src) * gain[k], k < K (the same values in every CTA).
SPEC_DEV void norm_into(const float* src, const float* gain, int K, float eps, float* dst, float* red, int tid) {
  float ss = 0.f;
  for (int k = tid; k < K; k += NTH) ss = fmaf(src[k], src[k], ss);
  const float inv = rsqrtf(block_sum(ss, red) / (float)K + eps);
  for (int k = tid; k < K; k += NTH) dst[k] = src[k] * inv * gain[k];
  __syncthreads();
}

// ---- cross-attention --------------------------------------------------------

template <int PER, typename KT>
SPEC_DEV void kv_per(const KT* p, float* o) {
  if (std::is_same<KT, float>::value) {
    if (PER == 4) {
      const float4 a = *reinterpret_cast<const float4*>(p);
      o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    } else {
      const float2 a = *reinterpret_cast<const float2*>(p);
      o[0] = a.x; o[1] = a.y;
    }
  } else {
    if (PER == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      o[0] = bf16lo(v.x); o[1] = bf16hi(v.x); o[2] = bf16lo(v.y); o[3] = bf16hi(v.y);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      o[0] = bf16lo(v); o[1] = bf16hi(v);
    }
  }
}

// Items are (kv head, page range); warp `gw` of the cluster takes item gw.
// The partial of item i, head g sits at part[(i * G + g) * (HD + 2)]: {o[HD], m, l}.
struct AttnSplit {
  int npg, ipk, ppi;
};
SPEC_DEV AttnSplit attn_split(int L0, int max_pages, int nkv, int nwt) {
  AttnSplit a;
  a.npg = min((L0 + PAGE - 1) / PAGE, max_pages);
  const int ipk = max(1, min(a.npg, nwt / nkv));
  a.ppi = a.npg > 0 ? (a.npg + ipk - 1) / ipk : 1;
  a.ipk = a.npg > 0 ? (a.npg + a.ppi - 1) / a.ppi : 0;
  return a;
}

template <int HD, typename KT>
SPEC_DEV void attend_items(const DraftDesc& D, int slot_b, int L0, const AttnSplit& S, const float* qrot,
                           float* pbuf, float* part, int gw, int warp, int lane) {
  constexpr int PER = HD / 32;
  const int G = D.dnq / D.nkv;
  if (gw >= D.nkv * S.ipk) return;
  const int kvh = gw / S.ipk, it = gw - kvh * S.ipk;
  const int pg0 = it * S.ppi, pg1 = min(S.npg, pg0 + S.ppi);
  const KT* pool = (const KT*)D.pool + D.layer_off;
  const float scale = rsqrtf((float)HD);
  float m[GMAX], l[GMAX], o[GMAX][PER];
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[g][i] = 0.f;
  }
  float* pw = pbuf + (size_t)warp * G * PAGE;
  for (int pg = pg0; pg < pg1; ++pg) {
    const int page = D.block_table[(size_t)slot_b * D.max_pages + pg];
    if (page < 0 || page >= D.n_pages) {
      if (lane == 0) set_error(D.err, SPEC_ERR_CAPACITY);
      continue;
    }
    const int nk = min(PAGE, L0 - pg * PAGE);
    const KT* kp = pool + ((size_t)page * 2 * D.nkv + kvh) * PAGE * HD;
    const KT* vp = pool + (((size_t)page * 2 + 1) * D.nkv + kvh) * PAGE * HD;
    const bool v0 = lane < nk, v1 = lane + 32 < nk;
    float s0[GMAX], s1[GMAX];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) s0[g] = s1[g] = 0.f;
    // scores: the lane's two keys against every q head of the group, K rows
    // loaded a batch of 4 x 16 bytes per key at a time
    constexpr int CH = HD / 8, BT = std::is_same<KT, float>::value ? 2 : 4;
    constexpr int KW = std::is_same<KT, float>::value ? 2 : 1;  // 16-byte words per 8 elements
#pragma unroll 1
    for (int c0 = 0; c0 < CH; c0 += BT) {
      uint4 ra[BT][KW], rb[BT][KW];
#pragma unroll
      for (int u = 0; u < BT; ++u)
#pragma unroll
        for (int w = 0; w < KW; ++w) {
          ra[u][w] = v0 ? *reinterpret_cast<const uint4*>(kp + (size_t)lane * HD + (c0 + u) * 8 + 4 * w) : make_uint4(0, 0, 0, 0);
          rb[u][w] = v1 ? *reinterpret_cast<const uint4*>(kp + (size_t)(lane + 32) * HD + (c0 + u) * 8 + 4 * w) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int u = 0; u < BT; ++u) {
        float k0[8], k1[8];
        if constexpr (std::is_same<KT, float>::value) {
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            k0[4 * w] = __uint_as_float(ra[u][w].x); k0[4 * w + 1] = __uint_as_float(ra[u][w].y);
            k0[4 * w + 2] = __uint_as_float(ra[u][w].z); k0[4 * w + 3] = __uint_as_float(ra[u][w].w);
            k1[4 * w] = __uint_as_float(rb[u][w].x); k1[4 * w + 1] = __uint_as_float(rb[u][w].y);
            k1[4 * w + 2] = __uint_as_float(rb[u][w].z); k1[4 * w + 3] = __uint_as_float(rb[u][w].w);
          }
        } else {
          const uint4 a = ra[u][0], bq = rb[u][0];
          k0[0] = bf16lo(a.x); k0[1] = bf16hi(a.x); k0[2] = bf16lo(a.y); k0[3] = bf16hi(a.y);
          k0[4] = bf16lo(a.z); k0[5] = bf16hi(a.z); k0[6] = bf16lo(a.w); k0[7] = bf16hi(a.w);
          k1[0] = bf16lo(bq.x); k1[1] = bf16hi(bq.x); k1[2] = bf16lo(bq.y); k1[3] = bf16hi(bq.y);
          k1[4] = bf16lo(bq.z); k1[5] = bf16hi(bq.z); k1[6] = bf16lo(bq.w); k1[7] = bf16hi(bq.w);
        }
        const int d0 = (c0 + u) * 8;
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
          if (g < G) {
            const float* qq = qrot + (size_t)(kvh * G + g) * HD + d0;
            const float4 qa = *reinterpret_cast<const float4*>(qq), qb = *reinterpret_cast<const float4*>(qq + 4);
            float a = s0[g], b = s1[g];
            a = fmaf(k0[0], qa.x, a); a = fmaf(k0[1], qa.y, a); a = fmaf(k0[2], qa.z, a); a = fmaf(k0[3], qa.w, a);
            a = fmaf(k0[4], qb.x, a); a = fmaf(k0[5], qb.y, a); a = fmaf(k0[6], qb.z, a); a = fmaf(k0[7], qb.w, a);
            b = fmaf(k1[0], qa.x, b); b = fmaf(k1[1], qa.y, b); b = fmaf(k1[2], qa.z, b); b = fmaf(k1[3], qa.w, b);
            b = fmaf(k1[4], qb.x, b); b = fmaf(k1[5], qb.y, b); b = fmaf(k1[6], qb.z, b); b = fmaf(k1[7], qb.w, b);
            s0[g] = a;
            s1[g] = b;
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
      if (g < G) {
        const float a0 = v0 ? s0[g] * scale : -INFINITY, a1 = v1 ? s1[g] * scale : -INFINITY;
        const float mn = fmaxf(m[g], warp_max(fmaxf(a0, a1)));
        const float corr = __expf(m[g] - mn);
        const float p0 = v0 ? __expf(a0 - mn) : 0.f, p1 = v1 ? __expf(a1 - mn) : 0.f;
        l[g] = l[g] * corr + warp_sum(p0 + p1);
        m[g] = mn;
#pragma unroll
        for (int i = 0; i < PER; ++i) o[g][i] *= corr;
        pw[g * PAGE + lane] = p0;
        pw[g * PAGE + lane + 32] = p1;
      }
    }
    __syncwarp();
    // o += p . V, V rows loaded 8 at a time
    constexpr int VB = 8;
#pragma unroll 1
    for (int j0 = 0; j0 < nk; j0 += VB) {
      float v[VB][PER];
#pragma unroll
      for (int u = 0; u < VB; ++u) {
        if (j0 + u < nk) kv_per<PER, KT>(vp + (size_t)(j0 + u) * HD + PER * lane, v[u]);
        else
#pragma unroll
          for (int i = 0; i < PER; ++i) v[u][i] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < VB; ++u) {
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
          if (g < G) {
            const float pj = pw[g * PAGE + ((j0 + u) & (PAGE - 1))];
#pragma unroll
            for (int i = 0; i < PER; ++i) o[g][i] = fmaf(pj, v[u][i], o[g][i]);
          }
        }
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    if (g < G) {
      float* pp = part + ((size_t)gw * G + g) * (HD + 2);
#pragma unroll
      for (int i = 0; i < PER; ++i) pp[PER * lane + i] = o[g][i];
      if (lane == 0) {
        pp[HD] = m[g];
        pp[HD + 1] = l[g];
      }
    }
  }
}

// att[hh] for q heads hh = gw, gw + nwt, ...: the fixed-order merge of the
// head's item partials (at most 64 per head), pushed into `att` of every CTA.
template <int HD>
SPEC_DEV void merge_heads(const DraftDesc& D, const AttnSplit& S, const float* part, float* att, int gw, int nwt,
                          unsigned ncta, int lane) {
  constexpr int PER = HD / 32;
  const int G = D.dnq / D.nkv;
  for (int hh = gw; hh < D.dnq; hh += nwt) {
    const int kvh = hh / G, g = hh - kvh * G;
    const float* base = part + ((size_t)kvh * S.ipk * G + g) * (HD + 2);
    const size_t istride = (size_t)G * (HD + 2);
    // lane i holds items i and i + 32: max, then weights and the l sum
    float mi[2], li[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = lane + 32 * e;
      mi[e] = i < S.ipk ? __ldcg(base + i * istride + HD) : -INFINITY;
      li[e] = i < S.ipk ? __ldcg(base + i * istride + HD + 1) : 0.f;
    }
    const float M = warp_max(fmaxf(mi[0], mi[1]));
    float wi[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) wi[e] = mi[e] == -INFINITY ? 0.f : __expf(mi[e] - M);
    // the l sum in item order: lanes reduce in a fixed tree
    const float L = warp_sum(li[0] * wi[0] + li[1] * wi[1]);
    float o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    for (int i0 = 0; i0 < S.ipk; i0 += 8) {
      float v[8][PER];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u;
#pragma unroll
        for (int e = 0; e < PER; ++e) v[u][e] = i < S.ipk ? __ldcg(base + i * istride + PER * lane + e) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u;
        const float w = __shfl_sync(FULL, (i & 32) ? wi[1] : wi[0], i & 31);
        if (i < S.ipk) {
#pragma unroll
          for (int e = 0; e < PER; ++e) o[e] = fmaf(w, v[u][e], o[e]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float* dst = att + (size_t)hh * HD + PER * lane;
    for (unsigned r = 0; r < ncta; ++r) {
      if (PER == 4) {
        st_remote4(dst, r, make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv));
      } else {
#pragma unroll
        for (int e = 0; e < PER; ++e) st_remote(dst + e, r, o[e] * inv);
      }
    }
  }
}

// ---- top-C cluster selection -------------------------------------------------

SPEC_DEV int block_scan_excl(int v, int* ws, int lane, int warp) {
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(FULL, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < DW ? ws[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(FULL, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < DW) ws[lane] = wi - w;
  }
  __syncthreads();
  const int r = ws[warp] + inc - v;
  __syncthreads();
  return r;
}

// The top_c clusters by (binary32 score desc, id asc), as ids in increasing
// order: radix select of the top_c-th key on its 32-bit ordered form, then the
// ties at that key taken lowest id first.
SPEC_DEV void select_clusters(const float* sc, int C, int top_c, int* chosen, int* hist, int* ws, int tid, int lane,
                              int warp) {
  unsigned prefix = 0, mask = 0;
  int need = top_c;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NTH) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < C; i += NTH) {
      const unsigned key = ord_key(sc[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      int cnt[8], loc = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = hist[8 * lane + i];
        loc += cnt[i];
      }
      int suf = loc;  // candidates in the bins of lanes >= this lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(FULL, suf, o);
        if (lane + o < 32) suf += t;
      }
      const int above = suf - loc;
      if (above < need && need <= suf) {
        int acc = above;
        for (int i = 7; i >= 0; --i) {
          if (acc + cnt[i] >= need) {
            ws[DW + 1] = 8 * lane + i;
            ws[DW + 2] = acc;
            break;
          }
          acc += cnt[i];
        }
      }
    }
    __syncthreads();
    prefix |= (unsigned)ws[DW + 1] << shift;
    mask |= 255u << shift;
    need -= ws[DW + 2];
    __syncthreads();
  }
  // keys above the threshold, then `need` of the keys equal to it, lowest id first
  const int per = (C + NTH - 1) / NTH, i0 = min(C, tid * per), i1 = min(C, i0 + per);
  int neq = 0;
  for (int i = i0; i < i1; ++i) neq += ord_key(sc[i]) == prefix;
  int eq_rank = block_scan_excl(neq, ws, lane, warp);
  int nsel = 0;
  for (int i = i0; i < i1; ++i) {
    const unsigned key = ord_key(sc[i]);
    nsel += key > prefix || (key == prefix && eq_rank++ < need);
  }
  int pos = block_scan_excl(nsel, ws, lane, warp);
  eq_rank -= neq;
  for (int i = i0; i < i1; ++i) {
    const unsigned key = ord_key(sc[i]);
    if (key > prefix || (key == prefix && eq_rank++ < need)) chosen[pos++] = i;
  }
  __syncthreads();
}

// ---- the kernel ---------------------------------------------------------------

SPEC_DEV float embed_elem(const Mat& E, int d, int tok, int k) {
  if (E.dtype == DT_F32) return ((const float*)E.data)[(size_t)tok * d + k];
  if (E.dtype == DT_BF16) return __bfloat162float(((const __nv_bfloat16*)E.data)[(size_t)tok * d + k]);
  const uint8_t* cb = (const uint8_t*)E.data + (size_t)tok * (d / 2);
  const int blk = k >> 5, i = k & 31;
  const uint8_t byte = cb[blk * 16 + (i & 15)];
  const int code = i < 16 ? (byte & 15) : (byte >> 4);
  return __half2float(((const __half*)E.scales)[(size_t)tok * (d / 32) + blk]) * (float)(code - 8);
}

template <int WT, int HD>
__global__ void __launch_bounds__(NTH, 1) draft_cluster_kernel(const DraftDesc D) {
  using KT = typename std::conditional<WT == DT_F32, float, __nv_bfloat16>::type;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[NS_MAX];
  __shared__ OpI ops_s[MAX_OPS];
  __shared__ ChE ch_s[MAX_CH], mch_s[MAX_MCH];
  __shared__ int seg_row_s[MAXSEG], seg_lrow_s[MAXSEG];
  __shared__ unsigned long long best_s[MAXC], cta_best;
  __shared__ float red[32], rope_s[HD];
  __shared__ int hist[256], ws[DW + 4], chosen_s[TOPC_MAX];
  __shared__ int tok_s, abort_v, sel_step, nch_s, nm_s, nseg_s, att_done_s;
  constexpr bool TC_ATT = !std::is_same<KT, float>::value;  // tensor-core attention (bf16 cache)

  Cta C;
  C.rank = cluster_rank();
  C.ncta = cluster_ctas();
  C.tid = threadIdx.x;
  C.lane = C.tid & 31;
  C.warp = C.tid >> 5;
  C.ring = smem;
  C.full = full;
  C.abort_s = &abort_v;
  C.seg_row = seg_row_s;
  C.seg_lrow = seg_lrow_s;
  C.nseg = &nseg_s;
  C.part = (float*)(smem + D.off_part);
  C.y = (float*)(smem + D.off_y);
  C.cta_best = &cta_best;
  C.q = 0;
  C.qs = 0;
  C.qp = 0;
  C.rec = D.trace != nullptr && blockIdx.y == 0 && C.rank == 0 && threadIdx.x == 0;
  C.tn = 0;
  float* U1 = (float*)(smem + D.off_u1);   // normalised input; rotated q + probabilities
  float* QAA = (float*)(smem + D.off_qaa); // q, attention output, GEGLU output, next h
  float* u_s = (float*)(smem + D.off_u);
  float* sc_s = (float*)(smem + D.off_sc);
  const int tid = C.tid, b = blockIdx.y, slot_b = D.seq_ids[b];
  const int gw = (int)C.rank * DW + C.warp, nwt = (int)C.ncta * DW;
  const int d = D.d, h = D.h, dq = D.dnq * HD, nop = n_ops(D.L, D.clustered);
  float* apart = D.part + (size_t)b * D.part_stride;

  if (tid == 0) {
    for (int s = 0; s < D.ns; ++s) mbar_init(&full[s], 1);
    mbar_init_fence();
    abort_v = 0;
    sel_step = 0;
    nm_s = 0;
    nseg_s = 0;
    att_done_s = 0;
    nch_s = build_tables<WT>(D, C.rank, C.ncta, ops_s, ch_s);
  }
  __syncthreads();
  C.T = Tabs{ops_s, ch_s, mch_s, nch_s, &nm_s, &sel_step, TC_ATT ? &att_done_s : nullptr, D.L};
  cluster_sync();  // every CTA runs before any distributed-shared-memory store
  mark(D, C);

  Filler F;
  F.j = 1;
  F.pos = 0;
  F.issued = 0;
  F.slot = 0;
  F.done = false;
  if (tid == 0) fill<WT>(D, F, 0, C.T, C.ring, full, C.abort_s);

  const int L0 = D.seq_len[slot_b];
  const AttnSplit S = attn_split(L0, D.max_pages, D.nkv, nwt);
  for (int j = 1; j <= D.k; ++j) {
    // input: [N(h_{j-1}); N(E[tok_{j-1}])] and the RoPE table of this step
    const int tok = j == 1 ? D.pending[slot_b] : tok_s;
    float sh = 0.f, se = 0.f;
    for (int k = tid; k < d; k += NTH) {
      const float hv = j == 1 ? D.hid[(size_t)slot_b * d + k] : QAA[k];
      const float ev = embed_elem(D.embed, d, tok, k);
      sh = fmaf(hv, hv, sh);
      se = fmaf(ev, ev, se);
      U1[k] = hv;
      U1[d + k] = ev;
    }
    const float ih = rsqrtf(block_sum(sh, red) / (float)d + D.eps);
    const float ie = rsqrtf(block_sum(se, red) / (float)d + D.eps);
    for (int k = tid; k < d; k += NTH) {
      U1[k] *= ih * D.g_in_h[k];
      U1[d + k] *= ie * D.g_in_e[k];
    }
    if (tid < HD / 2) {
      const int pos = L0 + j - 1;
      double sn, cs;
      sincos((double)pos * exp(-2.0 * tid / HD * log((double)D.theta)), &sn, &cs);
      rope_s[2 * tid] = (float)cs;
      rope_s[2 * tid + 1] = (float)sn;
      if (TC_ATT && C.rank == 0) {
        // the attention rotates its queries with this row (read after a barrier)
        D.rope[(size_t)b * HD + 2 * tid] = (float)cs;
        D.rope[(size_t)b * HD + 2 * tid + 1] = (float)sn;
      }
    }
    __syncthreads();

    // the step's operations in order; each run_op is followed by a cluster
    // barrier, except W_out, whose head shares its input u
    for (int ph = 0; ph < nop; ++ph) {
      const int type = ops_s[ph].type, l = ph >= 1 ? (ph - 1) >> 2 : 0;
      const float* x = U1;
      float* dst = nullptr;
      int epi = E_STORE;
      if (type == PH_WIN) {
        dst = u_s;
      } else if (type == PH_WQ) {
        norm_into(u_s, D.g_attn + (size_t)l * h, h, D.eps, U1, red, tid);
        if (TC_ATT) {
          epi = E_GLOBAL;
          dst = D.q + (size_t)b * dq;
        } else {
          dst = QAA;
        }
      } else if (type == PH_WO && TC_ATT) {
        // every chunk issued so far is consumed and the filler waits for this
        // attention: the ring's shared memory is free for its page buffers
        const int cpk = (int)C.ncta / D.nkv, kvh = (int)C.rank / cpk, split = (int)C.rank % cpk;
        const int npg = min((L0 + PAGE - 1) / PAGE, D.max_pages);
        AttnArgs a = {};
        a.q = D.q; a.ldq = dq; a.B = D.B; a.R = 1; a.nq = D.dnq; a.nkv = D.nkv; a.hd = HD; a.key_extra = 0;
        a.pool = D.pool; a.kv_dtype = DT_BF16; a.layer_elems = D.layer_elems; a.layer = D.tlayer;
        a.n_pages = D.n_pages; a.max_pages = D.max_pages; a.block_table = D.block_table; a.seq_ids = D.seq_ids;
        a.seq_len = D.seq_len; a.rope_cs = D.rope; a.n_split = cpk;
        a.pages_per_split = npg > 0 ? (npg + cpk - 1) / cpk : 1;
        a.part_o = D.part_o; a.part_ml = D.part_ml; a.out = D.att; a.err = D.err;
        if (!*C.abort_s)
          atc::AttnTc<HD>::run(a, a.pages_per_split, D.att_cnt, smem, b * D.nkv + kvh, split, false,
                               (size_t)D.ns * SLOT, D.pw_cap);
        // the ring's next bulk copies write where these threads wrote
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) att_done_s = att_done_s + 1;
        barrier_fill<WT>(D, C, F);
        mark(D, C);
        for (int t = tid; t < dq; t += NTH) QAA[t] = __ldcg(D.att + (size_t)b * dq + t);
        __syncthreads();
        mark(D, C);
        x = QAA;
        epi = E_ADD;
        dst = u_s;
      } else if (type == PH_WO) {
        // rotate-half RoPE of every q head into U1, the per-item partials, the merge
        for (int t = tid; t < dq; t += NTH) {
          const int dd = t % HD, half = HD / 2, i = dd % half;
          const float* qr = QAA + (t - dd);
          const float cs = rope_s[2 * i], sn = rope_s[2 * i + 1];
          U1[t] = dd < half ? qr[dd] * cs - qr[dd + half] * sn : qr[dd] * cs + qr[dd - half] * sn;
        }
        __syncthreads();
        if (!*C.abort_s) attend_items<HD, KT>(D, slot_b, L0, S, U1, U1 + dq, apart, gw, C.warp, C.lane);
        barrier_fill<WT>(D, C, F);
        mark(D, C);
        merge_heads<HD>(D, S, apart, QAA, gw, nwt, C.ncta, C.lane);
        barrier_fill<WT>(D, C, F);
        mark(D, C);
        x = QAA;
        epi = E_ADD;
        dst = u_s;
      } else if (type == PH_WGU) {
        norm_into(u_s, D.g_ffn + (size_t)l * h, h, D.eps, U1, red, tid);
        epi = E_GEGLU;
        dst = QAA;
      } else if (type == PH_WDOWN) {
        x = QAA;
        epi = E_ADD;
        dst = u_s;
      } else if (type == PH_WOUT) {
        // U1 = N_out(u) for the head; W_out reads the raw u
        norm_into(u_s, D.g_out, h, D.eps, U1, red, tid);
        x = u_s;
        dst = QAA;
      } else if (type == PH_HEAD) {
        epi = D.clustered ? E_STORE : E_BEST;
        dst = sc_s;
      } else {
        select_clusters(sc_s, D.C, D.top_c, chosen_s, hist, ws, tid, C.lane, C.warp);
        if (tid == 0) {
          nm_s = build_members<WT>(D, ops_s[ph], ph, chosen_s, mch_s, seg_row_s, seg_lrow_s, &nseg_s);
          sel_step = j;
          fill<WT>(D, F, C.q, C.T, C.ring, full, C.abort_s);
        }
        __syncthreads();
        epi = E_BEST;
      }
      run_op<WT>(D, C, F, ph, x, epi, dst, best_s);
      if (type != PH_WOUT) {
        barrier_fill<WT>(D, C, F);
        mark(D, C);
      }
    }
    if (C.warp == 0) {
      unsigned long long bst = C.lane < (int)C.ncta ? best_s[C.lane] : 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(FULL, bst, o);
        bst = t > bst ? t : bst;
      }
      if (C.lane == 0) {
        tok_s = (int)best_index(bst);
        if (C.rank == 0) D.drafts[(size_t)b * D.k + j - 1] = tok_s;
      }
    }
    __syncthreads();
  }
  // after an abort, let the copies still in flight land before the CTA exits
  if (tid == 0) {
    int s = C.qs;
    unsigned par = C.qp;
    for (int c = C.q; c < F.issued; ++c) {
      for (unsigned it = 0; it < SPIN_LIMIT; ++it)
        if (mbar_test(&full[s], par)) break;
      if (++s == D.ns) {
        s = 0;
        par ^= 1u;
      }
    }
  }
}

using KernelFn = void (*)(const DraftDesc);

KernelFn kernel_for(int wt, int hd) {
  if (wt == DT_F32) return hd == 128 ? draft_cluster_kernel<DT_F32, 128> : draft_cluster_kernel<DT_F32, 64>;
  if (wt == DT_BF16) return hd == 128 ? draft_cluster_kernel<DT_BF16, 128> : draft_cluster_kernel<DT_BF16, 64>;
  return hd == 128 ? draft_cluster_kernel<DT_Q4_0, 128> : draft_cluster_kernel<DT_Q4_0, 64>;
}

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// True when the GPU can co-schedule a cluster of `n` CTAs of this kernel.
bool cluster_fits(KernelFn kern, size_t smem, int n) {
  cudaLaunchConfig_t q = {};
  q.gridDim = dim3(n);
  q.blockDim = dim3(NTH);
  q.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = n;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  q.attrs = at;
  q.numAttrs = 1;
  int active = 0;
  const cudaError_t e = cudaOccupancyMaxActiveClusters(&active, kern, &q);
  cudaGetLastError();
  return e == cudaSuccess && active >= 1;
}

size_t align128(long long floats) { return ((size_t)floats * 4 + 127) & ~size_t(127); }

}  // namespace

long long draft_cluster_part_floats(int G, int hd) { return (long long)MAXC * DW * G * (hd + 2); }

bool draft_cluster_plan(DraftDesc& D) {
  if (D.nkv < 1 || D.dnq % D.nkv) return false;
  const int G = D.dnq / D.nkv;
  if (D.B < 1 || D.k < 1 || (D.hd != 64 && D.hd != 128) || G > GMAX) return false;
  if (D.L < 1 || n_ops(D.L, D.clustered) > MAX_OPS) return false;
  if ((D.wdtype == DT_F32) != (D.kv_dtype == DT_F32)) return false;
  if (D.d % 8 || D.h % 8) return false;
  const int dq = D.dnq * D.hd;
  const int Ks[5] = {2 * D.d, D.h, dq, D.ff, D.h};
  for (int K : Ks) {
    if (!piece_of(K)) return false;
    if (D.wdtype == DT_Q4_0 && K % 256) return false;
  }
  if (D.clustered && (D.top_c < 1 || D.top_c > TOPC_MAX || D.C < D.top_c || D.C > 8192 || D.cs < 1))
    return false;
  KernelFn kern = kernel_for(D.wdtype, D.hd);
  // dynamic shared memory: the per-block opt-in limit less the kernel's static tables
  int dev = 0, optin = 0;
  cudaFuncAttributes fa = {};
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const size_t limit = (size_t)optin - fa.sharedSizeBytes - 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int members_total = D.clustered ? D.top_c * D.cs : 0;
  for (int ncta : {MAXC, MAXC / 2}) {
    // every CTA's chunk tables must fit theirs
    bool fits = true;
    for (int rank = 0; rank < ncta && fits; ++rank) {
      int nch = 0;
      for (int ph = 0; ph < n_ops(D.L, D.clustered); ++ph) {
        int type, K, N;
        op_dims(ph, D.L, D.d, D.h, dq, D.ff, D.C, D.V, members_total, D.clustered, type, K, N);
        const int o0 = (int)((long long)N * rank / ncta), no = (int)((long long)N * (rank + 1) / ncta) - o0;
        const Geo g = geometry(K, D.wdtype);
        if (type == PH_MEMB) {
          int nm = 0, nseg = 0;
          for (int m = o0; m < o0 + no;) {
            const int c = m / D.cs, e = std::min(o0 + no, (c + 1) * D.cs);
            nm = add_chunks(nullptr, nm, 0, ph, 0, 0, e - m, K, g);
            ++nseg;
            m = e;
          }
          fits = fits && nm <= MAX_MCH && nseg <= MAXSEG;
        } else {
          nch = add_chunks(nullptr, nch, 0, ph, 0, 0, type == PH_WGU ? 2 * no : no, K, g);
        }
      }
      fits = fits && nch <= MAX_CH;
    }
    if (!fits) continue;
    const long long members = cdiv(members_total, ncta);
    const long long head_rows = cdiv(D.clustered ? D.C : D.V, ncta);
    // partial sums (rows x pieces) and outputs per CTA, over every operation
    long long part = 0, ymax = 0;
    auto op = [&](long long N, int K, int rows_mul) {
      part = std::max(part, cdiv(N, ncta) * rows_mul * (K / piece_of(K)));
      ymax = std::max(ymax, cdiv(N, ncta));
    };
    op(D.h, 2 * D.d, 1);
    op(dq, D.h, 1);
    op(D.h, dq, 1);
    op(D.ff, D.h, 2);
    op(D.h, D.ff, 1);
    op(D.d, D.h, 1);
    part = std::max(part, head_rows * (D.h / piece_of(D.h)));
    if (D.clustered) {
      ymax = std::max(ymax, head_rows);
      part = std::max(part, members * (D.h / piece_of(D.h)));
    }
    const long long u1 = std::max<long long>({2LL * D.d, (long long)D.h, (long long)dq + (long long)DW * G * PAGE});
    const long long qaa = std::max<long long>({(long long)dq, (long long)D.ff, (long long)D.d});
    const size_t vec = align128(u1) + align128(qaa) + align128(D.h) + align128(D.clustered ? D.C : 1) +
                       align128(part) + align128(ymax);
    if (vec + 2 * (size_t)SLOT > limit) continue;
    const int ns = (int)std::min<size_t>(NS_MAX, (limit - vec) / SLOT);
    // the tensor-core attention runs in the ring: its page slots must fit there
    int pw_cap = 0;
    if (D.kv_dtype == DT_BF16) {
      if (ncta % D.nkv) continue;
      for (int pw = 4; pw >= 1 && !pw_cap; --pw)
        if (attention_tc_smem_slots(D.hd, G, 1, pw) <= (size_t)ns * SLOT) pw_cap = pw;
      if (!pw_cap) continue;
    }
    size_t off = (size_t)ns * SLOT;
    auto take = [&](long long floats) {
      const size_t o = off;
      off += align128(floats);
      return (int)o;
    };
    D.off_u1 = take(u1);
    D.off_qaa = take(qaa);
    D.off_u = take(D.h);
    D.off_sc = take(D.clustered ? D.C : 1);
    D.off_part = take(part);
    D.off_y = take(ymax);
    D.smem = off;
    D.ns = ns;
    D.pw_cap = pw_cap;
    if (!cluster_fits(kern, D.smem, ncta)) continue;
    D.ncta = ncta;
    D.part_stride = draft_cluster_part_floats(G, D.hd);
    return true;
  }
  return false;
}

int draft_cluster(const DraftDesc& D, cudaStream_t st) {
  KernelFn kern = kernel_for(D.wdtype, D.hd);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(D.ncta, D.B);
  cfg.blockDim = dim3(NTH);
  cfg.dynamicSmemBytes = D.smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = D.ncta;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, D) == cudaSuccess ? 1 : -1;
}

}  // namespace spec
