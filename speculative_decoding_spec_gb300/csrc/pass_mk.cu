// pass_mk.cu -- one target pass (prefill / verify / decode) as a single
// persistent kernel.
//
// The verify pass is a chain of dependent steps (embed, then per layer QKV +
// RoPE + KV append, attention, O projection, gate/up, down, then the LM head
// with argmax and greedy accept, then the hidden-state commit). Run as
// separate kernels, every step pays a launch ramp and a serial start (stage
// the activations, then first weight loads). Here one cooperative launch of
// one 16-warp CTA per SM walks all the steps; between two steps every CTA
// (1) pulls its slice of the NEXT step's weights (or KV pages) towards L2 and
// (2) meets the others at a grid barrier. Weights do not depend on the
// activations, so HBM keeps streaming across step boundaries.
//
// The grid barrier is a counter and a generation word in the workspace; its
// waits are bounded: after 2^26 polls (around a second) a CTA gives up, raises the abort flag and
// records SPEC_ERR_TIMEOUT, and every CTA leaves at the next step boundary.
//
// Step bodies are the same device code as the stand-alone kernels
// (gemv_tc.cuh, attn_tc.cuh); data written by another CTA in the same launch
// is read with L2-only loads.
#include <math.h>

#include "attn_tc.cuh"
#include "gemv_tc.cuh"

namespace spec {

namespace {

constexpr int MK_WARPS = 8;               // 255-register budget: no spills in the fused steps
constexpr int MK_THREADS = MK_WARPS * 32;
enum { PH_EMBED = 1, PH_GEMV = 2, PH_ATTN = 3, PH_COMMIT = 4 };

struct Phase {
  int type;
  int map;
  GemvArgs g;
  tc::SkPlan plan;
  AttnArgs at;
};

SPEC_DEV float dq_elem(const Mat& W, int K, long long row, int col) {
  if (W.dtype == DT_F32) return ((const float*)W.data)[row * K + col];
  if (W.dtype == DT_BF16) return __bfloat162float(((const __nv_bfloat16*)W.data)[row * K + col]);
  const uint8_t* c = (const uint8_t*)W.data + row * (K / 2);
  const int b = col >> 5, i = col & 31;
  const uint8_t byte = c[b * 16 + (i & 15)];
  const int code = i < 16 ? (byte & 15) : (byte >> 4);
  return __half2float(((const __half*)W.scales)[row * (K / 32) + b]) * (float)(code - 8);
}

// Arguments of step i of the pass (built by one thread into shared memory).
SPEC_DEV void make_phase(const PassDesc& D, int i, Phase& ph) {
  const int M = D.B * D.R, d = D.d, hd = D.hd, nq = D.nq, nkv = D.nkv, ff = D.ff;
  const int nqkv = (nq + 2 * nkv) * hd, qd = nq * hd;
  ph = Phase{};
  if (i == 0) {
    ph.type = PH_EMBED;
    return;
  }
  if (i == 2 + 5 * D.L) {
    ph.type = PH_COMMIT;
    return;
  }
  GemvArgs& g = ph.g;
  g.M = M;
  g.pdl = 0;
  g.tc_fix = D.tc_fix;
  g.tc_cnt = D.tc_cnt;
  if (i == 1 + 5 * D.L) {  // LM head (tied embedding) + argmax + accept
    g.X = D.x; g.ldx = d; g.N = D.V; g.K = d; g.W = D.embed;
    g.gain = D.g_final; g.eps = D.eps;
    g.epi = EPI_ARGMAX; g.Y = D.logits; g.ldy = D.V; g.best = D.best;
    TailArgs& t = g.tail;
    t.mode = D.mode; t.B = D.B; t.R = D.R; t.k = D.R - 1; t.seq_ids = D.seq_ids; t.drafts = D.tokens;
    t.out_tokens = D.out_tokens; t.n_emitted = D.n_emitted; t.seq_len = D.seq_len; t.pending = D.pending;
    t.stats = D.stats; t.sel_row = D.sel_row; t.best_all = D.best; t.counter = D.counter; t.err = D.err;
  } else {
    const int l = (i - 1) / 5, s = (i - 1) % 5;
    if (s == 1) {
      ph.type = PH_ATTN;
      AttnArgs& at = ph.at;
      at.q = D.qkv; at.ldq = nqkv; at.B = D.B; at.R = D.R; at.nq = nq; at.nkv = nkv; at.hd = hd;
      at.key_extra = 1; at.pool = D.pool; at.kv_dtype = DT_BF16; at.layer_elems = D.layer_elems;
      at.layer = l; at.n_pages = D.n_pages; at.max_pages = D.max_pages; at.block_table = D.block_table;
      at.seq_ids = D.seq_ids; at.seq_len = D.seq_len; at.rope_cs = nullptr; at.n_split = D.n_split;
      at.pages_per_split = D.pps; at.part_o = D.part_o; at.part_ml = D.part_ml; at.out = D.att; at.err = D.err;
      return;
    }
    if (s == 0) {
      g.X = D.x; g.ldx = d; g.N = nqkv; g.K = d; g.W = mat_layer(D.wqkv, l, nqkv, d);
      g.gain = D.g_attn + (size_t)l * d; g.eps = D.eps; g.epi = EPI_ROPE; g.Y = D.qkv; g.ldy = nqkv;
      RopeEpi& e = g.rope;
      e.nq = nq; e.nkv = nkv; e.hd = hd; e.R = D.R; e.rope_cs = D.rope_cs; e.pos = D.pos; e.seq_ids = D.seq_ids;
      e.pool = D.pool; e.layer_off = (long long)l * D.layer_elems; e.n_pages = D.n_pages;
      e.max_pages = D.max_pages; e.block_table = D.block_table; e.err = D.err;
    } else if (s == 2) {
      g.X = D.att; g.ldx = qd; g.N = d; g.K = qd; g.W = mat_layer(D.wo, l, d, qd);
      g.epi = EPI_ADD; g.Y = D.x; g.ldy = d;
    } else if (s == 3) {
      g.X = D.x; g.ldx = d; g.N = 2 * ff; g.K = d; g.W = mat_layer(D.wgu, l, 2 * ff, d);
      g.gain = D.g_ffn + (size_t)l * d; g.eps = D.eps; g.epi = EPI_GEGLU; g.geglu_half = ff; g.Y = D.act;
      g.ldy = ff;
    } else {
      g.X = D.act; g.ldx = ff; g.N = d; g.K = ff; g.W = mat_layer(D.wdown, l, d, ff);
      g.epi = EPI_ADD; g.Y = D.x; g.ldy = d;
    }
  }
  ph.type = PH_GEMV;
  ph.map = tc::map_of(g.epi);
  ph.plan = tc::plan<MK_WARPS>(g, ph.map, D.nsm);
}

SPEC_DEV void gemv_step(const Phase& cur, const PassDesc& D, unsigned char* smem, int phase) {
  tc::Sk<MK_WARPS> k{cur.g, cur.plan, cur.map};
  tc::sk_bind(k, smem, D.tc_fix, D.tc_cnt, blockIdx.x, false);
  if (D.trace) k.trace = D.trace + ((size_t)phase * gridDim.x + blockIdx.x) * 6 + 1;
  k.run();
}

SPEC_DEV void embed_step(const PassDesc& D) {
  const int M = D.B * D.R;
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    const int b = m / D.R, i = m % D.R, slot = D.seq_ids[b];
    int tok;
    if (D.mode == TAIL_PREFILL) tok = D.tokens[b * D.R + i];
    else tok = i == 0 ? D.pending[slot] : D.tokens[b * (D.R - 1) + i - 1];
    if (tok < 0 || tok >= D.V) {
      if (threadIdx.x == 0) set_error(D.err, SPEC_ERR_TOKEN);
      tok = 0;
    }
    const int pos = D.seq_len[slot] + i;
    if (threadIdx.x == 0) D.pos[m] = pos;
    for (int c = threadIdx.x; c < D.d; c += blockDim.x) D.x[(size_t)m * D.d + c] = dq_elem(D.embed, D.d, tok, c);
    const double lt = log((double)D.theta);
    for (int j = threadIdx.x; j < D.hd / 2; j += blockDim.x) {
      double s, c;
      sincos((double)pos * exp(-2.0 * j / D.hd * lt), &s, &c);
      D.rope_cs[(size_t)m * D.hd + 2 * j] = (float)c;
      D.rope_cs[(size_t)m * D.hd + 2 * j + 1] = (float)s;
    }
  }
}

// final-normed hidden state of the row the accept step chose -> slot state
SPEC_DEV void commit_step(const PassDesc& D, float* red) {
  for (int b = blockIdx.x; b < D.B; b += gridDim.x) {
    const int row = __ldcg(D.sel_row + b);
    const float* xr = D.x + (size_t)row * D.d;
    float ss = 0.f;
    for (int c = threadIdx.x; c < D.d; c += blockDim.x) {
      const float v = __ldcg(xr + c);
      ss = fmaf(v, v, ss);
    }
    const float inv = rsqrtf(block_sum(ss, red) / (float)D.d + D.eps);
    float* out = D.hid + (size_t)D.seq_ids[b] * D.d;
    for (int c = threadIdx.x; c < D.d; c += blockDim.x) out[c] = __ldcg(xr + c) * inv * D.g_final[c];
    __syncthreads();
  }
}

SPEC_DEV unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <int HD>
SPEC_DEV void attn_step(const PassDesc& D, const AttnArgs& at, unsigned char* smem) {
  const int nb = D.B * D.nkv, total = nb * at.n_split;
  for (int vb = blockIdx.x; vb < total; vb += gridDim.x) {
    atc::AttnTc<HD>::run(at, D.pps, D.attn_cnt, smem, vb % nb, vb / nb, false, D.smem_bytes);
    __syncthreads();
  }
}

template <int HD>
SPEC_DEV void attn_prefetch(const PassDesc& D, const AttnArgs& at) {
  const int nb = D.B * D.nkv, total = nb * at.n_split;
  for (int vb = blockIdx.x; vb < total; vb += gridDim.x) atc::AttnTc<HD>::prefetch(at, D.pps, vb % nb, vb / nb);
}

SPEC_DEV void grid_barrier(const PassDesc& D) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int* count = D.bar;
    unsigned int* gen = D.bar + 1;
    const unsigned int g = ld_acquire(gen);
    __threadfence();
    const unsigned int arrived = atomic_add_acq_rel(count, 1u);
    if (arrived == gridDim.x - 1) {
      *count = 0u;
      st_release(gen, g + 1u);
    } else {
      unsigned int it = 0;
      while (ld_acquire(gen) == g) {
        if (++it > (1u << 26)) {  // about a second or more: give up, let every CTA leave
          atomicExch(D.abort_flag, 1);
          set_error(D.err, SPEC_ERR_TIMEOUT);
          break;
        }
      }
    }
  }
  __syncthreads();
}

template <int HD>
__global__ void __launch_bounds__(MK_THREADS, 1) pass_kernel(PassDesc D) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Phase ph[2];
  __shared__ float red[32];
  const int n = 3 + 5 * D.L;
  if (threadIdx.x == 0) make_phase(D, 0, ph[0]);
  __syncthreads();
  for (int i = 0; i < n; ++i) {
    const Phase& cur = ph[i & 1];
    if (D.trace && threadIdx.x == 0) D.trace[((size_t)i * gridDim.x + blockIdx.x) * 6] = gtimer();
    if (cur.type == PH_EMBED) {
      embed_step(D);
    } else if (cur.type == PH_GEMV) {
      if ((int)blockIdx.x < cur.plan.grid) gemv_step(cur, D, smem, i);
    } else if (cur.type == PH_ATTN) {
      attn_step<HD>(D, cur.at, smem);
    } else {
      commit_step(D, red);
    }
    if (D.trace) {
      __syncthreads();
      if (threadIdx.x == 0) D.trace[((size_t)i * gridDim.x + blockIdx.x) * 6 + 3] = gtimer();
    }
    if (i + 1 < n) {
      __syncthreads();
      Phase& nxt = ph[(i + 1) & 1];
      if (threadIdx.x == 0) make_phase(D, i + 1, nxt);
      __syncthreads();
      // pull this CTA's share of the next step towards L2 before the barrier
      if (!D.prefetch) {
      } else if (nxt.type == PH_GEMV && (int)blockIdx.x < nxt.plan.grid) {
        tc::Sk<MK_WARPS> k{nxt.g, nxt.plan, nxt.map};
        k.bid = blockIdx.x;
        k.prefetch_slice(tc::unit_begin(blockIdx.x, nxt.plan), tc::unit_begin(blockIdx.x + 1, nxt.plan));
      } else if (nxt.type == PH_ATTN) {
        attn_prefetch<HD>(D, nxt.at);
      }
      if (D.trace) {
        __syncthreads();
        if (threadIdx.x == 0) D.trace[((size_t)i * gridDim.x + blockIdx.x) * 6 + 4] = gtimer();
      }
      grid_barrier(D);
      if (*(volatile int*)D.abort_flag) return;
    }
  }
}

size_t pass_smem(const PassDesc& D) {
  // largest projection plan of the pass, and the attention buffers
  size_t s = 0;
  const int M = D.B * D.R;
  const int Ks[3] = {D.d, D.nq * D.hd, D.ff};
  for (int K : Ks) {
    GemvArgs g = {};
    g.M = M; g.N = 16; g.K = K;
    s = std::max(s, tc::plan<MK_WARPS>(g, tc::MAP_PLAIN, D.nsm).smem);
  }
  const int qn = D.R * (D.nq / D.nkv);
  s = std::max(s, attention_tc_smem(D.hd, qn, D.R));
  const size_t merge = ((size_t)qn * D.n_split + 4) * 4 + (size_t)qn * D.n_split * D.hd * 4;
  if (merge <= 200 * 1024) s = std::max(s, merge);
  return s;
}

}  // namespace

bool pass_persistent_supported(int hd, int max_rows) { return (hd == 64 || hd == 128) && max_rows <= 8; }

int pass_persistent(const PassDesc& D, cudaStream_t st) {
  if (!pass_persistent_supported(D.hd, D.B * D.R)) return -2;
  const size_t smem = pass_smem(D);
  // dynamic + static shared memory must stay within the per-block opt-in limit
  constexpr size_t DYN_MAX = 227 * 1024 - 4096;
  if (smem > DYN_MAX) return -2;
  auto kern = D.hd == 128 ? pass_kernel<128> : pass_kernel<64>;
  static int attr[2] = {0, 0};
  int& state = attr[D.hd == 128 ? 1 : 0];
  if (state == 0)
    state = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DYN_MAX) == cudaSuccess ? 1 : -1;
  if (state < 0) return -2;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, MK_THREADS, smem) != cudaSuccess || per_sm < 1)
    return -2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(D.nsm);
  cfg.blockDim = dim3(MK_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  PassDesc Dl = D;
  Dl.smem_bytes = smem;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, Dl) == cudaSuccess ? 1 : -1;
}

}  // namespace spec
