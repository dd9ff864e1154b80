// attn.cu -- pass setup, RoPE + KV append, and causal attention of the
// verified rows over the paged KV cache.
//
// The target verifies all drafted positions in one forward pass ("Gemma 4's
// MTP drafter explained" (molayo1419.me), section "How does speculative
// decoding work?"); row i of a sequence sits at position seq_len + i and
// attends keys 0 .. seq_len + i, which include the keys of the rows before it
// appended in the same pass. The drafter's cross-attention uses the same
// kernels over the target's last-layer pages with keys 0 .. seq_len - 1 and no
// writes ("Accelerating Gemini Nano on Pixel with frozen multi-token
// prediction" (ai-news-spoon), section "Zero-copy architecture").
//
// Attention is split by KV page: one CTA per (sequence, KV head, page) scores
// all rows x GQA-group queries of that sequence against the page's 64 keys and
// writes an unnormalised partial (max, sum, o); a merge kernel combines the
// partials of each query with the usual log-sum-exp rescaling.
#include <math.h>

#include <algorithm>

#include "common.cuh"

namespace spec {

namespace {
constexpr int PAGE = 64;

SPEC_DEV float dequant_elem(const Mat& W, int K, long long row, int col) {
  if (W.dtype == DT_F32) return ((const float*)W.data)[row * K + col];
  if (W.dtype == DT_BF16) return __bfloat162float(((const __nv_bfloat16*)W.data)[row * K + col]);
  const uint8_t* c = (const uint8_t*)W.data + row * (K / 2);
  const int b = col >> 5, i = col & 31;
  const uint8_t byte = c[b * 16 + (i & 15)];
  const int code = i < 16 ? (byte & 15) : (byte >> 4);
  return __half2float(((const __half*)W.scales)[row * (K / 32) + b]) * (float)(code - 8);
}

// cos/sin of pos * theta^(-2j/hd), evaluated in double then rounded.
SPEC_DEV void rope_table_row(float* cs, int pos, int hd, float theta) {
  const double lt = log((double)theta);
  for (int j = threadIdx.x; j < hd / 2; j += blockDim.x) {
    const double ang = (double)pos * exp(-2.0 * j / hd * lt);
    double s, c;
    sincos(ang, &s, &c);
    cs[2 * j] = (float)c;
    cs[2 * j + 1] = (float)s;
  }
}

__global__ void embed_rows_kernel(RowsArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x, b = m / a.R, i = m % a.R;
  const int slot = a.seq_ids[b];
  int tok;
  if (a.mode == TAIL_PREFILL) tok = a.tokens[(size_t)b * a.tok_ld + i];
  else tok = i == 0 ? a.pending[slot] : a.tokens[b * (a.R - 1) + i - 1];
  if (tok < 0 || tok >= a.vocab) {
    if (threadIdx.x == 0) set_error(a.err, SPEC_ERR_TOKEN);
    tok = 0;
  }
  const int pos = a.seq_len[slot] + i;  // the row's cache slot
  int rpos = pos;                       // and its position (RoPE)
  if (a.parents) {
    // tree verify: row i > 0 is draft node i - 1; its depth below the root
    // gives its position, its ancestors (and itself, and the root) its mask
    unsigned int mask = 1u;
    int depth = 0;
    if (i > 0) {
      mask |= 1u << i;
      depth = 1;
      int x = a.parents[b * (a.R - 1) + i - 1];
      for (int guard = 0; x >= 0 && guard < 32; ++guard) {
        if (x >= i - 1) {  // parents must come earlier; a bad one is treated as the root
          if (threadIdx.x == 0) set_error(a.err, SPEC_ERR_TOKEN);
          break;
        }
        mask |= 1u << (x + 1);
        ++depth;
        x = a.parents[b * (a.R - 1) + x];
      }
    }
    rpos = a.seq_len[slot] + depth;
    if (threadIdx.x == 0) a.tree_mask[m] = mask;
  }
  if (threadIdx.x == 0) a.pos[m] = pos;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) a.x[(size_t)m * a.d + c] = dequant_elem(a.embed, a.d, tok, c);
  rope_table_row(a.rope_cs + (size_t)m * a.hd, rpos, a.hd, a.theta);
}

template <typename KT>
__global__ void rope_append_kernel(RopeAppendArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x, half = a.hd / 2;
  const int nqkv = (a.nq + 2 * a.nkv) * a.hd;
  float* row = a.qkv + (size_t)m * nqkv;
  const float* cs = a.rope_cs + (size_t)m * a.hd;
  const int pos = a.pos[m];
  const int slot = a.seq_ids[m / a.R];
  const int pidx = pos / PAGE;
  int page = -1;
  if (pidx < a.max_pages) page = a.block_table[(size_t)slot * a.max_pages + pidx];
  const bool ok = page >= 0 && page < a.n_pages;
  if (!ok && threadIdx.x == 0) set_error(a.err, SPEC_ERR_CAPACITY);
  KT* pool = (KT*)a.pool + (size_t)a.layer * a.layer_elems;
  // rotate q heads and k heads (rotate-half pairing), then store k and v
  for (int t = threadIdx.x; t < (a.nq + a.nkv) * half; t += blockDim.x) {
    const int h = t / half, j = t % half;
    float* v = row + h * a.hd;  // k heads follow the q heads
    const float c = cs[2 * j], s = cs[2 * j + 1];
    const float x0 = v[j], x1 = v[j + half];
    const float y0 = x0 * c - x1 * s, y1 = x1 * c + x0 * s;
    v[j] = y0;
    v[j + half] = y1;
    if (h >= a.nq && ok) {
      const int kh = h - a.nq;
      KT* kp = pool + ((((size_t)page * 2 + 0) * a.nkv + kh) * PAGE + pos % PAGE) * a.hd;
      store_kv(kp + j, y0);
      store_kv(kp + j + half, y1);
    }
  }
  if (ok)
    for (int t = threadIdx.x; t < a.nkv * a.hd; t += blockDim.x) {
      const int kh = t / a.hd, i = t % a.hd;
      KT* vp = pool + ((((size_t)page * 2 + 1) * a.nkv + kh) * PAGE + pos % PAGE) * a.hd;
      store_kv(vp + i, row[(a.nq + a.nkv) * a.hd + t]);
    }
}

// One CTA per (sequence b, KV head, page). Keys are staged in fp32 with a
// one-float row pad so that lanes reading different keys hit different banks.
template <typename KT>
__global__ void __launch_bounds__(256) attn_page_kernel(AttnArgs a) {
  extern __shared__ __align__(16) float sm[];
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x / a.nkv, kvh = blockIdx.x % a.nkv, pg = blockIdx.y;
  const int slot = a.seq_ids[b];
  const int L0 = a.seq_len[slot];
  const int lmax = L0 + a.R - 1 + a.key_extra;  // keys of the last row
  const int key0 = pg * PAGE;
  if (key0 >= lmax) return;
  const int page = a.block_table[(size_t)slot * a.max_pages + pg];
  if (page < 0 || page >= a.n_pages) {
    if (threadIdx.x == 0) set_error(a.err, SPEC_ERR_CAPACITY);
    return;
  }
  const int hd = a.hd, G = a.nq / a.nkv, QN = a.R * G;
  const int kst = hd + 1;
  float* Ks = sm;                    // [64][hd+1]
  float* Vs = Ks + PAGE * kst;       // [64][hd]
  float* Qs = Vs + PAGE * hd;        // [QN][hd]
  const KT* base = (const KT*)a.pool + (size_t)a.layer * a.layer_elems;
  const KT* kp = base + (((size_t)page * 2 + 0) * a.nkv + kvh) * PAGE * hd;
  const KT* vp = base + (((size_t)page * 2 + 1) * a.nkv + kvh) * PAGE * hd;
  const int nk = min(PAGE, lmax - key0);
  for (int t = threadIdx.x; t < nk * hd; t += blockDim.x) {
    const int j = t / hd, i = t % hd;
    Ks[j * kst + i] = load_kv(kp + t);
    Vs[t] = load_kv(vp + t);
  }
  // query q = i*G + g is head kvh*G + g of row b*R + i
  for (int t = threadIdx.x; t < QN * hd; t += blockDim.x) {
    const int q = t / hd, d = t % hd, i = q / G, g = q % G;
    const int m = b * a.R + i, h = kvh * G + g;
    const float* qr = a.q + (size_t)m * a.ldq + h * hd;
    float v = qr[d];
    if (a.rope_cs) {
      const float* cs = a.rope_cs + (size_t)m * hd;
      const int half = hd / 2, j = d % half;
      const float c = cs[2 * j], s = cs[2 * j + 1];
      v = d < half ? qr[d] * c - qr[d + half] * s : qr[d] * c + qr[d - half] * s;
    }
    Qs[t] = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float scale = rsqrtf((float)hd);
  for (int q = warp; q < QN; q += blockDim.x >> 5) {
    const int i = q / G, g = q % G;
    const int nkeys = L0 + i + a.key_extra;  // keys [0, nkeys)
    const int valid = min(PAGE, nkeys - key0);
    if (valid <= 0) continue;
    const unsigned int tmask = a.tree_mask ? a.tree_mask[b * a.R + i] : ~0u;
    const float* qv = Qs + q * hd;
    float s[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = lane + 32 * c;
      float acc = 0.f;
      if (j < valid && tree_visible(tmask, L0, key0 + j)) {
        const float* kr = Ks + j * kst;
        for (int d = 0; d < hd; ++d) acc = fmaf(qv[d], kr[d], acc);
        s[c] = acc * scale;
      } else {
        s[c] = -INFINITY;
      }
    }
    const float mx = warp_max(fmaxf(s[0], s[1]));
    const float p0 = s[0] == -INFINITY ? 0.f : __expf(s[0] - mx);
    const float p1 = s[1] == -INFINITY ? 0.f : __expf(s[1] - mx);
    const float l = warp_sum(p0 + p1);
    const int m = b * a.R + i, h = kvh * G + g;
    const size_t pidx = ((size_t)m * a.nq + h) * a.n_split + pg;
    for (int d = lane; d < hd; d += 32) {
      float o = 0.f;
      for (int j = 0; j < valid; ++j) {
        const float pj = __shfl_sync(FULL, j < 32 ? p0 : p1, j & 31);
        o = fmaf(pj, Vs[j * hd + d], o);
      }
      a.part_o[pidx * hd + d] = o;
    }
    if (lane == 0) {
      a.part_ml[pidx * 2 + 0] = mx;
      a.part_ml[pidx * 2 + 1] = l;
    }
  }
}

// One CTA per (sequence, layer): the accepted path's rows j = 1..A move from
// slot L0 + path[j] to L0 + j, in order (path[j] >= j, so no row is
// overwritten before it is read). Both planes, every KV head.
__global__ void tree_move_kernel(TreeMoveArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  if (a.err && *(const volatile int*)a.err) return;
  const int b = blockIdx.x, l = blockIdx.y;
  const int slot = a.seq_ids[b], n = a.n_emitted[b], A = n - 1;
  const int L0 = a.seq_len[slot] - n;
  char* base = (char*)a.pool + (size_t)l * a.layer_elems * a.kv_bytes;
  const int row_bytes = a.hd * a.kv_bytes;
  for (int j = 1; j <= A; ++j) {
    const int src = a.path[b * a.path_ld + j];
    if (src == j) continue;
    const int ps = L0 + src, pd = L0 + j;
    const int gs = a.block_table[(size_t)slot * a.max_pages + ps / PAGE];
    const int gd = a.block_table[(size_t)slot * a.max_pages + pd / PAGE];
    if (gs < 0 || gs >= a.n_pages || gd < 0 || gd >= a.n_pages) continue;  // recorded by the pass already
    for (int e = threadIdx.x; e < 2 * a.nkv * row_bytes / 4; e += blockDim.x) {
      const int w = e % (row_bytes / 4), ph = e / (row_bytes / 4), plane = ph / a.nkv, h = ph % a.nkv;
      const size_t so = ((((size_t)gs * 2 + plane) * a.nkv + h) * PAGE + ps % PAGE) * row_bytes;
      const size_t dof = ((((size_t)gd * 2 + plane) * a.nkv + h) * PAGE + pd % PAGE) * row_bytes;
      reinterpret_cast<uint32_t*>(base + dof)[w] = reinterpret_cast<const uint32_t*>(base + so)[w];
    }
    __syncthreads();
  }
}

// out[m][h*hd + d] = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M)
__global__ void attn_merge_kernel(AttnArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x, h = blockIdx.y;
  const int b = m / a.R, i = m % a.R;
  const int nkeys = a.seq_len[a.seq_ids[b]] + i + a.key_extra;
  const int np = min((nkeys + PAGE - 1) / PAGE, a.n_split);
  const size_t base = ((size_t)m * a.nq + h) * a.n_split;
  float M = -INFINITY;
  for (int s = 0; s < np; ++s) M = fmaxf(M, a.part_ml[(base + s) * 2]);
  float L = 0.f;
  for (int s = 0; s < np; ++s) L += a.part_ml[(base + s) * 2 + 1] * __expf(a.part_ml[(base + s) * 2] - M);
  for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
    float o = 0.f;
    for (int s = 0; s < np; ++s) o += a.part_o[(base + s) * a.hd + d] * __expf(a.part_ml[(base + s) * 2] - M);
    a.out[(size_t)m * a.nq * a.hd + h * a.hd + d] = np > 0 ? o / L : 0.f;
  }
}

cudaLaunchConfig_t pdl_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

int embed_rows(const RowsArgs& a, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(a.B * a.R), dim3(256), 0, st, at);
  return cudaLaunchKernelEx(&cfg, embed_rows_kernel, a) == cudaSuccess ? 1 : -1;
}

int rope_append(const RopeAppendArgs& a, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(a.M), dim3(256), 0, st, at);
  cudaError_t e = a.kv_dtype == DT_F32 ? cudaLaunchKernelEx(&cfg, rope_append_kernel<float>, a)
                                       : cudaLaunchKernelEx(&cfg, rope_append_kernel<__nv_bfloat16>, a);
  return e == cudaSuccess ? 1 : -1;
}

int tree_move(const TreeMoveArgs& a, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(a.B, a.L), dim3(256), 0, st, at);
  return cudaLaunchKernelEx(&cfg, tree_move_kernel, a) == cudaSuccess ? 1 : -1;
}

size_t attention_smem(int hd, int qn) { return (size_t)(PAGE * (hd + 1) + PAGE * hd + qn * hd) * 4; }

void setup_attn_attributes() {
  cudaFuncSetAttribute(attn_page_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(attn_page_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

int attention(const AttnArgs& a, cudaStream_t st) {
  const int QN = a.R * (a.nq / a.nkv);
  const size_t smem = attention_smem(a.hd, QN);
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(a.B * a.nkv, a.n_split), dim3(256), smem, st, at);
  cudaError_t e = a.kv_dtype == DT_F32 ? cudaLaunchKernelEx(&cfg, attn_page_kernel<float>, a)
                                       : cudaLaunchKernelEx(&cfg, attn_page_kernel<__nv_bfloat16>, a);
  if (e != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg2 = pdl_cfg(dim3(a.B * a.R, a.nq), dim3(std::min(a.hd, 128)), 0, st, at);
  if (cudaLaunchKernelEx(&cfg2, attn_merge_kernel, a) != cudaSuccess) return -1;
  return 2;
}

}  // namespace spec
