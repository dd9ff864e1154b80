// draft.cu -- drafter-specific kernels and small pass helpers.
//
// The drafter is a light head on the target's last layer: it starts from the
// target's final hidden state and predicts future tokens autoregressively
// ("Accelerating Gemini Nano on Pixel with frozen multi-token prediction"
// (ai-news-spoon), section "The late-exit strategy"), reads the target's KV
// cache instead of keeping its own (section "Zero-copy architecture"), and
// scores its output through a clustered shortcut of 2048 centroids ("Gemma 4's
// MTP drafter explained" (molayo1419.me), section "What is different about
// Gemma 4's drafter?"; "Gemma 4 acceleration with MTP drafters"
// (cafe.daangn.com), section "MTP drafter internal optimisations": clustering
// in the embedder because the final logits are the bottleneck).
#include <math.h>

#include <algorithm>

#include "common.cuh"

namespace spec {

namespace {

SPEC_DEV float elem(const Mat& W, int K, long long row, int col) {
  if (W.dtype == DT_F32) return ((const float*)W.data)[row * K + col];
  if (W.dtype == DT_BF16) return __bfloat162float(((const __nv_bfloat16*)W.data)[row * K + col]);
  const uint8_t* c = (const uint8_t*)W.data + row * (K / 2);
  const int b = col >> 5, i = col & 31;
  const uint8_t byte = c[b * 16 + (i & 15)];
  const int code = i < 16 ? (byte & 15) : (byte >> 4);
  return __half2float(((const __half*)W.scales)[row * (K / 32) + b]) * (float)(code - 8);
}

__global__ void commit_hidden_kernel(int B, const int32_t* seq_ids, const int32_t* sel_row, const float* x,
                                     int d, const float* g, float eps, float* hid, const int* err) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  // a pass that recorded a device error commits nothing (its tail left
  // seq_len and pending as they were; the hidden state stays with them)
  if (err && *(const volatile int*)err) return;
  const int b = blockIdx.x;
  const float* xr = x + (size_t)sel_row[b] * d;
  float ss = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) ss = fmaf(xr[c], xr[c], ss);
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
  float* out = hid + (size_t)seq_ids[b] * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) out[c] = xr[c] * inv * g[c];
}

// Four consecutive elements of a weight row (col % 4 == 0).
SPEC_DEV void elem4(const Mat& W, int K, long long row, int col, float (&v)[4]) {
  if (W.dtype == DT_F32) {
    const float4 u = __ldg(reinterpret_cast<const float4*>((const float*)W.data + row * K + col));
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  } else if (W.dtype == DT_BF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>((const __nv_bfloat16*)W.data + row * K + col));
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = elem(W, K, row, col + i);
  }
}

// [N(h); N(E[tok])] of each row (one CTA per row, four columns a thread: d %
// 4 == 0), and the RoPE pairs of its query position.
__global__ void __launch_bounds__(1024) draft_input_kernel(DraftInArgs a) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, slot = a.seq_ids[b], d = a.d;
  const float* h = a.h_from_state ? a.h_prev + (size_t)slot * d : a.h_prev + (size_t)b * d;
  const int tok = a.j == 1 ? a.pending[slot] : a.drafts[b * a.k + a.j - 2];
  float sh = 0.f, se = 0.f;
  for (int c = 4 * threadIdx.x; c < d; c += 4 * blockDim.x) {
    const float4 hv = __ldcg(reinterpret_cast<const float4*>(h + c));
    float e[4];
    elem4(a.embed, d, tok, c, e);
    sh = fmaf(hv.x, hv.x, fmaf(hv.y, hv.y, fmaf(hv.z, hv.z, fmaf(hv.w, hv.w, sh))));
    se = fmaf(e[0], e[0], fmaf(e[1], e[1], fmaf(e[2], e[2], fmaf(e[3], e[3], se))));
  }
  const float ih = rsqrtf(block_sum(sh, red) / (float)d + a.eps);
  const float ie = rsqrtf(block_sum(se, red) / (float)d + a.eps);
  float* cat = a.cat + (size_t)b * 2 * d;
  for (int c = 4 * threadIdx.x; c < d; c += 4 * blockDim.x) {
    const float4 hv = __ldcg(reinterpret_cast<const float4*>(h + c));
    float e[4];
    elem4(a.embed, d, tok, c, e);
    const float hh[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cat[c + i] = hh[i] * ih * a.g_h[c + i];
      cat[d + c + i] = e[i] * ie * a.g_e[c + i];
    }
  }
  // the drafter's query for step j sits at the position of its input token
  const int pos = a.seq_len[slot] + a.j - 1;
  const double lt = log((double)a.theta);
  for (int j = threadIdx.x; j < a.hd / 2; j += blockDim.x) {
    double s, c;
    sincos((double)pos * exp(-2.0 * j / a.hd * lt), &s, &c);
    a.rope_cs[(size_t)b * a.hd + 2 * j] = (float)c;
    a.rope_cs[(size_t)b * a.hd + 2 * j + 1] = (float)s;
  }
}

// Top-C clusters of one row: the top_c largest packed (binary32 score, id)
// keys -- larger score first, lower cluster id on ties; the keys are distinct,
// so exactly top_c keys are >= the top_c-th largest. That key is found by a
// most-significant-digit-first radix select (8 passes of 8 bits: a shared
// histogram of the keys that still match the prefix, then the digit where the
// count from the top reaches the number still needed), and the keys at or
// above it are written in any order (the member scoring does not depend on
// it).
__global__ void __launch_bounds__(1024) topc_kernel(ClusterArgs a, int unused) {
  __shared__ int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need, s_out;
  grid_dep_wait();
  grid_dep_launch();
  (void)unused;
  const int b = blockIdx.x, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_prefix = 0ull;
    s_need = a.top_c;
    s_out = 0;
  }
  unsigned long long mask = 0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    for (int i = threadIdx.x; i < a.C; i += blockDim.x) {
      const unsigned long long key = pack_best(a.scores[(size_t)b * a.C + i], (uint32_t)i);
      if ((key & mask) == prefix) atomicAdd(&hist[(int)((key >> shift) & 255ull)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l sums bins 255 - 8l .. 248 - 8l (from the top), then a suffix
      // scan over the lanes finds the digit holding the need-th key
      int c[8], tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c[k] = hist[255 - 8 * lane - k];
        tot += c[k];
      }
      int incl = tot;  // keys in the bins above and including this lane's
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int need = s_need, above = incl - tot;
      if (above < need && need <= incl) {
        int run = above;
        for (int k = 0; k < 8; ++k) {
          if (run + c[k] >= need) {
            s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - k) << shift);
            s_need = need - run;
            break;
          }
          run += c[k];
        }
      }
    }
    mask |= 255ull << shift;
    __syncthreads();
  }
  const unsigned long long kth = s_prefix;  // the top_c-th largest key itself
  for (int i = threadIdx.x; i < a.C; i += blockDim.x) {
    const unsigned long long key = pack_best(a.scores[(size_t)b * a.C + i], (uint32_t)i);
    if (key >= kth) {
      const int slot = atomicAdd(&s_out, 1);
      if (slot < a.top_c) a.chosen[b * a.top_c + slot] = i;
    }
  }
}

// Score the member rows of one chosen cluster; the best (score, token id) of a
// row wins with the lower token id on ties. The last CTA writes the draft.
__global__ void __launch_bounds__(256) members_kernel(ClusterArgs a) {
  extern __shared__ float ub[];  // normalised drafter state [h]
  __shared__ float red[32];
  __shared__ unsigned long long wbest[8];
  __shared__ int last;
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, ci = blockIdx.y, h = a.h;
  const float* u = a.u + (size_t)b * h;
  float ss = 0.f;
  for (int c = threadIdx.x; c < h; c += blockDim.x) ss = fmaf(u[c], u[c], ss);
  const float inv = rsqrtf(block_sum(ss, red) / (float)h + a.eps);
  for (int c = threadIdx.x; c < h; c += blockDim.x) ub[c] = u[c] * inv * a.g_out[c];
  __syncthreads();
  const int cl = a.chosen[b * a.top_c + ci];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long best = 0ull;
  if (a.vocab.dtype == DT_BF16 && h == 256 && a.cs % 64 == 0) {
    // bf16 rows of 256: lane i holds elements 8i..8i+7 of the state and
    // loads its 16 bytes of each of the warp's rows, 8 rows in flight at a time
    float uv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) uv[i] = ub[8 * lane + i];
    const __nv_bfloat16* V = (const __nv_bfloat16*)a.vocab.data;
    for (int r0 = warp; r0 < a.cs; r0 += 64) {
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        q[j] = ldg_stream(V + ((long long)cl * a.cs + r0 + 8 * j) * 256 + 8 * lane);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t wv[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(uv[2 * i], bf16lo(wv[i]), acc);
          acc = fmaf(uv[2 * i + 1], bf16hi(wv[i]), acc);
        }
        acc = warp_sum(acc);
        const long long p = (long long)cl * a.cs + r0 + 8 * j;
        const unsigned long long key = pack_best(acc, (uint32_t)a.perm[p]);
        best = key > best ? key : best;
      }
    }
  } else {
    for (int r = warp; r < a.cs; r += 8) {
      const long long p = (long long)cl * a.cs + r;
      float acc = 0.f;
      for (int c = lane; c < h; c += 32) acc = fmaf(ub[c], elem(a.vocab, h, p, c), acc);
      acc = warp_sum(acc);
      const unsigned long long key = pack_best(acc, (uint32_t)a.perm[p]);
      best = key > best ? key : best;
    }
  }
  if (lane == 0) wbest[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0ull;
    for (int w = 0; w < 8; ++w) m = wbest[w] > m ? wbest[w] : m;
    atomicMax(&a.best[b], m);
    __threadfence();
    const unsigned int done = atomicAdd(a.tail.counter, 1u);
    last = done == gridDim.x * gridDim.y - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int bb = threadIdx.x; bb < a.B; bb += blockDim.x) {
    const unsigned long long k = volatile_load(a.best + bb);
    a.tail.draft_out[bb * a.tail.draft_ld + a.tail.draft_j] = (int32_t)best_index(k);
  }
  __syncthreads();
  for (int bb = threadIdx.x; bb < a.B; bb += blockDim.x) a.best[bb] = 0ull;
  if (threadIdx.x == 0) *a.tail.counter = 0u;
}

__global__ void inject_kernel(int B, int k, const int32_t* seq_ids, const int32_t* seq_len, int32_t* drafts,
                              const int32_t* ref, int ref_len, float alpha, const float* draws,
                              const int32_t* offsets, int vocab, int* err) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = threadIdx.x;
  if (t >= B * k) return;
  const int b = t / k, j = t % k + 1, slot = seq_ids[b];
  const int pos = seq_len[slot] + j;
  if (pos >= ref_len) {
    set_error(err, SPEC_ERR_REF);
    return;
  }
  const int g = ref[(size_t)slot * ref_len + pos];
  drafts[t] = draws[t] < alpha ? g : (int32_t)(((long long)g + offsets[t]) % vocab);
}

cudaLaunchConfig_t cfg_pdl(dim3 grid, dim3 block, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr) {
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

int commit_hidden(int B, const int32_t* seq_ids, const int32_t* sel_row, const float* x, int d,
                  const float* g_final, float eps, float* hid_state, const int* err, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = cfg_pdl(dim3(B), dim3(256), 0, st, at);
  return cudaLaunchKernelEx(&cfg, commit_hidden_kernel, B, seq_ids, sel_row, x, d, g_final, eps, hid_state,
                            err) == cudaSuccess ? 1 : -1;
}

int draft_input(const DraftInArgs& a, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  if (a.d % 4) return -1;
  const int threads = std::min(1024, std::max(64, (a.d / 4 + 31) / 32 * 32));
  cudaLaunchConfig_t cfg = cfg_pdl(dim3(a.B), dim3(threads), 0, st, at);
  return cudaLaunchKernelEx(&cfg, draft_input_kernel, a) == cudaSuccess ? 1 : -1;
}

void setup_draft_attributes() {}

int cluster_head(const ClusterArgs& a, cudaStream_t st) {
  if (a.top_c < 1 || a.top_c > a.C) return -1;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = cfg_pdl(dim3(a.B), dim3(1024), 0, st, at);
  if (cudaLaunchKernelEx(&cfg, topc_kernel, a, 0) != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg2 = cfg_pdl(dim3(a.B, a.top_c), dim3(256), (size_t)a.h * 4, st, at);
  if (cudaLaunchKernelEx(&cfg2, members_kernel, a) != cudaSuccess) return -1;
  return 2;
}

int inject_drafts(int B, int k, const int32_t* seq_ids, const int32_t* seq_len, int32_t* drafts,
                  const int32_t* ref, int ref_len, float alpha, const float* draws, const int32_t* offsets,
                  int vocab, int* err, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = cfg_pdl(dim3(1), dim3(((B * k + 31) / 32) * 32), 0, st, at);
  return cudaLaunchKernelEx(&cfg, inject_kernel, B, k, seq_ids, seq_len, drafts, ref, ref_len, alpha, draws,
                            offsets, vocab, err) == cudaSuccess ? 1 : -1;
}

// SM count of the current device (looked up once per device).
int num_sms() {
  static int n[MAX_DEVICES] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) dev = 0;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

}  // namespace spec
