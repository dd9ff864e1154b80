// accept_topm.cu -- lenient accept of a verify pass: a draft is kept while it
// ranks among the target's top_m tokens at its row.
//
// The pages name verification leniency -- relaxing the strict token match
// between draft and verification for some uses -- without a rule
// ("Accelerating Gemini Nano on Pixel with frozen multi-token prediction"
// (ai-news-spoon), section "Future directions"). Here draft d_j is accepted
// while every earlier draft was and d_j's rank among the binary32 logits of
// row j-1 (tokens with a higher logit, or the same logit and a lower index)
// is below top_m; the step emits the accepted drafts followed by the target's
// own choice at the first row not accepted past. top_m = 1 is greedy accept.
//
// The verify pass's LM head writes every row's logits; CTA (b, j, part)
// counts the tokens of one vocabulary part ranked before draft d_j; the last
// CTA to finish adds nothing more but walks every sequence's drafts, emits,
// and commits (length, pending token, counters) unless the pass recorded a
// device error, like the greedy tail.
#include "common.cuh"

namespace spec {

namespace {

__global__ void __launch_bounds__(256) topm_kernel(TopmArgs a) {
  __shared__ unsigned int red[8];
  __shared__ int last;
  grid_dep_wait();
  const int bj = blockIdx.x / a.S, part = blockIdx.x % a.S;
  const int b = bj / a.k, j = bj % a.k;
  const int d = a.drafts[b * a.k + j];
  unsigned int cnt = 0;
  if (d >= 0 && d < a.V) {
    const float* row = a.logits + (size_t)(b * (a.k + 1) + j) * a.V;
    const float fd = row[d];
    const int v0 = (int)(((long long)a.V * part) / a.S), v1 = (int)(((long long)a.V * (part + 1)) / a.S);
    for (int v = v0 + (int)threadIdx.x; v < v1; v += blockDim.x) {
      const float f = __ldcg(row + v);
      cnt += (f > fd || (f == fd && v < d)) ? 1u : 0u;
    }
  } else if (part == 0 && threadIdx.x == 0) {
    cnt = 0xffffu;  // an out-of-range draft is never accepted (the embedding recorded it)
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(FULL, cnt, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    atomicAdd(a.rank + bj, tot);
    __threadfence();
    last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int R = a.k + 1;
  const int err = a.err ? *(volatile int*)a.err : 0;
  for (int bb = threadIdx.x; bb < a.B; bb += blockDim.x) {
    const int slot = a.seq_ids[bb];
    int A = 0;
    while (A < a.k && *(volatile unsigned int*)(a.rank + bb * a.k + A) < (unsigned)a.top_m) ++A;
    const int t = (int)best_index(volatile_load(a.best + bb * R + A));
    for (int i = 0; i < R; ++i) a.out_tokens[bb * R + i] = i < A ? a.drafts[bb * a.k + i] : (i == A ? t : -1);
    a.n_emitted[bb] = A + 1;
    if (!err) {
      a.seq_len[slot] += A + 1;
      a.pending[slot] = t;
      a.stats[slot * 4 + 0] += 1;
      a.stats[slot * 4 + 1] += a.k;
      a.stats[slot * 4 + 2] += A;
      a.stats[slot * 4 + 3] += A + 1;
    }
    a.sel_row[bb] = bb * R + A;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.B * R; i += blockDim.x) a.best[i] = 0ull;
  for (int i = threadIdx.x; i < a.B * a.k; i += blockDim.x) a.rank[i] = 0u;
  if (threadIdx.x == 0) *a.counter = 0u;
}

}  // namespace

int topm_accept(const TopmArgs& a0, cudaStream_t st) {
  TopmArgs a = a0;
  if (a.k < 1 || a.B < 1) return -1;
  a.S = 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.k * a.S);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topm_kernel, a) == cudaSuccess ? 1 : -1;
}

}  // namespace spec
