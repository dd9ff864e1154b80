// moe.cu -- the mixture-of-experts FFN of a verify (or prefill) pass.
//
// A 26B mixture-of-experts target is one of the pages' targets ("Gemma 4
// acceleration: faster inference with multi-token prediction drafters"
// (cafe.daangn.com), section "MTP drafter internal optimisations": little gain
// at batch 1 because of routing, about 2.2x at batch 4-8); the pages do not
// define the layer. Here: router scores z = W_r . xn on the FFN's normalised
// input, each row's top_k experts by binary32 score (ties to the lower id),
// softmax weights over the chosen scores, and gated-GELU experts
// y = sum_j w_j * W_down,e_j (GELU(W_gate,e_j xn) * W_up,e_j xn).
//
// A verify pass of B*(k+1) rows touches each expert for the rows routed to
// it: the grouped kernels stream every used expert's weights once for all of
// its rows (the rows gathered into shared memory), and skip unused experts.
// Each row's expert outputs land in per-selection buffers that one kernel adds
// to the residual in selection order, so results do not depend on timing.
#include "common.cuh"

namespace spec {

namespace {

constexpr int ROWS_CHUNK = 8;  // rows of one expert multiplied per weight pass

__global__ void rmsnorm_rows_kernel(const float* x, int d, const float* g, float eps, float* xn) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const float* r = x + (size_t)blockIdx.x * d;
  float ss = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) ss = fmaf(r[c], r[c], ss);
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
  for (int c = threadIdx.x; c < d; c += blockDim.x) xn[(size_t)blockIdx.x * d + c] = r[c] * inv * g[c];
}

// One CTA: each row's top_k experts and weights; then, in row order, every
// expert's list of (row * top_k + slot) selections.
__global__ void moe_route_kernel(MoeArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) {
    const float* z = a.z + (size_t)m * a.E;
    int sel[8];
    float sc[8];
    for (int j = 0; j < a.K; ++j) {
      int best = -1;
      for (int e = 0; e < a.E; ++e) {
        bool taken = false;
        for (int i = 0; i < j; ++i) taken |= sel[i] == e;
        if (!taken && (best < 0 || z[e] > z[best])) best = e;
      }
      sel[j] = best;
      sc[j] = z[best];
    }
    const float mx = sc[0];  // the first choice holds the largest score
    float tot = 0.f;
    for (int j = 0; j < a.K; ++j) tot += expf(sc[j] - mx);
    for (int j = 0; j < a.K; ++j) {
      a.sel[m * a.K + j] = sel[j];
      a.wts[m * a.K + j] = expf(sc[j] - mx) / tot;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int e = 0; e < a.E; ++e) a.cnt[e] = 0;
    for (int m = 0; m < a.M; ++m)
      for (int j = 0; j < a.K; ++j) {
        const int e = a.sel[m * a.K + j];
        a.list[(size_t)e * a.M + a.cnt[e]++] = m * a.K + j;
      }
  }
}

template <typename WT>
SPEC_DEV void load8(const WT* p, float (&v)[8]);
template <>
SPEC_DEV void load8<float>(const float* p, float (&v)[8]) {
  const uint4 a = ldg_stream(p), b = ldg_stream(p + 4);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}
template <>
SPEC_DEV void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = ldg_stream(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
}

// dot products of weight row `wr` (length K) with the chunk's n rows in smem
// (rows at stride K), one result per row reduced over the warp
template <typename WT>
SPEC_DEV void warp_dots(const WT* wr, const float* xs, int K, int n, float (&acc)[ROWS_CHUNK]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < ROWS_CHUNK; ++r) acc[r] = 0.f;
  for (int c = lane * 8; c < K; c += 256) {
    float w[8];
    load8<WT>(wr + c, w);
#pragma unroll
    for (int r = 0; r < ROWS_CHUNK; ++r) {
      if (r < n) {
        const float* x = xs + (size_t)r * K + c;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r] = fmaf(w[i], x[i], acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < ROWS_CHUNK; ++r) acc[r] = warp_sum(acc[r]);
}

// CTA (e, tile): intermediate columns j = 8*tile + warp of expert e for every
// row routed to e: act[sel][j] = GELU(gate_j . xn) * (up_j . xn).
template <typename WT>
__global__ void __launch_bounds__(256) moe_gateup_kernel(MoeArgs a, const WT* wgu) {
  extern __shared__ __align__(16) float xs[];  // [ROWS_CHUNK][d]
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.x, j = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int n_all = a.cnt[e];
  if (n_all == 0) return;
  const WT* W = wgu + (size_t)e * 2 * a.ff * a.d;
  for (int r0 = 0; r0 < n_all; r0 += ROWS_CHUNK) {
    const int n = min(ROWS_CHUNK, n_all - r0);
    __syncthreads();
    for (int i = threadIdx.x; i < n * a.d; i += blockDim.x) {
      const int r = i / a.d, c = i - r * a.d;
      xs[i] = a.xn[(size_t)(a.list[(size_t)e * a.M + r0 + r] / a.K) * a.d + c];
    }
    __syncthreads();
    if (j >= a.ff) continue;
    float g[ROWS_CHUNK], u[ROWS_CHUNK];
    warp_dots<WT>(W + (size_t)j * a.d, xs, a.d, n, g);
    warp_dots<WT>(W + (size_t)(a.ff + j) * a.d, xs, a.d, n, u);
    if (lane == 0)
      for (int r = 0; r < n; ++r) {
        const float gl = 0.5f * g[r] * (1.f + erff(g[r] * 0.70710678118654752f));
        a.act[(size_t)a.list[(size_t)e * a.M + r0 + r] * a.ff + j] = gl * u[r];
      }
  }
}

// CTA (e, tile): output columns n = 8*tile + warp of expert e's down projection
// for every row routed to e: out[sel][n] = down_n . act[sel].
template <typename WT>
__global__ void __launch_bounds__(256) moe_down_kernel(MoeArgs a, const WT* wdown) {
  extern __shared__ __align__(16) float xs[];  // [ROWS_CHUNK][ff]
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.x, n = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int n_all = a.cnt[e];
  if (n_all == 0) return;
  const WT* W = wdown + (size_t)e * a.d * a.ff;
  for (int r0 = 0; r0 < n_all; r0 += ROWS_CHUNK) {
    const int nr = min(ROWS_CHUNK, n_all - r0);
    __syncthreads();
    for (int i = threadIdx.x; i < nr * a.ff; i += blockDim.x) {
      const int r = i / a.ff, c = i - r * a.ff;
      xs[i] = a.act[(size_t)a.list[(size_t)e * a.M + r0 + r] * a.ff + c];
    }
    __syncthreads();
    if (n >= a.d) continue;
    float o[ROWS_CHUNK];
    warp_dots<WT>(W + (size_t)n * a.ff, xs, a.ff, nr, o);
    if (lane == 0)
      for (int r = 0; r < nr; ++r) a.out[(size_t)a.list[(size_t)e * a.M + r0 + r] * a.d + n] = o[r];
  }
}

// x[m] += sum_j wts[m][j] * out[m*K + j], slots in order.
__global__ void moe_combine_kernel(MoeArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < a.K; ++j) acc = fmaf(a.wts[m * a.K + j], a.out[((size_t)m * a.K + j) * a.d + c], acc);
    a.x[(size_t)m * a.d + c] += acc;
  }
}

cudaLaunchConfig_t cfg_of(dim3 grid, dim3 block, size_t smem, cudaStream_t st, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

void setup_moe_attributes() {
  for (const void* f : {(const void*)moe_gateup_kernel<float>, (const void*)moe_gateup_kernel<__nv_bfloat16>,
                        (const void*)moe_down_kernel<float>, (const void*)moe_down_kernel<__nv_bfloat16>})
    cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

size_t moe_smem(int d, int ff) { return (size_t)ROWS_CHUNK * std::max(d, ff) * sizeof(float); }

// Normalised rows and router scores are computed by the caller (rmsnorm_rows,
// then a projection); this launches routing, the grouped experts and the
// combine. Returns the number of kernels, or -1.
int moe_ffn(const MoeArgs& a, const void* wgu_layer, const void* wdown_layer, int wdtype, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  int n = 0;
  cudaLaunchConfig_t c1 = cfg_of(dim3(1), dim3(256), 0, st, at);
  if (cudaLaunchKernelEx(&c1, moe_route_kernel, a) != cudaSuccess) return -1;
  ++n;
  cudaLaunchConfig_t c2 = cfg_of(dim3(a.E, (a.ff + 7) / 8), dim3(256), (size_t)ROWS_CHUNK * a.d * 4, st, at);
  cudaError_t e = wdtype == DT_F32 ? cudaLaunchKernelEx(&c2, moe_gateup_kernel<float>, a, (const float*)wgu_layer)
                                   : cudaLaunchKernelEx(&c2, moe_gateup_kernel<__nv_bfloat16>, a,
                                                        (const __nv_bfloat16*)wgu_layer);
  if (e != cudaSuccess) return -1;
  ++n;
  cudaLaunchConfig_t c3 = cfg_of(dim3(a.E, (a.d + 7) / 8), dim3(256), (size_t)ROWS_CHUNK * a.ff * 4, st, at);
  e = wdtype == DT_F32 ? cudaLaunchKernelEx(&c3, moe_down_kernel<float>, a, (const float*)wdown_layer)
                       : cudaLaunchKernelEx(&c3, moe_down_kernel<__nv_bfloat16>, a, (const __nv_bfloat16*)wdown_layer);
  if (e != cudaSuccess) return -1;
  ++n;
  cudaLaunchConfig_t c4 = cfg_of(dim3(a.M), dim3(256), 0, st, at);
  if (cudaLaunchKernelEx(&c4, moe_combine_kernel, a) != cudaSuccess) return -1;
  return n + 1;
}

int rmsnorm_rows(const float* x, int M, int d, const float* g, float eps, float* xn, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t c = cfg_of(dim3(M), dim3(256), 0, st, at);
  return cudaLaunchKernelEx(&c, rmsnorm_rows_kernel, x, d, g, eps, xn) == cudaSuccess ? 1 : -1;
}

}  // namespace spec
