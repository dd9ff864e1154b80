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

// One CTA: a warp per row picks its top_k experts (a warp argmax per pick,
// binary32 scores, ties to the lower id) and their softmax weights; then a
// warp per expert lists, in row order, the selections (row * top_k + slot)
// routed to it, taking ballots over 32 selections at a time.
__global__ void __launch_bounds__(1024) moe_route_kernel(MoeArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int m = warp; m < a.M; m += nw) {
    const float* z = a.z + (size_t)m * a.E;
    unsigned long long taken[4] = {0ull, 0ull, 0ull, 0ull};  // E <= 256
    float sc[8];
    int sel[8];
    for (int j = 0; j < a.K; ++j) {
      unsigned long long best = 0ull;
      for (int e = lane; e < a.E; e += 32)
        if (!((taken[e >> 6] >> (e & 63)) & 1ull)) {
          const unsigned long long key = pack_best(z[e], (uint32_t)e);
          best = key > best ? key : best;
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(FULL, best, o);
        best = other > best ? other : best;
      }
      const int e = (int)best_index(best);
      taken[e >> 6] |= 1ull << (e & 63);
      sel[j] = e;
      sc[j] = z[e];
    }
    if (lane == 0) {
      const float mx = sc[0];  // the first pick holds the largest score
      float tot = 0.f;
      for (int j = 0; j < a.K; ++j) tot += expf(sc[j] - mx);
      for (int j = 0; j < a.K; ++j) {
        a.sel[m * a.K + j] = sel[j];
        a.wts[m * a.K + j] = expf(sc[j] - mx) / tot;
      }
    }
  }
  __syncthreads();
  const int total = a.M * a.K;
  for (int e = warp; e < a.E; e += nw) {
    int n = 0;
    for (int i0 = 0; i0 < total; i0 += 32) {
      const int i = i0 + lane;
      const bool hit = i < total && a.sel[i] == e;
      const unsigned bal = __ballot_sync(FULL, hit);
      if (hit) a.list[(size_t)e * a.M + n + __popc(bal & ((1u << lane) - 1u))] = i;
      n += __popc(bal);
    }
    if (lane == 0) a.cnt[e] = n;
  }
}

// Eight consecutive weights as loaded (raw bits), widened to fp32 only when
// they are multiplied, so that many loads can be in flight in few registers.
template <typename WT>
struct Raw8;
template <>
struct Raw8<float> {
  uint4 lo, hi;
  SPEC_DEV void load(const float* p) {
    lo = ldg_stream(p);
    hi = ldg_stream(p + 4);
  }
  SPEC_DEV float operator[](int i) const {
    const uint4& q = i < 4 ? lo : hi;
    const int j = i & 3;
    return __uint_as_float(j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w);
  }
};
template <>
struct Raw8<__nv_bfloat16> {
  uint4 q;
  SPEC_DEV void load(const __nv_bfloat16* p) { q = ldg_stream(p); }
  SPEC_DEV float operator[](int i) const {
    const uint32_t w = (i >> 1) == 0 ? q.x : (i >> 1) == 1 ? q.y : (i >> 1) == 2 ? q.z : q.w;
    return (i & 1) ? bf16hi(w) : bf16lo(w);
  }
};

// Dot products of NW weight rows wr[w] (length K, K % 8 == 0) with the chunk's
// n rows in smem (rows at stride K), one result per (weight row, row) reduced
// over the warp. Each lane keeps U loads of 8 weights per weight row in flight
// before it multiplies, so that a CTA has enough bytes outstanding to stream,
// and each shared-memory read of the rows serves NW weight rows.
template <typename WT, int NW, int U>
SPEC_DEV void warp_dots(const WT* const (&wr)[NW], const float* xs, int K, int n,
                        float (&acc)[NW][ROWS_CHUNK]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 0; w < NW; ++w)
#pragma unroll
    for (int r = 0; r < ROWS_CHUNK; ++r) acc[w][r] = 0.f;
  for (int c0 = lane * 8; c0 < K; c0 += 256 * U) {
    Raw8<WT> v[NW][U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + u * 256 < K)
#pragma unroll
        for (int w = 0; w < NW; ++w) v[w][u].load(wr[w] + c0 + u * 256);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c0 + u * 256 >= K) break;
#pragma unroll
      for (int r = 0; r < ROWS_CHUNK; ++r) {
        if (r < n) {
          const float4* x = reinterpret_cast<const float4*>(xs + (size_t)r * K + c0 + u * 256);
          const float4 x0 = x[0], x1 = x[1];
          const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[w][r] = fmaf(v[w][u][i], xv[i], acc[w][r]);
        }
      }
    }
  }
#pragma unroll
  for (int w = 0; w < NW; ++w)
#pragma unroll
    for (int r = 0; r < ROWS_CHUNK; ++r) acc[w][r] = warp_sum(acc[w][r]);
}

// Copies n (<= ROWS_CHUNK) rows of `width` floats (width % 4 == 0) into xs:
// row r of the chunk is src row list[r] / div. The row numbers go through shared
// memory first and each thread issues its float4 loads four at a time, so that
// the copy costs a few memory latencies, not one per element.
SPEC_DEV void gather_rows(float* xs, int* rows_s, const float* src, const int* list, int div, int n, int width) {
  if ((int)threadIdx.x < n) rows_s[threadIdx.x] = list[threadIdx.x] / div;
  __syncthreads();
  const int w4 = width >> 2, total = n * w4;
  const float4* s4 = reinterpret_cast<const float4*>(src);
  float4* x4 = reinterpret_cast<float4*>(xs);
  for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < total) {
        const int r = i / w4;
        v[u] = s4[(size_t)rows_s[r] * w4 + (i - r * w4)];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u * blockDim.x < total) x4[i0 + u * blockDim.x] = v[u];
  }
}

// Expert kernels: CTA (e, tile) owns 64 output columns of expert e and covers
// every row routed to e; warp w takes, in each of 8 / GH iterations, columns
// c_h = 64*tile + 8*GH*i + 8*h + w for h < GH. GH columns share one pass over
// the rows in shared memory, with U loads per weight row in flight (bf16; one
// for fp32 weights, whose raw bits take twice the registers).
constexpr int GU_GH = 2, GU_U = 2;    // gate/up: 4 weight rows per warp pass
constexpr int DN_GH = 2, DN_U = 4;    // down: 2 weight rows per warp pass

// act[sel][j] = GELU(gate_j . xn[row]) * (up_j . xn[row]) for the intermediate
// columns j of expert e. Rows are gathered once per 64 columns (512 KB of bf16
// gate and up rows at d = 2048).
template <typename WT>
__global__ void __launch_bounds__(256, 2) moe_gateup_kernel(MoeArgs a, const WT* wgu) {
  extern __shared__ __align__(16) float xs[];  // [ROWS_CHUNK][d]
  __shared__ int rows_s[ROWS_CHUNK];
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.x, lane = threadIdx.x & 31;
  const int n_all = a.cnt[e];
  if (n_all == 0) return;
  const WT* W = wgu + (size_t)e * 2 * a.ff * a.d;
  for (int r0 = 0; r0 < n_all; r0 += ROWS_CHUNK) {
    const int n = min(ROWS_CHUNK, n_all - r0);
    __syncthreads();
    gather_rows(xs, rows_s, a.xn, a.list + (size_t)e * a.M + r0, a.K, n, a.d);
    __syncthreads();
    for (int i = 0; i < 8 / GU_GH; ++i) {
      const int c0 = blockIdx.y * 64 + i * 8 * GU_GH + (threadIdx.x >> 5);
      if (c0 >= a.ff) break;
      int col[GU_GH];
      const WT* rows[2 * GU_GH];
#pragma unroll
      for (int h = 0; h < GU_GH; ++h) {
        col[h] = c0 + 8 * h < a.ff ? c0 + 8 * h : -1;
        const int j = col[h] < 0 ? c0 : col[h];
        rows[2 * h] = W + (size_t)j * a.d;
        rows[2 * h + 1] = W + (size_t)(a.ff + j) * a.d;
      }
      float gu[2 * GU_GH][ROWS_CHUNK];
      warp_dots<WT, 2 * GU_GH, sizeof(WT) == 2 ? GU_U : 1>(rows, xs, a.d, n, gu);
      if (lane == 0)
        for (int r = 0; r < n; ++r) {
          float* act = a.act + (size_t)a.list[(size_t)e * a.M + r0 + r] * a.ff;
#pragma unroll
          for (int h = 0; h < GU_GH; ++h)
            if (col[h] >= 0) {
              const float g = gu[2 * h][r];
              act[col[h]] = 0.5f * g * (1.f + erff(g * 0.70710678118654752f)) * gu[2 * h + 1][r];
            }
        }
    }
  }
}

// out[sel][c] = down_c . act[sel] for the output columns c of expert e.
template <typename WT>
__global__ void __launch_bounds__(256, 2) moe_down_kernel(MoeArgs a, const WT* wdown) {
  extern __shared__ __align__(16) float xs[];  // [ROWS_CHUNK][ff]
  __shared__ int rows_s[ROWS_CHUNK];
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.x, lane = threadIdx.x & 31;
  const int n_all = a.cnt[e];
  if (n_all == 0) return;
  const WT* W = wdown + (size_t)e * a.d * a.ff;
  for (int r0 = 0; r0 < n_all; r0 += ROWS_CHUNK) {
    const int nr = min(ROWS_CHUNK, n_all - r0);
    __syncthreads();
    gather_rows(xs, rows_s, a.act, a.list + (size_t)e * a.M + r0, 1, nr, a.ff);
    __syncthreads();
    for (int i = 0; i < 8 / DN_GH; ++i) {
      const int c0 = blockIdx.y * 64 + i * 8 * DN_GH + (threadIdx.x >> 5);
      if (c0 >= a.d) break;
      int col[DN_GH];
      const WT* rows[DN_GH];
#pragma unroll
      for (int h = 0; h < DN_GH; ++h) {
        col[h] = c0 + 8 * h < a.d ? c0 + 8 * h : -1;
        rows[h] = W + (size_t)(col[h] < 0 ? c0 : col[h]) * a.ff;
      }
      float o[DN_GH][ROWS_CHUNK];
      warp_dots<WT, DN_GH, sizeof(WT) == 2 ? DN_U : 1>(rows, xs, a.ff, nr, o);
      if (lane == 0)
        for (int r = 0; r < nr; ++r) {
          float* out = a.out + (size_t)a.list[(size_t)e * a.M + r0 + r] * a.d;
#pragma unroll
          for (int h = 0; h < DN_GH; ++h)
            if (col[h] >= 0) out[col[h]] = o[h][r];
        }
    }
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
  cudaLaunchConfig_t c1 = cfg_of(dim3(1), dim3(1024), 0, st, at);
  if (cudaLaunchKernelEx(&c1, moe_route_kernel, a) != cudaSuccess) return -1;
  ++n;
  cudaLaunchConfig_t c2 = cfg_of(dim3(a.E, (a.ff + 63) / 64), dim3(256), (size_t)ROWS_CHUNK * a.d * 4, st, at);
  cudaError_t e = wdtype == DT_F32 ? cudaLaunchKernelEx(&c2, moe_gateup_kernel<float>, a, (const float*)wgu_layer)
                                   : cudaLaunchKernelEx(&c2, moe_gateup_kernel<__nv_bfloat16>, a,
                                                        (const __nv_bfloat16*)wgu_layer);
  if (e != cudaSuccess) return -1;
  ++n;
  cudaLaunchConfig_t c3 = cfg_of(dim3(a.E, (a.d + 63) / 64), dim3(256), (size_t)ROWS_CHUNK * a.ff * 4, st, at);
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
