// gemv_tc.cu -- weight-streaming projection for bf16 weights on the tensor
// cores (mma.sync m16n8k16, fp32 accumulate), for M <= 8 rows per pass.
//
// The verify pass reads every weight once for the k+1 rows of each sequence
// ("Gemma 4's MTP drafter explained" (molayo1419.me), section "Why is
// generating one token at a time slow?"), so this kernel is bound by HBM: the
// tensor cores only remove the per-element ALU cost of the CUDA-core version.
//
// Fragments. A warp owns a 16-row weight tile. Lane (g = lane/4, c = lane%4)
// loads 16 bytes (8 consecutive bf16) of tile rows g and g+8 per 32-column
// step; those 8 columns feed two k16 MMAs through a fixed permutation of the
// reduction index (k-slot 2c+j <-> column 8c+j, 2c+8+j <-> 8c+2+j, then the
// next 4 columns), and the activation fragment of row n = g is the same 16
// bytes of X[g] in shared memory. The output fragment holds rows g and g+8 of
// the tile for m = 2c, 2c+1, so a pair of weight rows that must meet in the
// epilogue (gate/up of a GELU-gated FFN) is mapped to g and g+8.
//
// Precision. X is held as bf16 hi + lo (x = hi + lo to 2^-17 relative) and
// each step runs two MMAs, so the result matches an fp32-activation dot
// product of the exact bf16 weights. Each row's result depends only on that
// row and X, never on M.
//
// Work split. Persistent CTAs of 16 warps; CTA c owns a balanced range of row
// tiles. When a CTA has fewer tiles than warps, K is cut into slices and the
// slice partials are added in a fixed order; when X does not fit in shared
// memory, K is staged in chunks (each chunk a further set of slices).
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "tail.cuh"

namespace spec {

namespace {

constexpr int TW = 16;                  // warps per CTA
constexpr int XPAD = 32;                // bf16 pad per staged row (64 B): conflict-free 16-byte reads
constexpr int SMEM_MAX = 227 * 1024;

enum { MAP_PLAIN = 0, MAP_PAIR = 1 };

struct TcPlan {
  int tiles, grid, tiles_cta, kc, n_kc, s_sub, S;
  size_t smem;
};

SPEC_DEV void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

SPEC_DEV uint32_t bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct Tc {
  const GemvArgs& a;
  TcPlan p;
  int map;
  uint16_t *xhi, *xlo;
  float* part;
  float* inv_rms;
  unsigned long long* best;
  int* flag;
  int xs;  // staged row stride (elements)

  SPEC_DEV int row_g(int t, int g) const { return map == MAP_PAIR ? 8 * t + g : 16 * t + g; }
  SPEC_DEV int row_g8(int t, int g) const { return map == MAP_PAIR ? a.geglu_half + 8 * t + g : 16 * t + 8 + g; }
  SPEC_DEV bool ok_g(int t, int g) const { return map == MAP_PAIR ? 8 * t + g < a.geglu_half : 16 * t + g < a.N; }
  SPEC_DEV bool ok_g8(int t, int g) const {
    return map == MAP_PAIR ? 8 * t + g < a.geglu_half : 16 * t + 8 + g < a.N;
  }

  SPEC_DEV void norms() {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (w < 8) {
      float ss = 0.f;
      if (w < a.M)
        for (int c = lane * 4; c < a.K; c += 128) {
          const float4 v = *reinterpret_cast<const float4*>(a.X + (size_t)w * a.ldx + c);
          ss = fmaf(v.x, v.x, ss);
          ss = fmaf(v.y, v.y, ss);
          ss = fmaf(v.z, v.z, ss);
          ss = fmaf(v.w, v.w, ss);
        }
      ss = warp_sum(ss);
      if (lane == 0) inv_rms[w] = a.gain ? rsqrtf(ss / (float)a.K + a.eps) : 1.f;
    }
    __syncthreads();
  }

  // Stage X[:, k0 : k0+kc) as bf16 hi/lo planes (rows >= M are zero).
  SPEC_DEV void stage(int k0, int kc) {
    const int per_row = kc / 8;
    for (int idx = threadIdx.x; idx < 8 * per_row; idx += blockDim.x) {
      const int m = idx / per_row, c8 = (idx - m * per_row) * 8;
      const int col = k0 + c8;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
      if (m < a.M && col < a.K) {
        const float4 u0 = *reinterpret_cast<const float4*>(a.X + (size_t)m * a.ldx + col);
        const float4 u1 = *reinterpret_cast<const float4*>(a.X + (size_t)m * a.ldx + col + 4);
        v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
        v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
        if (a.gain) {
          const float s = inv_rms[m];
          const float4 g0 = *reinterpret_cast<const float4*>(a.gain + col);
          const float4 g1 = *reinterpret_cast<const float4*>(a.gain + col + 4);
          v[0] *= s * g0.x; v[1] *= s * g0.y; v[2] *= s * g0.z; v[3] *= s * g0.w;
          v[4] *= s * g1.x; v[5] *= s * g1.y; v[6] *= s * g1.z; v[7] *= s * g1.w;
        }
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
        hi[i] = bf16x2(v[2 * i], v[2 * i + 1]);
        lo[i] = bf16x2(v[2 * i] - __bfloat162float(h0), v[2 * i + 1] - __bfloat162float(h1));
      }
      *reinterpret_cast<uint4*>(xhi + m * xs + c8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(xlo + m * xs + c8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }

  // One task: tile t, k-steps [s0, s1) of the staged chunk (32 columns each).
  SPEC_DEV void task(int t, int k0, int s0, int s1, float (&c)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const bool vg = ok_g(t, g), vg8 = ok_g8(t, g);
    const __nv_bfloat16* W = (const __nv_bfloat16*)a.W.data;
    const __nv_bfloat16* rg = W + (size_t)(vg ? row_g(t, g) : 0) * a.K + k0 + 8 * q;
    const __nv_bfloat16* rg8 = W + (size_t)(vg8 ? row_g8(t, g) : 0) * a.K + k0 + 8 * q;
    const uint16_t* bh = xhi + g * xs + 8 * q;
    const uint16_t* bl = xlo + g * xs + 8 * q;
    constexpr int U = 4;
    uint4 wa[U], wb[U];
    int st = s0;
    auto load = [&](int base) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int s = base + u;
        wa[u] = (vg && s < s1) ? ldg_stream(rg + s * 32) : make_uint4(0, 0, 0, 0);
        wb[u] = (vg8 && s < s1) ? ldg_stream(rg8 + s * 32) : make_uint4(0, 0, 0, 0);
      }
    };
    load(st);
    while (st < s1) {
      uint4 ca[U], cb[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ca[u] = wa[u];
        cb[u] = wb[u];
      }
      const int cur = st;
      st += U;
      if (st < s1) load(st);  // next group in flight while this one is used
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int s = cur + u;
        if (s >= s1) break;
        const uint4 xh = *reinterpret_cast<const uint4*>(bh + s * 32);
        const uint4 xl = *reinterpret_cast<const uint4*>(bl + s * 32);
        mma16816(c, ca[u].x, cb[u].x, ca[u].y, cb[u].y, xh.x, xh.y);
        mma16816(c, ca[u].x, cb[u].x, ca[u].y, cb[u].y, xl.x, xl.y);
        mma16816(c, ca[u].z, cb[u].z, ca[u].w, cb[u].w, xh.z, xh.w);
        mma16816(c, ca[u].z, cb[u].z, ca[u].w, cb[u].w, xl.z, xl.w);
      }
    }
  }

  SPEC_DEV void epilogue(int t, const float (&c)[4], unsigned long long (&mybest)[2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int m0 = 2 * q, m1 = 2 * q + 1;
    if (map == MAP_PAIR) {
      if (!ok_g(t, g)) return;
      const int j = 8 * t + g;
      auto gl = [](float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); };
      if (m0 < a.M) a.Y[(size_t)m0 * a.ldy + j] = gl(c[0]) * c[2];
      if (m1 < a.M) a.Y[(size_t)m1 * a.ldy + j] = gl(c[1]) * c[3];
      return;
    }
    const int rows[2] = {row_g(t, g), row_g8(t, g)};
    const bool oks[2] = {ok_g(t, g), ok_g8(t, g)};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!oks[h]) continue;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = 2 * q + i;
        if (m >= a.M) continue;
        const float v = c[2 * h + i];
        float* y = a.Y ? a.Y + (size_t)m * a.ldy + rows[h] : nullptr;
        if (a.epi == EPI_STORE) *y = v;
        else if (a.epi == EPI_ADD) *y += v;
        else {
          if (y) *y = v;
          const unsigned long long key = pack_best(v, (uint32_t)rows[h]);
          mybest[i] = key > mybest[i] ? key : mybest[i];
        }
      }
    }
  }

  SPEC_DEV void run() {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cta = blockIdx.x;
    const int t0 = (int)(((long long)cta * p.tiles) / p.grid), t1 = (int)(((long long)(cta + 1) * p.tiles) / p.grid);
    const int nt = t1 - t0;

    // the first weight lines of this CTA do not depend on the previous kernel
    if (nt > 0) {
      const int g = lane >> 2, q = lane & 3;
      const int t = t0 + (warp % nt);
      if (ok_g(t, g)) prefetch_l2((const __nv_bfloat16*)a.W.data + (size_t)row_g(t, g) * a.K + 64 * q);
    }
    grid_dep_wait();
    grid_dep_launch();
    norms();

    unsigned long long mybest[2] = {0ull, 0ull};
    const int steps_total = (a.K + 31) / 32;
    for (int kc = 0; kc < p.n_kc; ++kc) {
      const int k0 = kc * p.kc;
      const int kcols = min(p.kc, a.K - k0);
      if (kc) __syncthreads();
      stage(k0, (kcols + 31) / 32 * 32);
      __syncthreads();
      const int steps = (kcols + 31) / 32;
      (void)steps_total;
      const int tasks = nt * p.s_sub;
      for (int task_i = warp; task_i < tasks; task_i += TW) {
        const int tl = task_i / p.s_sub, sub = task_i - tl * p.s_sub;
        const int s0 = (int)(((long long)sub * steps) / p.s_sub), s1 = (int)(((long long)(sub + 1) * steps) / p.s_sub);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        task(t0 + tl, k0, s0, s1, c);
        if (p.S == 1) {
          epilogue(t0 + tl, c, mybest);
        } else {
          float4* dst = reinterpret_cast<float4*>(part) + ((size_t)tl * p.S + kc * p.s_sub + sub) * 32 + lane;
          *dst = make_float4(c[0], c[1], c[2], c[3]);
        }
      }
    }
    if (p.S > 1) {
      __syncthreads();
      for (int tl = warp; tl < nt; tl += TW) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s = 0; s < p.S; ++s) {
          const float4 v = reinterpret_cast<const float4*>(part)[((size_t)tl * p.S + s) * 32 + lane];
          c[0] += v.x; c[1] += v.y; c[2] += v.z; c[3] += v.w;
        }
        epilogue(t0 + tl, c, mybest);
      }
    }
    if (a.epi == EPI_ARGMAX) argmax_tail(mybest);
  }

  SPEC_DEV void argmax_tail(unsigned long long (&mybest)[2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // lanes with the same q (= lane & 3) hold the same two rows m
#pragma unroll
    for (int o = 4; o < 32; o <<= 1)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const unsigned long long other = __shfl_xor_sync(FULL, mybest[i], o);
        mybest[i] = other > mybest[i] ? other : mybest[i];
      }
    if (lane < 4) {
      best[warp * 8 + 2 * lane] = mybest[0];
      best[warp * 8 + 2 * lane + 1] = mybest[1];
    }
    __syncthreads();
    if (threadIdx.x < a.M) {
      unsigned long long b = 0ull;
      for (int w = 0; w < TW; ++w) b = best[w * 8 + threadIdx.x] > b ? best[w * 8 + threadIdx.x] : b;
      if (b) atomicMax(&a.best[threadIdx.x], b);
    }
    if (a.tail.mode == TAIL_NONE) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned int done = atomicAdd(a.tail.counter, 1u);
      *flag = done == gridDim.x - 1;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    run_tail(a.tail);
  }
};

size_t fixed_smem() { return 8 * 4 + TW * 8 * 8 + 16; }

TcPlan plan(const GemvArgs& a, int map) {
  TcPlan p;
  p.tiles = map == MAP_PAIR ? (a.geglu_half + 7) / 8 : (a.N + 15) / 16;
  p.grid = std::min(p.tiles, num_sms());
  if (a.epi == EPI_ARGMAX) p.grid = std::min(p.tiles, num_sms());
  p.tiles_cta = (p.tiles + p.grid - 1) / p.grid;
  const int kpad = (a.K + 31) / 32 * 32;
  // largest K chunk (multiple of 256 columns, or all of K) whose staged
  // planes plus slice partials fit in shared memory
  for (int kc = kpad;; kc = (kc > 256 ? (kc - 1) / 256 * 256 : 0)) {
    if (kc <= 0) {
      p.smem = SIZE_MAX;
      return p;
    }
    p.kc = kc;
    p.n_kc = (a.K + kc - 1) / kc;
    const int steps = kc / 32;
    p.s_sub = std::max(1, std::min(TW / std::max(1, p.tiles_cta), steps / 2));
    p.S = p.n_kc * p.s_sub;
    const size_t xb = (size_t)8 * (kc + XPAD) * 2 * 2;
    const size_t pb = p.S > 1 ? (size_t)p.tiles_cta * p.S * 32 * 16 : 0;
    p.smem = fixed_smem() + xb + pb;
    if (p.smem <= (size_t)SMEM_MAX) break;
  }
  return p;
}

__global__ void __launch_bounds__(TW * 32, 1) gemv_tc_kernel(GemvArgs a, TcPlan p, int map) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int xs = p.kc + XPAD;
  Tc k{a, p, map};
  k.xhi = reinterpret_cast<uint16_t*>(smem_raw);
  k.xlo = k.xhi + 8 * xs;
  k.part = reinterpret_cast<float*>(k.xlo + 8 * xs);
  float* tail = k.part + (p.S > 1 ? (size_t)p.tiles_cta * p.S * 32 * 4 : 0);
  k.inv_rms = tail;
  k.best = reinterpret_cast<unsigned long long*>(tail + 8);
  k.flag = reinterpret_cast<int*>(k.best + TW * 8);
  k.xs = xs;
  k.run();
}

}  // namespace

void setup_gemv_tc_attributes() {
  cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
}

// bf16 weights, M <= 8. Returns 1 on launch, -2 when the plan does not fit
// (caller falls back to the CUDA-core kernel), -1 on a launch error.
int gemv_tc(const GemvArgs& a, cudaStream_t st) {
  const int map = a.epi == EPI_GEGLU ? MAP_PAIR : MAP_PLAIN;
  const TcPlan p = plan(a, map);
  if (p.smem > (size_t)SMEM_MAX || a.K % 32 || a.M > 8) return -2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(TW * 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_tc_kernel, a, p, map) == cudaSuccess ? 1 : -1;
}

}  // namespace spec
