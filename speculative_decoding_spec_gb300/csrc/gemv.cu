// gemv.cu -- multi-row weight-streaming projection for small M (CUDA cores).
//
// Y[M][N] = X[M][K] . W[N][K]^T with W streamed from HBM exactly once per
// launch. Verification runs k+1 positions per sequence in ONE pass so the
// weights are read once for all of them ("Gemma 4's MTP drafter explained"
// (molayo1419.me), section "Why is generating one token at a time slow?":
// checking several tokens reads the same weights once with a little more
// arithmetic).
//
// Work split: a CTA of 8 warps = (8/KW) row groups x KW K-slices. A row group
// holds RPW = 4 weight rows; lane l of K-slice s reads weight unit
// u = (i*KW + s)*32 + l (16 B of bf16, 32 B of fp32, or half a Q4_0 block) so a
// warp reads contiguous 512 B runs. Activations are staged once in shared
// memory in a plane layout that makes every 16-byte read conflict-free. Each
// lane keeps RPW x M partial sums; a transposing butterfly leaves one finished
// (row, m) value per lane, then the K-slices are added in a fixed order. The
// reduction order of a row does not depend on M, so a row's result is the same
// in a one-row decode and a k+1-row verify.
//
// Prologue: optional RMSNorm of X (gain g, eps). Epilogues: store, residual
// add, GELU-gated pair (rows j and j+half), or argmax over rows with the
// lowest row index on ties, followed by a last-CTA tail (greedy accept, prefill
// commit, or draft write) -- no CTA ever waits for another.
#include <algorithm>

#include "common.cuh"
#include "tail.cuh"

namespace spec {


namespace {

constexpr int NWARP = 8;
constexpr int RPW = 4;
constexpr int XS_WHOLE = 96 * 1024;   // stage all of K when X fits in this
constexpr int XS_CHUNK = 48 * 1024;   // otherwise stage K in chunks of this

template <int WT> struct UnitT;
template <> struct UnitT<DT_F32> { static constexpr int E = 8; };
template <> struct UnitT<DT_BF16> { static constexpr int E = 8; };
template <> struct UnitT<DT_Q4_0> { static constexpr int E = 16; };

constexpr int pow2_at_least(int x) { return x <= 1 ? 1 : x <= 2 ? 2 : x <= 4 ? 4 : x <= 8 ? 8 : 16; }

// Column of unit element e (0..E-1) of unit u, for the weight format.
template <int WT>
SPEC_DEV int unit_col(int u, int e) {
  if (WT == DT_Q4_0) {
    // unit = half a block: bytes [8h, 8h+8) of block b hold elements 8h+i (low
    // nibbles) and 16+8h+i (high nibbles)
    const int b = u >> 1, h = u & 1;
    return b * 32 + (e < 8 ? 8 * h + e : 16 + 8 * h + (e - 8));
  }
  return u * 8 + e;
}

// Load unit u of row n (raw bits) and, for Q4_0, its block scale.
template <int WT>
SPEC_DEV void load_unit(const Mat& W, int K, int n, int u, uint4& a, uint4& b, float& s) {
  if (WT == DT_BF16) {
    a = ldg_stream((const char*)W.data + ((size_t)n * K + (size_t)u * 8) * 2);
  } else if (WT == DT_F32) {
    const char* p = (const char*)W.data + ((size_t)n * K + (size_t)u * 8) * 4;
    a = ldg_stream(p);
    b = ldg_stream(p + 16);
  } else {
    const uint2 c = ldg_stream8((const char*)W.data + (size_t)n * (K / 2) + (size_t)u * 8);
    a.x = c.x;
    a.y = c.y;
    s = __half2float(((const __half*)W.scales)[(size_t)n * (K / 32) + (u >> 1)]);
  }
}

// Unpack a unit to E floats (Q4_0: code - 8, scale applied later).
template <int WT>
SPEC_DEV void unpack_unit(const uint4& a, const uint4& b, float* w) {
  if (WT == DT_BF16) {
    w[0] = bf16lo(a.x); w[1] = bf16hi(a.x); w[2] = bf16lo(a.y); w[3] = bf16hi(a.y);
    w[4] = bf16lo(a.z); w[5] = bf16hi(a.z); w[6] = bf16lo(a.w); w[7] = bf16hi(a.w);
  } else if (WT == DT_F32) {
    w[0] = __uint_as_float(a.x); w[1] = __uint_as_float(a.y);
    w[2] = __uint_as_float(a.z); w[3] = __uint_as_float(a.w);
    w[4] = __uint_as_float(b.x); w[5] = __uint_as_float(b.y);
    w[6] = __uint_as_float(b.z); w[7] = __uint_as_float(b.w);
  } else {
    // byte j of a word -> 0x4B0000jj = 2^23 + code; subtracting 2^23 + 8 gives code - 8 exactly
    const uint32_t lo0 = a.x & 0x0f0f0f0fu, lo1 = a.y & 0x0f0f0f0fu;
    const uint32_t hi0 = (a.x >> 4) & 0x0f0f0f0fu, hi1 = (a.y >> 4) & 0x0f0f0f0fu;
    const uint32_t words[4] = {lo0, lo1, hi0, hi1};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[q * 4 + j] = __uint_as_float(__byte_perm(words[q], 0x4bu, j | (5 << 4) | (5 << 8) | (4 << 12))) -
                       8388616.f;
  }
}

struct Smem {
  float* xs;        // staged X planes
  float* red;       // K-slice partials [NWARP][32]
  float* inv_rms;   // [16]
  unsigned long long* best;  // [NWARP][8]
  int* flag;
};

template <int WT, int MT>
struct Gemv {
  static constexpr int E = UnitT<WT>::E;
  static constexpr int NP = E / 4;          // float4 planes per unit
  static constexpr int MTP = pow2_at_least(MT);
  static constexpr int NV = RPW * MTP;      // values per lane before the butterfly
  static constexpr int SHIFT = 5 - (NV == 32 ? 5 : NV == 16 ? 4 : NV == 8 ? 3 : NV == 4 ? 2 : 1);

  // Stage X[:, unit u0 .. u0+units) (normalised when a gain is given) as
  // planes: plane p of unit u for row m at xs[((m*NP + p)*units + u)*4 .. +3].
  // A plane is 4 consecutive columns, so it is read with one 16-byte load.
  static SPEC_DEV void stage(const GemvArgs& a, const Smem& sm, int u0, int units) {
    float4* xs4 = reinterpret_cast<float4*>(sm.xs);
    for (int idx = threadIdx.x; idx < MT * units; idx += blockDim.x) {
      const int m = idx / units, u = idx - m * units;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const int col = unit_col<WT>(u0 + u, p * 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < a.M && col < a.K) {
          v = *reinterpret_cast<const float4*>(a.X + (size_t)m * a.ldx + col);
          if (a.gain) {
            const float4 g = *reinterpret_cast<const float4*>(a.gain + col);
            const float s = sm.inv_rms[m];
            v = make_float4(v.x * s * g.x, v.y * s * g.y, v.z * s * g.z, v.w * s * g.w);
          }
        }
        xs4[(m * NP + p) * units + u] = v;
      }
    }
  }

  static SPEC_DEV void row_norms(const GemvArgs& a, const Smem& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int m = w; m < MT; m += NWARP) {
      float ss = 0.f;
      if (m < a.M)
        for (int c = lane; c < a.K; c += 32) {
          const float v = a.X[(size_t)m * a.ldx + c];
          ss = fmaf(v, v, ss);
        }
      ss = warp_sum(ss);
      if (lane == 0) sm.inv_rms[m] = rsqrtf(ss / (float)a.K + a.eps);
    }
    __syncthreads();
  }

  // Physical weight row of value slot r in row group starting at logical row j0.
  static SPEC_DEV int phys_row(const GemvArgs& a, int j0, int r) {
    if (a.epi == EPI_GEGLU) return r < RPW / 2 ? j0 + r : a.geglu_half + j0 + (r - RPW / 2);
    return j0 + r;
  }
  static SPEC_DEV bool row_ok(const GemvArgs& a, int j0, int r) {
    if (a.epi == EPI_GEGLU) return j0 + (r % (RPW / 2)) < a.geglu_half;
    return j0 + r < a.N;
  }

  static SPEC_DEV void run(const GemvArgs& a, const Smem& sm, int KW) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int groups = NWARP / KW, grp = warp / KW, ks = warp % KW;
    const int lrows = a.epi == EPI_GEGLU ? RPW / 2 : RPW;     // logical outputs per group
    const int n_logical = a.epi == EPI_GEGLU ? a.geglu_half : a.N;
    const int rows_per_cta = groups * lrows;
    const int n_blocks = (n_logical + rows_per_cta - 1) / rows_per_cta;
    const int units_total = (a.K + E - 1) / E;
    const bool whole = MT * units_total * E * 4 <= XS_WHOLE;
    const int chunk_units = whole ? units_total : (XS_CHUNK / (MT * E * 4)) / (32 * KW) * (32 * KW);

    // weights of this CTA's first block do not depend on the previous kernel
    if ((int)blockIdx.x < n_blocks) {
      const int j0 = blockIdx.x * rows_per_cta;
      const size_t row_bytes = WT == DT_Q4_0 ? (size_t)a.K / 2 : (size_t)a.K * (WT == DT_F32 ? 4 : 2);
      for (int r = 0; r < rows_per_cta * (a.epi == EPI_GEGLU ? 2 : 1); ++r) {
        const int n = a.epi == EPI_GEGLU ? (r < rows_per_cta ? j0 + r : a.geglu_half + j0 + r - rows_per_cta)
                                         : j0 + r;
        if (n >= a.N) continue;
        for (size_t off = (size_t)threadIdx.x * 128; off < row_bytes; off += (size_t)blockDim.x * 128)
          prefetch_l2((const char*)a.W.data + n * row_bytes + off);
      }
    }
    grid_dep_wait();
    grid_dep_launch();

    if (a.gain) row_norms(a, sm);
    if (whole) {
      stage(a, sm, 0, units_total);
      __syncthreads();
    }

    unsigned long long mybest = 0ull;
    for (int blk = blockIdx.x; blk < n_blocks; blk += gridDim.x) {
      const int j0 = blk * rows_per_cta + grp * lrows;
      float acc[RPW][MTP];
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int m = 0; m < MTP; ++m) acc[r][m] = 0.f;
      int rown[RPW];
      bool rvalid[RPW];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        rvalid[r] = row_ok(a, j0, r);
        rown[r] = phys_row(a, j0, r);
      }

      for (int cu0 = 0; cu0 < units_total; cu0 += chunk_units) {
        const int cunits = min(chunk_units, units_total - cu0);
        if (!whole) {
          __syncthreads();
          stage(a, sm, cu0, cunits);
          __syncthreads();
        }
        const int ustride = 32 * KW;
        // two units per lane per trip: all 2*RPW weight loads are in flight
        // before the first one is used
        for (int uu0 = ks * 32 + lane; uu0 < cunits; uu0 += 2 * ustride) {
          uint4 wa[2][RPW], wb[2][RPW];
          float ws[2][RPW];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int uu = uu0 + q * ustride;
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
              wa[q][r] = make_uint4(0, 0, 0, 0);
              wb[q][r] = make_uint4(0, 0, 0, 0);
              ws[q][r] = 0.f;
              if (uu < cunits && rvalid[r]) load_unit<WT>(a.W, a.K, rown[r], cu0 + uu, wa[q][r], wb[q][r], ws[q][r]);
            }
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int uu = uu0 + q * ustride;
            if (uu >= cunits) break;
            if (WT == DT_Q4_0) {
#pragma unroll
              for (int r = 0; r < RPW; ++r) {
                float w[E];
                unpack_unit<WT>(wa[q][r], wb[q][r], w);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                  float t = 0.f;
#pragma unroll
                  for (int p = 0; p < NP; ++p) {
                    const float4 xv = reinterpret_cast<const float4*>(sm.xs)[(m * NP + p) * cunits + uu];
                    t = fmaf(w[p * 4 + 0], xv.x, t);
                    t = fmaf(w[p * 4 + 1], xv.y, t);
                    t = fmaf(w[p * 4 + 2], xv.z, t);
                    t = fmaf(w[p * 4 + 3], xv.w, t);
                  }
                  acc[r][m] = fmaf(ws[q][r], t, acc[r][m]);
                }
              }
            } else {
              float w[RPW][E];
#pragma unroll
              for (int r = 0; r < RPW; ++r) unpack_unit<WT>(wa[q][r], wb[q][r], w[r]);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                  const float4 xv = reinterpret_cast<const float4*>(sm.xs)[(m * NP + p) * cunits + uu];
#pragma unroll
                  for (int r = 0; r < RPW; ++r) {
                    float t = acc[r][m];
                    t = fmaf(w[r][p * 4 + 0], xv.x, t);
                    t = fmaf(w[r][p * 4 + 1], xv.y, t);
                    t = fmaf(w[r][p * 4 + 2], xv.z, t);
                    t = fmaf(w[r][p * 4 + 3], xv.w, t);
                    acc[r][m] = t;
                  }
                }
              }
            }
          }
        }
      }

      // transposing butterfly: afterwards lane holds value index (lane >> SHIFT)
      float v[NV];
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int m = 0; m < MTP; ++m) v[r * MTP + m] = acc[r][m];
#pragma unroll
      for (int o = 16, n = NV; n > 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float send = up ? v[i] : v[i + n / 2];
          const float keep = up ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(FULL, send, o);
        }
      }
#pragma unroll
      for (int o = (1 << SHIFT) >> 1; o > 0; o >>= 1) v[0] += __shfl_xor_sync(FULL, v[0], o);
      const int vid = lane >> SHIFT;
      const int vr = vid / MTP, vm = vid % MTP;
      const bool owner = (lane & ((1 << SHIFT) - 1)) == 0;

      // add the K-slices in a fixed order
      float val = v[0];
      if (KW > 1) {
        __syncthreads();
        sm.red[warp * 32 + lane] = val;
        __syncthreads();
        val = 0.f;
        for (int s = 0; s < KW; ++s) val += sm.red[(grp * KW + s) * 32 + lane];
      }
      const bool lead = ks == 0;

      if (a.epi == EPI_GEGLU) {
        // gate slots r < RPW/2 pair with up slots r + RPW/2
        const int src = ((vid + (RPW / 2) * MTP) << SHIFT) & 31;
        const float up = __shfl_sync(FULL, val, src);
        if (lead && owner && vr < RPW / 2 && vm < MT && rvalid[vr]) {
          const float g = val;
          const float gl = 0.5f * g * (1.f + erff(g * 0.70710678118654752f));
          a.Y[(size_t)vm * a.ldy + j0 + vr] = gl * up;
        }
      } else if (lead && owner && vm < MT && vr < RPW && rvalid[vr]) {
        const int n = j0 + vr;
        float* y = a.Y ? a.Y + (size_t)vm * a.ldy + n : nullptr;
        if (a.epi == EPI_STORE) *y = val;
        else if (a.epi == EPI_ADD) *y += val;
        else {
          if (y) *y = val;
          const unsigned long long key = pack_best(val, (uint32_t)n);
          mybest = key > mybest ? key : mybest;
        }
      }
    }

    if (a.epi == EPI_ARGMAX) argmax_tail(a, sm, mybest);
  }

  // Combine per-lane bests per m, one atomicMax per CTA and m, then the last CTA
  // to arrive runs the tail.
  static SPEC_DEV void argmax_tail(const GemvArgs& a, const Smem& sm, unsigned long long mybest) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int vid = lane >> SHIFT, vm = vid % MTP;
    // lanes sharing vm differ in the row bits of vid
#pragma unroll
    for (int o = 16; o >= (MTP << SHIFT); o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(FULL, mybest, o);
      mybest = other > mybest ? other : mybest;
    }
    if (lane < (MTP << SHIFT) && (lane & ((1 << SHIFT) - 1)) == 0 && vm < MT) sm.best[warp * 8 + vm] = mybest;
    __syncthreads();
    if (threadIdx.x < MT) {
      unsigned long long b = 0ull;
      for (int w = 0; w < NWARP; ++w) b = sm.best[w * 8 + threadIdx.x] > b ? sm.best[w * 8 + threadIdx.x] : b;
      if (b) atomicMax(&a.best[threadIdx.x], b);
    }
    if (a.tail.mode == TAIL_NONE) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned int done = atomicAdd(a.tail.counter, 1u);
      *sm.flag = done == gridDim.x - 1;
    }
    __syncthreads();
    if (!*sm.flag) return;
    __threadfence();
    run_tail(a.tail);
  }
};

}  // namespace

template <int WT, int MT>
__global__ void __launch_bounds__(NWARP * 32) gemv_kernel(GemvArgs a, int KW) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem sm;
  sm.red = reinterpret_cast<float*>(smem_raw);                             // 256 floats
  sm.inv_rms = sm.red + NWARP * 32;                                        // 16 floats
  sm.best = reinterpret_cast<unsigned long long*>(sm.inv_rms + 16);        // 64 u64
  sm.flag = reinterpret_cast<int*>(sm.best + NWARP * 8);                   // 4 ints
  sm.xs = reinterpret_cast<float*>(sm.flag + 4);
  Gemv<WT, MT>::run(a, sm, KW);
}

namespace {

constexpr size_t SMEM_FIXED = (NWARP * 32 + 16) * 4 + NWARP * 8 * 8 + 16;

template <int WT>
constexpr int unit_elems() { return UnitT<WT>::E; }

int pick_kw(int n_logical_rows, int K, int unit_cols) {
  // enough warps in flight to cover HBM latency, but at least one unit per lane per slice
  const int warp_rows = (n_logical_rows + RPW - 1) / RPW;
  const int target = num_sms() * 16;
  int kw = 1;
  while (kw < NWARP && warp_rows * kw < target && (K / unit_cols) >= 32 * kw * 2) kw *= 2;
  return kw;
}

template <int WT, int MT>
int launch_mt(const GemvArgs& a, cudaStream_t st) {
  constexpr int E = UnitT<WT>::E;
  const int units_total = (a.K + E - 1) / E;
  const bool whole = MT * units_total * E * 4 <= XS_WHOLE;
  const int lrows = a.epi == EPI_GEGLU ? RPW / 2 : RPW;
  const int n_logical = a.epi == EPI_GEGLU ? a.geglu_half : a.N;
  int KW = pick_kw(n_logical * (a.epi == EPI_GEGLU ? 2 : 1), a.K, E);
  if (!whole) {
    // chunks hold a whole number of 32*KW-unit sweeps
    while (KW > 1 && (XS_CHUNK / (MT * E * 4)) / (32 * KW) == 0) KW /= 2;
  }
  const size_t xs = whole ? (size_t)MT * units_total * E * 4 : (size_t)XS_CHUNK;
  const size_t smem = SMEM_FIXED + xs;
  const int rows_per_cta = (NWARP / KW) * lrows;
  const int n_blocks = (n_logical + rows_per_cta - 1) / rows_per_cta;
  int grid = n_blocks;
  if (a.epi == EPI_ARGMAX) grid = std::min(n_blocks, 2 * num_sms());
  if (grid <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NWARP * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, gemv_kernel<WT, MT>, a, KW) != cudaSuccess) return -1;
  return 1;
}

template <int WT>
int launch_wt(const GemvArgs& a, cudaStream_t st) {
  switch (a.M) {
    case 1: return launch_mt<WT, 1>(a, st);
    case 2: return launch_mt<WT, 2>(a, st);
    case 3: return launch_mt<WT, 3>(a, st);
    case 4: return launch_mt<WT, 4>(a, st);
    case 5: return launch_mt<WT, 5>(a, st);
    case 6: return launch_mt<WT, 6>(a, st);
    case 7: return launch_mt<WT, 7>(a, st);
    case 8: return launch_mt<WT, 8>(a, st);
  }
  return -1;
}

template <int WT>
void set_attrs_wt() {
  const int s = (int)(SMEM_FIXED + XS_WHOLE);
  cudaFuncSetAttribute(gemv_kernel<WT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 5>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 7>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
  cudaFuncSetAttribute(gemv_kernel<WT, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
}

}  // namespace

void setup_gemv_attributes() {
  setup_gemv_tc_attributes();
  setup_gemv_wide_attributes();
  set_attrs_wt<DT_F32>();
  set_attrs_wt<DT_BF16>();
  set_attrs_wt<DT_Q4_0>();
}

// More than 8 rows of bf16 / Q4_0 weights, or a bf16 matrix of at least
// WIDE_MIN_ELEMS elements, with the tcgen05 scratch present: passes of up to
// 64 rows through the tcgen05 kernel (gemm_wide.cu), each streaming the
// weights once. Otherwise passes of at most 8 rows on the register-fragment
// kernel (each streams W again). The choice for a matrix does not depend on
// the row count when the matrix is large, so a one-row decode and a k+1-row
// verify of it run the same kernel.
bool gemv_goes_wide(const GemvArgs& a0) {
  GemvArgs first = a0;
  first.M = std::min(64, a0.M);
  const bool large = a0.W.dtype == DT_BF16 && (long long)a0.N * a0.K >= WIDE_MIN_ELEMS && a0.K >= WIDE_MIN_K;
  return (a0.M > 8 || large) && gemv_wide_ok(first);
}

int gemv(const GemvArgs& a0, cudaStream_t st) {
  int launched = 0;
  const bool wide = gemv_goes_wide(a0);
  const int step = wide ? 64 : 8;
  for (int m0 = 0; m0 < a0.M; m0 += step) {
    GemvArgs a = a0;
    a.M = std::min(step, a0.M - m0);
    a.X = a0.X + (size_t)m0 * a0.ldx;
    a.m_base = a0.m_base + m0;
    if (a.Y) a.Y = a0.Y + (size_t)m0 * a0.ldy;
    if (a0.epi == EPI_ARGMAX) {
      a.best = a0.best + m0;
      // only the last pass runs the tail, over every row
      if (m0 + step < a0.M) a.tail.mode = TAIL_NONE;
    }
    if (wide) {
      const int r = gemv_wide(a, st);
      if (r < 0) return -1;
      launched += r;
      continue;
    }
    int r = -2;
    if (a.W.dtype == DT_BF16 || a.W.dtype == DT_Q4_0) r = gemv_tc(a, a.tc_fix, a.tc_cnt, st);
    if (r == -1 || (r == -2 && a.epi == EPI_ROPE)) return -1;
    if (r >= 0) {
      launched += r;
      continue;
    }
    if (a.W.dtype == DT_BF16) r = launch_wt<DT_BF16>(a, st);
    else if (a.W.dtype == DT_F32) r = launch_wt<DT_F32>(a, st);
    else r = launch_wt<DT_Q4_0>(a, st);
    if (r < 0) return r;
    launched += r;
  }
  return launched;
}

}  // namespace spec
