// gemv_tc.cuh -- weight-streaming projection for bf16 weights on the tensor
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
// Work split. One CTA of 16 warps per SM; CTA c owns a balanced range of
// whole 16-row tiles (no tile is shared between CTAs), and its warps split the
// CTA's (tile, 128-column chunk) units evenly; a tile cut between warps is
// summed in shared memory in chunk order.
#pragma once
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "tail.cuh"

#define HOSTDEV_INLINE __host__ __forceinline__

namespace spec {
namespace tc {

constexpr int TW_DEFAULT = 16;          // warps per CTA of the stand-alone kernel
constexpr int XPAD = 32;                // bf16 pad per staged row (64 B): conflict-free 16-byte reads
constexpr int SMEM_MAX = 227 * 1024;

enum { MAP_PLAIN = 0, MAP_PAIR = 1, MAP_ROPE = 2 };

struct SkPlan {
  int T;         // 16-row output tiles
  int C;         // 128-column K chunks
  int U;         // units = T * C, tile-major
  int grid;
  int Ms;        // staged activation rows (= M)
  int xs;        // staged row stride (bf16 elements)
  size_t smem;
};

constexpr int KCH = 128;   // columns per unit (4 k-steps of 32)

static SPEC_DEV void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

static SPEC_DEV uint32_t bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// fp16 inputs (the Q4_0 weights, dequantized in registers, and the matching
// fp16 hi/lo activations), fp32 accumulate
static SPEC_DEV void mma16816_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                  uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A pair of activations as hi + lo halves of the MMA input type.
template <bool Q4>
static SPEC_DEV void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  if (Q4) {
    const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
    const __half2 hh = __halves2half2(h0, h1);
    const __half2 ll = __floats2half2_rn(x0 - __half2float(h0), x1 - __half2float(h1));
    hi = *reinterpret_cast<const uint32_t*>(&hh);
    lo = *reinterpret_cast<const uint32_t*>(&ll);
  } else {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
    hi = bf16x2(x0, x1);
    lo = bf16x2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
  }
}

// Eight Q4_0 codes of one row (one nibble in each byte of `raw`: the low
// nibble for elements 0..15 of the 32-value block, the high one for 16..31) as
// four fp16 pairs of code - 8, exact: 0x6400 | code is the fp16 1024 + code,
// and subtracting 1032 leaves the small integer. The block scale is applied to
// the step's partial sum in fp32 (a step never crosses a block).
static SPEC_DEV void codes8(uint2 raw, bool high, uint32_t (&v)[4]) {
  const uint32_t n0 = (high ? raw.x >> 4 : raw.x) & 0x0F0F0F0Fu, n1 = (high ? raw.y >> 4 : raw.y) & 0x0F0F0F0Fu;
  const uint32_t w[4] = {__byte_perm(n0, 0x6464u, 0x5140), __byte_perm(n0, 0x6464u, 0x5342),
                         __byte_perm(n1, 0x6464u, 0x5140), __byte_perm(n1, 0x6464u, 0x5342)};
  const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&w[i]), off);
    v[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

// first unit of CTA b
// First unit of CTA b: every CTA owns whole 16-row tiles (the tile counts of
// two CTAs differ by at most one), so no tile is split between CTAs and no
// cross-CTA partial sums are needed; the warps of a CTA split its units.
__device__ HOSTDEV_INLINE int unit_begin(int b, const SkPlan& p) {
  return (int)(((long long)b * p.T) / p.grid) * p.C;
}

// Q4: Q4_0 weights (codes and fp16 scales, K % 128 == 0): the codes enter
// fp16 MMAs exactly as code - 8 and the activations as fp16 hi + lo; each
// 32-column step is one block, whose scale multiplies the step's fp32 partial.
// Otherwise bf16 weights and bf16 MMAs.
template <int TW, bool Q4 = false>
struct Sk {
  const GemvArgs& a;
  const SkPlan& p;
  int map;
  uint16_t *xhi, *xlo;
  float* seg;               // [TW][2][32][4] flushed partial segments
  int* seg_tag;             // [TW][2]: tile, or -1
  int* seg_c0;              // [TW][2]: first chunk of the segment
  int* seg_c1;              // [TW][2]: one past the last chunk
  float* inv_rms;           // [8]
  float* red;               // [TW][8] norm partials
  unsigned long long* best; // [TW][8]
  int* flag;
  float* fix;               // global [grid][2][32][4]
  unsigned int* cnt;        // global [T]
  int bid;                  // this CTA's index in the launch (or phase)
  bool standalone;          // own launch (PDL waits) or a phase of the persistent pass kernel
  unsigned long long* trace;  // optional: [0] after staging, [1] after the main loop; stand-alone
                              // launches also [2] entry, [3] past the dependency wait, [4] done

  // MAP_ROPE: tile t covers elements 8u..8u+7 of head h (row g) and the
  // elements hd/2 further on (row g+8), the pairs RoPE rotates together
  SPEC_DEV int row_g(int t, int g) const {
    if (map == MAP_ROPE) {
      const int hpt = a.rope.hd / 16;
      return (t / hpt) * a.rope.hd + 8 * (t % hpt) + g;
    }
    return map == MAP_PAIR ? 8 * t + g : 16 * t + g;
  }
  SPEC_DEV int row_g8(int t, int g) const {
    if (map == MAP_ROPE) return row_g(t, g) + a.rope.hd / 2;
    return map == MAP_PAIR ? a.geglu_half + 8 * t + g : 16 * t + 8 + g;
  }
  SPEC_DEV bool ok_g(int t, int g) const { return map == MAP_PAIR ? 8 * t + g < a.geglu_half : 16 * t + g < a.N; }
  SPEC_DEV bool ok_g8(int t, int g) const {
    return map == MAP_PAIR ? 8 * t + g < a.geglu_half : 16 * t + 8 + g < a.N;
  }

  // Issue the 8 weight loads of unit u (rows g and g+8 of its tile, 4 k-steps).
  SPEC_DEV void load_unit(int u, uint4 (&wa)[4], uint4 (&wb)[4]) const {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int t = u / p.C, ch = u - t * p.C;
    const int k0 = ch * KCH, steps = min(4, (a.K - k0) / 32);
    const bool vg = ok_g(t, g), vg8 = ok_g8(t, g);
    if (Q4) {
      // step s is 32-value block 4*ch + s: this lane's 8 values are the
      // nibbles of bytes 8*(q&1) .. +7 (low nibbles for q < 2, high for q >= 2);
      // the unit's 4 block scales of a row are 8 contiguous bytes.
      // wa[s] = {code bytes, code bytes, scale bits, unused}
      const uint8_t* C = (const uint8_t*)a.W.data;
      const uint16_t* S = (const uint16_t*)a.W.scales;
      const size_t ra = (size_t)(vg ? row_g(t, g) : 0), rb = (size_t)(vg8 ? row_g8(t, g) : 0);
      const uint8_t* ca = C + ra * (a.K / 2) + (size_t)ch * 64 + 8 * (q & 1);
      const uint8_t* cb = C + rb * (a.K / 2) + (size_t)ch * 64 + 8 * (q & 1);
      const uint2 sa = vg ? ldg_stream8(S + ra * (a.K / 32) + 4 * ch) : make_uint2(0, 0);
      const uint2 sb = vg8 ? ldg_stream8(S + rb * (a.K / 32) + 4 * ch) : make_uint2(0, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint2 xa = vg ? ldg_stream8(ca + s * 16) : make_uint2(0, 0);
        const uint2 xb = vg8 ? ldg_stream8(cb + s * 16) : make_uint2(0, 0);
        const uint32_t sba = (s < 2 ? sa.x : sa.y) >> (16 * (s & 1)), sbb = (s < 2 ? sb.x : sb.y) >> (16 * (s & 1));
        wa[s] = make_uint4(xa.x, xa.y, sba & 0xFFFFu, 0u);
        wb[s] = make_uint4(xb.x, xb.y, sbb & 0xFFFFu, 0u);
      }
      return;
    }
    const __nv_bfloat16* W = (const __nv_bfloat16*)a.W.data;
    const __nv_bfloat16* rg = W + (size_t)(vg ? row_g(t, g) : 0) * a.K + k0 + 8 * q;
    const __nv_bfloat16* rg8 = W + (size_t)(vg8 ? row_g8(t, g) : 0) * a.K + k0 + 8 * q;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      wa[s] = (vg && s < steps) ? ldg_stream(rg + s * 32) : make_uint4(0, 0, 0, 0);
      wb[s] = (vg8 && s < steps) ? ldg_stream(rg8 + s * 32) : make_uint4(0, 0, 0, 0);
    }
  }

  // L2 prefetch of the weight rows of units [u0, u1), at most 512 KB: one
  // bulk prefetch (cp.async.bulk.prefetch.L2) per row segment, so issuing it
  // costs a few instructions per tile rather than one per 128-byte line.
  SPEC_DEV void prefetch_slice(int u0, int u1) const {
    if (u1 <= u0) return;
    const int t0 = u0 / p.C, t1 = (u1 - 1) / p.C;
    const int max_tiles = max(1, (512 << 10) / (16 * a.K * 2));
    const int nt = min(t1 - t0 + 1, max_tiles);
    const __nv_bfloat16* W = (const __nv_bfloat16*)a.W.data;
    for (int i = threadIdx.x; i < nt * 16; i += blockDim.x) {
      const int t = t0 + (i >> 4), r = i & 15, g = r & 7;
      const bool hi_row = r >= 8;
      if (!(hi_row ? ok_g8(t, g) : ok_g(t, g))) continue;
      const int row = hi_row ? row_g8(t, g) : row_g(t, g);
      const int cs = t == t0 ? u0 - t0 * p.C : 0, ce = t == t1 ? u1 - t1 * p.C : p.C;
      const int col0 = cs * KCH, col1 = min(a.K, ce * KCH);
      if (col1 > col0) prefetch_l2_bulk(W + (size_t)row * a.K + col0, (unsigned)(col1 - col0) * 2);
    }
  }

  SPEC_DEV void mma_unit(int u, const uint4 (&wa)[4], const uint4 (&wb)[4], float (&c)[4]) const {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int ch = u % p.C, k0 = ch * KCH, steps = min(4, (a.K - k0) / 32);
    const bool xrow = g < p.Ms;
    const uint16_t* bh = xhi + g * p.xs + k0 + 8 * q;
    const uint16_t* bl = xlo + g * p.xs + k0 + 8 * q;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s >= steps) break;
      uint4 xh = make_uint4(0, 0, 0, 0), xl = make_uint4(0, 0, 0, 0);
      if (xrow) {
        xh = *reinterpret_cast<const uint4*>(bh + s * 32);
        xl = *reinterpret_cast<const uint4*>(bl + s * 32);
      }
      if (Q4) {
        // exact codes through the MMAs, then each row's block scale in fp32
        const bool high = q >= 2;
        uint32_t va[4], vb[4];
        codes8(make_uint2(wa[s].x, wa[s].y), high, va);
        codes8(make_uint2(wb[s].x, wb[s].y), high, vb);
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816_f16(t, va[0], vb[0], va[1], vb[1], xh.x, xh.y);
        mma16816_f16(t, va[0], vb[0], va[1], vb[1], xl.x, xl.y);
        mma16816_f16(t, va[2], vb[2], va[3], vb[3], xh.z, xh.w);
        mma16816_f16(t, va[2], vb[2], va[3], vb[3], xl.z, xl.w);
        const float sa = __half2float(__ushort_as_half((unsigned short)wa[s].z));
        const float sb = __half2float(__ushort_as_half((unsigned short)wb[s].z));
        c[0] = fmaf(sa, t[0], c[0]);
        c[1] = fmaf(sa, t[1], c[1]);
        c[2] = fmaf(sb, t[2], c[2]);
        c[3] = fmaf(sb, t[3], c[3]);
      } else {
        mma16816(c, wa[s].x, wb[s].x, wa[s].y, wb[s].y, xh.x, xh.y);
        mma16816(c, wa[s].x, wb[s].x, wa[s].y, wb[s].y, xl.x, xl.y);
        mma16816(c, wa[s].z, wb[s].z, wa[s].w, wb[s].w, xh.z, xh.w);
        mma16816(c, wa[s].z, wb[s].z, wa[s].w, wb[s].w, xl.z, xl.w);
      }
    }
  }

  // Stage X*gain as bf16 hi/lo planes (all of K, M rows) and the row norms:
  // RMSNorm's 1/rms is a per-row factor, applied in the epilogue.
  SPEC_DEV void stage() {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_row = a.K / 8;
    const int items = p.Ms * per_row;
    constexpr int BATCH = TW >= 16 ? 4 : 8;  // items per thread whose loads are all in flight together
    float ss[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) ss[m] = 0.f;
    for (int base = 0; base < items; base += BATCH * blockDim.x) {
      float4 u0[BATCH], u1[BATCH];
#pragma unroll
      for (int j = 0; j < BATCH; ++j) {
        const int idx = base + j * blockDim.x + threadIdx.x;
        if (idx < items) {
          const int m = idx / per_row, c8 = (idx - m * per_row) * 8;
          // activations come from other CTAs of the same persistent launch: L2 only
          u0[j] = __ldcg(reinterpret_cast<const float4*>(a.X + (size_t)m * a.ldx + c8));
          u1[j] = __ldcg(reinterpret_cast<const float4*>(a.X + (size_t)m * a.ldx + c8 + 4));
        }
      }
#pragma unroll
      for (int j = 0; j < BATCH; ++j) {
        const int idx = base + j * blockDim.x + threadIdx.x;
        if (idx >= items) continue;
        const int m = idx / per_row, c8 = (idx - m * per_row) * 8;
        float v[8] = {u0[j].x, u0[j].y, u0[j].z, u0[j].w, u1[j].x, u1[j].y, u1[j].z, u1[j].w};
        if (a.gain) {
          float sq = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) sq = fmaf(v[i], v[i], sq);
#pragma unroll
          for (int mm = 0; mm < 8; ++mm)
            if (mm == m) ss[mm] += sq;
          const float4 g0 = *reinterpret_cast<const float4*>(a.gain + c8);
          const float4 g1 = *reinterpret_cast<const float4*>(a.gain + c8 + 4);
          v[0] *= g0.x; v[1] *= g0.y; v[2] *= g0.z; v[3] *= g0.w;
          v[4] *= g1.x; v[5] *= g1.y; v[6] *= g1.z; v[7] *= g1.w;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_pair<Q4>(v[2 * i], v[2 * i + 1], hi[i], lo[i]);
        *reinterpret_cast<uint4*>(xhi + m * p.xs + c8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(xlo + m * p.xs + c8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    if (a.gain) {
      // fixed-order reduction: lanes, then warps
      for (int m = 0; m < p.Ms; ++m) {
        const float v = warp_sum(ss[m]);
        if (lane == 0) red[warp * 8 + m] = v;
      }
    }
    __syncthreads();
    if (threadIdx.x < 8) {
      float inv = 1.f;
      if (a.gain && (int)threadIdx.x < p.Ms) {
        float t = 0.f;
        for (int w = 0; w < TW; ++w) t += red[w * 8 + threadIdx.x];
        inv = rsqrtf(t / (float)a.K + a.eps);
      }
      inv_rms[threadIdx.x] = inv;
    }
    __syncthreads();
  }

  SPEC_DEV void finish(int t, float (&c)[4], unsigned long long (&mybest)[2]) {
    const int q = (threadIdx.x & 31) & 3;
    const float s0 = inv_rms[2 * q], s1 = inv_rms[2 * q + 1];
    c[0] *= s0; c[1] *= s1; c[2] *= s0; c[3] *= s1;
    epilogue(t, c, mybest);
  }

  SPEC_DEV void epilogue(int t, const float (&c)[4], unsigned long long (&mybest)[2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int m0 = 2 * q, m1 = 2 * q + 1;
    if (map == MAP_ROPE) {
      const RopeEpi& e = a.rope;
      const int hpt = e.hd / 16, h = t / hpt, j = 8 * (t % hpt) + g, half = e.hd / 2;
      const bool rot = h < e.nq + e.nkv, is_q = h < e.nq;
      // every table read of both rows first (rotation, position, page), then
      // the writes: the reads do not wait behind the writes
      float co[2] = {1.f, 1.f}, si[2] = {0.f, 0.f};
      int pos[2] = {0, 0}, page[2] = {-1, -1};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = 2 * q + i, am = a.m_base + m;
        if (m >= a.M) continue;
        if (rot) {
          co[i] = __ldcg(e.rope_cs + (size_t)am * e.hd + 2 * j);
          si[i] = __ldcg(e.rope_cs + (size_t)am * e.hd + 2 * j + 1);
        }
        if (!is_q) pos[i] = __ldcg(e.pos + am);
      }
      if (!is_q) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int m = 2 * q + i, am = a.m_base + m;
          if (m >= a.M) continue;
          const int slot = e.seq_ids[am / e.R], pidx = pos[i] / 64;
          page[i] = pidx < e.max_pages ? e.block_table[(size_t)slot * e.max_pages + pidx] : -1;
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = 2 * q + i;
        if (m >= a.M) continue;
        float y0 = c[i], y1 = c[2 + i];
        if (rot) {
          const float x0 = y0, x1 = y1;
          y0 = x0 * co[i] - x1 * si[i];
          y1 = x1 * co[i] + x0 * si[i];
        }
        if (is_q) {
          a.Y[(size_t)m * a.ldy + h * e.hd + j] = y0;
          a.Y[(size_t)m * a.ldy + h * e.hd + j + half] = y1;
        } else {
          if (page[i] < 0 || page[i] >= e.n_pages) {
            set_error(e.err, SPEC_ERR_CAPACITY);
            continue;
          }
          const int plane = rot ? 0 : 1;
          const int kh = h - e.nq - plane * e.nkv;
          __nv_bfloat16* dst = (__nv_bfloat16*)e.pool + e.layer_off +
                               ((((size_t)page[i] * 2 + plane) * e.nkv + kh) * 64 + pos[i] % 64) * e.hd;
          dst[j] = __float2bfloat16_rn(y0);
          dst[j + half] = __float2bfloat16_rn(y1);
        }
      }
      return;
    }
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
    if (a.epi == EPI_ADD) {
      // residual add: all four reads in flight before any write (the writes
      // would otherwise order each read behind the previous write)
      float old[4];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int m = 2 * q + i;
          old[2 * h + i] = oks[h] && m < a.M ? __ldcg(a.Y + (size_t)m * a.ldy + rows[h]) : 0.f;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int m = 2 * q + i;
          if (oks[h] && m < a.M) a.Y[(size_t)m * a.ldy + rows[h]] = old[2 * h + i] + c[2 * h + i];
        }
      return;
    }
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
    const int b = bid;
    const int u0 = unit_begin(b, p), u1 = unit_begin(b + 1, p);
    const int nu = u1 - u0;
    const int wa_ = u0 + (int)(((long long)warp * nu) / TW), wb_ = u0 + (int)(((long long)(warp + 1) * nu) / TW);

    // weights do not depend on the previous kernel: pull this CTA's slice
    // towards L2 (capped) and put the first unit in flight before the wait
    uint4 wa[4], wb[4];
    if (standalone) {
      if (trace && threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(trace[2]));
      if (a.prefetch && !Q4) prefetch_slice(u0, u1);
      if (wa_ < wb_) load_unit(wa_, wa, wb);
      grid_dep_wait();
      grid_dep_launch();
      if (trace && threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(trace[3]));
    }
    if (threadIdx.x < TW * 2) seg_tag[threadIdx.x] = -1;
    stage();
    // in the persistent pass the slice was pulled to L2 before the barrier;
    // first weight loads only now, so they do not queue ahead of the staging
    if (!standalone && wa_ < wb_) load_unit(wa_, wa, wb);
    if (trace && threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(trace[0]));

    unsigned long long mybest[2] = {0ull, 0ull};
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    int nseg = 0;
    int seg_start = wa_;
    for (int u = wa_; u < wb_; ++u) {
      uint4 ca[4], cb[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        ca[s] = wa[s];
        cb[s] = wb[s];
      }
      if (u + 1 < wb_) load_unit(u + 1, wa, wb);  // next unit in flight
      mma_unit(u, ca, cb, c);
      const int t = u / p.C;
      const bool tile_end = u + 1 == wb_ || (u + 1) / p.C != t;
      if (tile_end) {
        const int c0 = seg_start - t * p.C, c1 = u + 1 - t * p.C;
        if (c0 == 0 && c1 == p.C) {
          finish(t, c, mybest);
        } else {
          // a warp range holds at most two partial tiles: its first and its last
          const int slot = warp * 2 + (nseg > 0 ? 1 : 0);
          reinterpret_cast<float4*>(seg)[slot * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
          if (lane == 0) {
            seg_tag[slot] = t;
            seg_c0[slot] = c0;
            seg_c1[slot] = c1;
          }
        }
        ++nseg;
        c[0] = c[1] = c[2] = c[3] = 0.f;
        seg_start = u + 1;
      }
    }
    __syncthreads();
    if (trace && threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(trace[1]));

    // partial tiles of this CTA: add segments in chunk order; a tile whole in
    // this CTA is finished here, one shared with neighbours goes to the fixup.
    // Slots are in (warp, first/last) order, i.e. in tile and chunk order, so a
    // tile's segments are consecutive valid slots; each group starts at a slot
    // whose previous valid slot holds another tile.
    const int t_first = u0 / p.C;
    if (nu > 0) {
      for (int sl0 = warp; sl0 < TW * 2; sl0 += TW) {
        const int tt = seg_tag[sl0];
        if (tt < 0) continue;
        int prev = sl0 - 1;
        while (prev >= 0 && seg_tag[prev] < 0) --prev;
        if (prev >= 0 && seg_tag[prev] == tt) continue;  // not the first segment of its tile
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sl = sl0; sl < TW * 2; ++sl) {
          const int tg = seg_tag[sl];
          if (tg < 0) continue;
          if (tg != tt) break;
          const float4 v = reinterpret_cast<const float4*>(seg)[sl * 32 + lane];
          acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
        }
        const int tb = tt * p.C, te = tb + p.C;
        if (tb >= u0 && te <= u1) {
          finish(tt, acc, mybest);
          continue;
        }
        // shared with other CTAs: publish, and the last contributor finishes
        const int slot = tt == t_first ? 0 : 1;
        reinterpret_cast<float4*>(fix)[((size_t)b * 2 + slot) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncwarp();
        unsigned int done = 0;
        const int b_first = cta_of(tb), b_lastc = cta_of(te - 1);
        if (lane == 0) done = atomic_add_acq_rel(cnt + tt, 1u);
        done = __shfl_sync(FULL, done, 0);
        if ((int)done != b_lastc - b_first) continue;
        float tot[4] = {0.f, 0.f, 0.f, 0.f};
        for (int bb = b_first; bb <= b_lastc; ++bb) {
          const int s2 = tt == unit_begin(bb, p) / p.C ? 0 : 1;
          const float4 v = __ldcg(reinterpret_cast<const float4*>(fix) + ((size_t)bb * 2 + s2) * 32 + lane);
          tot[0] += v.x; tot[1] += v.y; tot[2] += v.z; tot[3] += v.w;
        }
        if (lane == 0) cnt[tt] = 0u;
        finish(tt, tot, mybest);
      }
    }
    if (a.epi == EPI_ARGMAX) argmax_tail(mybest);
    if (standalone && trace && threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(trace[4]));
  }

  // CTA whose unit range holds unit u
  SPEC_DEV int cta_of(int u) const {
    int bb = (int)((((long long)u + 1) * p.grid - 1) / p.U);
    while (bb > 0 && unit_begin(bb, p) > u) --bb;
    while (bb + 1 < p.grid && unit_begin(bb + 1, p) <= u) ++bb;
    return bb;
  }

  SPEC_DEV void argmax_tail(unsigned long long (&mybest)[2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
      unsigned long long bst = 0ull;
      for (int w = 0; w < TW; ++w) bst = best[w * 8 + threadIdx.x] > bst ? best[w * 8 + threadIdx.x] : bst;
      if (bst) atomicMax(&a.best[threadIdx.x], bst);
    }
    if (a.tail.mode == TAIL_NONE) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned int done = atomicAdd(a.tail.counter, 1u);
      *flag = done == (unsigned int)p.grid - 1;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    run_tail(a.tail);
  }
};

__host__ __device__ inline int map_of(int epi) {
  return epi == EPI_GEGLU ? MAP_PAIR : epi == EPI_ROPE ? MAP_ROPE : MAP_PLAIN;
}

// Plan: T tiles x C chunks over min(T, nsm) CTAs of TW warps.
template <int TW = 16>
__host__ __device__ inline SkPlan plan(const GemvArgs& a, int map, int nsm) {
  SkPlan p;
  p.T = map == MAP_PAIR ? (a.geglu_half + 7) / 8 : map == MAP_ROPE ? a.N / 16 : (a.N + 15) / 16;
  p.C = (a.K + KCH - 1) / KCH;
  p.U = p.T * p.C;
  p.grid = p.T < nsm ? p.T : nsm;
  p.Ms = a.M;
  p.xs = a.K + XPAD;
  const size_t xb = (size_t)(p.Ms > 1 ? p.Ms : 1) * p.xs * 2 * 2;
  p.smem = xb + (size_t)TW * 2 * 32 * 16 + TW * 2 * 3 * 4 + 8 * 4 + TW * 8 * 4 + TW * 8 * 8 + 16;
  return p;
}

// Carve the dynamic shared memory for a projection CTA.
template <int TW, bool Q4>
__device__ inline void sk_bind(Sk<TW, Q4>& k, unsigned char* smem_raw, float* fix, unsigned int* cnt, int bid,
                               bool standalone) {
  const SkPlan& p = k.p;
  k.xhi = reinterpret_cast<uint16_t*>(smem_raw);
  k.xlo = k.xhi + (size_t)(p.Ms > 1 ? p.Ms : 1) * p.xs;
  k.seg = reinterpret_cast<float*>(k.xlo + (size_t)(p.Ms > 1 ? p.Ms : 1) * p.xs);
  k.seg_tag = reinterpret_cast<int*>(k.seg + TW * 2 * 32 * 4);
  k.seg_c0 = k.seg_tag + TW * 2;
  k.seg_c1 = k.seg_c0 + TW * 2;
  k.inv_rms = reinterpret_cast<float*>(k.seg_c1 + TW * 2);
  k.red = k.inv_rms + 8;
  k.best = reinterpret_cast<unsigned long long*>(k.red + TW * 8);
  k.flag = reinterpret_cast<int*>(k.best + TW * 8);
  k.fix = fix;
  k.cnt = cnt;
  k.bid = bid;
  k.standalone = standalone;
  k.trace = nullptr;
}

}  // namespace tc
}  // namespace spec
