// attn_tc.cu -- causal attention of the verified rows over a bf16 paged KV
// cache on the tensor cores (mma.sync m16n8k16, fp32 accumulate).
//
// Row i of sequence b sits at position seq_len + i and attends keys
// 0 .. seq_len + i (its own key and those of earlier rows of the same pass
// included): the target checks every drafted position in one pass ("Gemma 4's
// MTP drafter explained" (molayo1419.me), section "How does speculative
// decoding work?"). The drafter's cross-attention reuses this kernel on the
// target's last-layer pages with keys 0 .. seq_len - 1 ("Accelerating Gemini
// Nano on Pixel with frozen multi-token prediction" (ai-news-spoon), section
// "Zero-copy architecture").
//
// CTA (sequence b, KV head, split s) walks pages [s*pps, (s+1)*pps) with a
// two-stage cp.async pipeline. All rows x GQA-group queries of the sequence
// form 16-query tiles, one warp per tile: S = Q K^T (scores), online softmax,
// O += P V with V fragments from ldmatrix.trans. Q and P enter the MMAs as
// bf16 hi + lo pairs (two MMAs each), so scores and outputs carry fp32-level
// accuracy against the exact bf16 keys and values. Each split writes an
// unnormalised partial (max, sum, O); the last CTA of (b, KV head) to finish
// merges the splits with log-sum-exp weights -- no CTA waits for another.
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"

namespace spec {

namespace {

constexpr int PAGE = 64;

SPEC_DEV void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

SPEC_DEV uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// hi = bf16(x), lo = bf16(x - hi), for a pair
SPEC_DEV void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = pack2(x0, x1);
  lo = pack2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

SPEC_DEV void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
SPEC_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SPEC_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

SPEC_DEV void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, const void* smem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(s));
}

template <int HD>
struct AttnTc {
  static constexpr int ST = HD + 8;  // padded smem row (elements): 16-byte aligned, conflict-free
  static constexpr int NDT = HD / 8; // output d-tiles
  static constexpr int NKS = HD / 16;

  static SPEC_DEV void load_page(const AttnArgs& a, const __nv_bfloat16* base, int page, int kvh, int nk,
                                 __nv_bfloat16* Ks, __nv_bfloat16* Vs) {
    const __nv_bfloat16* kp = base + (((size_t)page * 2 + 0) * a.nkv + kvh) * PAGE * HD;
    const __nv_bfloat16* vp = base + (((size_t)page * 2 + 1) * a.nkv + kvh) * PAGE * HD;
    constexpr int CPR = HD / 8;  // 16-byte chunks per row
    for (int t = threadIdx.x; t < PAGE * CPR; t += blockDim.x) {
      const int r = t / CPR, ch = t % CPR;
      if (r < nk) {
        cp_async16(Ks + r * ST + ch * 8, kp + r * HD + ch * 8);
        cp_async16(Vs + r * ST + ch * 8, vp + r * HD + ch * 8);
      } else {
        *reinterpret_cast<uint4*>(Ks + r * ST + ch * 8) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(Vs + r * ST + ch * 8) = make_uint4(0, 0, 0, 0);
      }
    }
  }

  static SPEC_DEV void run(const AttnArgs& a, int pps, unsigned int* counters, unsigned char* smem) {
    const int b = blockIdx.x / a.nkv, kvh = blockIdx.x % a.nkv, split = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
    const int G = a.nq / a.nkv, QN = a.R * G, QT = (QN + 15) / 16;
    __nv_bfloat16* Qh = reinterpret_cast<__nv_bfloat16*>(smem);
    __nv_bfloat16* Ql = Qh + QT * 16 * ST;
    __nv_bfloat16* Kb = Ql + QT * 16 * ST;      // [2][64][ST]
    __nv_bfloat16* Vb = Kb + 2 * PAGE * ST;     // [2][64][ST]
    __shared__ int s_last;

    // sequence lengths and page tables are only written by the previous pass,
    // so the pages can be pulled towards L2 before waiting for the kernel that
    // appends this pass's keys
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int lmax = L0 + a.R - 1 + a.key_extra;  // keys of the last row
    const int npages = min((lmax + PAGE - 1) / PAGE, a.max_pages);
    const int p0 = split * pps, p1 = min(p0 + pps, npages);
    const __nv_bfloat16* base = (const __nv_bfloat16*)a.pool + (size_t)a.layer * a.layer_elems;
    {
      constexpr int LINES = PAGE * HD * 2 / 128;  // 128-byte lines per K (or V) plane
      for (int i = threadIdx.x; i < (p1 - p0) * 2 * LINES; i += blockDim.x) {
        const int p = p0 + i / (2 * LINES), r = i % (2 * LINES), plane = r / LINES, ln = r % LINES;
        const int pg = a.block_table[(size_t)slot * a.max_pages + p];
        if (pg >= 0 && pg < a.n_pages)
          prefetch_l2(base + (((size_t)pg * 2 + plane) * a.nkv + kvh) * PAGE * HD + ln * 64);
      }
    }
    grid_dep_wait();
    grid_dep_launch();

    // page ids (validated before any load)
    bool pages_ok = true;
    for (int p = p0; p < p1; ++p) {
      const int pg = a.block_table[(size_t)slot * a.max_pages + p];
      if (pg < 0 || pg >= a.n_pages) pages_ok = false;
    }
    if (!pages_ok && threadIdx.x == 0) set_error(a.err, SPEC_ERR_CAPACITY);
    const int pend = pages_ok ? p1 : p0;

    if (p0 < pend) {
      const int pg = a.block_table[(size_t)slot * a.max_pages + p0];
      load_page(a, base, pg, kvh, min(PAGE, lmax - p0 * PAGE), Kb, Vb);
    }
    cp_async_commit();

    // queries: q = i*G + gg is head kvh*G + gg of row b*R + i (RoPE applied on load if asked)
    for (int t = threadIdx.x; t < QT * 16 * (HD / 2); t += blockDim.x) {
      const int q = t / (HD / 2), d2 = (t % (HD / 2)) * 2;
      float x0 = 0.f, x1 = 0.f;
      if (q < QN) {
        const int i = q / G, gg = q % G;
        const int m = b * a.R + i, h = kvh * G + gg;
        const float* qr = a.q + (size_t)m * a.ldq + h * HD;
        if (a.rope_cs) {
          const float* cs = a.rope_cs + (size_t)m * HD;
          float v[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d = d2 + e, half = HD / 2, j = d % half;
            const float co = cs[2 * j], si = cs[2 * j + 1];
            v[e] = d < half ? qr[d] * co - qr[d + half] * si : qr[d] * co + qr[d - half] * si;
          }
          x0 = v[0];
          x1 = v[1];
        } else {
          x0 = qr[d2];
          x1 = qr[d2 + 1];
        }
      }
      uint32_t hi, lo;
      split2(x0, x1, hi, lo);
      *reinterpret_cast<uint32_t*>(Qh + q * ST + d2) = hi;
      *reinterpret_cast<uint32_t*>(Ql + q * ST + d2) = lo;
    }

    // per-warp online-softmax state for query rows r0 = 16*warp + g and r1 = r0 + 8
    const int r0 = 16 * warp + g, r1 = r0 + 8;
    const int nk0 = r0 < QN ? L0 + r0 / G + a.key_extra : 0;
    const int nk1 = r1 < QN ? L0 + r1 / G + a.key_extra : 0;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[NDT][4];
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    const float scale = rsqrtf((float)HD);

    for (int p = p0; p < pend; ++p) {
      const int st = (p - p0) & 1;
      if (p + 1 < pend) {
        const int pg = a.block_table[(size_t)slot * a.max_pages + p + 1];
        load_page(a, base, pg, kvh, min(PAGE, lmax - (p + 1) * PAGE), Kb + (st ^ 1) * PAGE * ST,
                  Vb + (st ^ 1) * PAGE * ST);
      }
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      const __nv_bfloat16* Ks = Kb + st * PAGE * ST;
      const __nv_bfloat16* Vs = Vb + st * PAGE * ST;
      if (warp < QT) {
        // S = Q K^T for the 64 keys of this page (8 n-tiles of 8 keys)
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          const __nv_bfloat16* qa = Qh + r0 * ST + 16 * ks + 2 * c;
          const __nv_bfloat16* qb = Ql + r0 * ST + 16 * ks + 2 * c;
          const uint32_t ah0 = *reinterpret_cast<const uint32_t*>(qa);
          const uint32_t ah1 = *reinterpret_cast<const uint32_t*>(qa + 8 * ST);
          const uint32_t ah2 = *reinterpret_cast<const uint32_t*>(qa + 8);
          const uint32_t ah3 = *reinterpret_cast<const uint32_t*>(qa + 8 * ST + 8);
          const uint32_t al0 = *reinterpret_cast<const uint32_t*>(qb);
          const uint32_t al1 = *reinterpret_cast<const uint32_t*>(qb + 8 * ST);
          const uint32_t al2 = *reinterpret_cast<const uint32_t*>(qb + 8);
          const uint32_t al3 = *reinterpret_cast<const uint32_t*>(qb + 8 * ST + 8);
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            const __nv_bfloat16* kr = Ks + (8 * nt + g) * ST + 16 * ks + 2 * c;
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 8);
            mma_bf16(s[nt], ah0, ah1, ah2, ah3, b0, b1);
            mma_bf16(s[nt], al0, al1, al2, al3, b0, b1);
          }
        }
        // mask, scale, online softmax (rows r0: elements 0,1; r1: elements 2,3)
        const int key0 = p * PAGE;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = key0 + 8 * nt + 2 * c + e;
            s[nt][e] = key < nk0 ? s[nt][e] * scale : -INFINITY;
            s[nt][2 + e] = key < nk1 ? s[nt][2 + e] * scale : -INFINITY;
            mx0 = fmaxf(mx0, s[nt][e]);
            mx1 = fmaxf(mx1, s[nt][2 + e]);
          }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al_0 = mn0 == -INFINITY ? 1.f : __expf(m0 - mn0);
        const float al_1 = mn1 == -INFINITY ? 1.f : __expf(m1 - mn1);
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            s[nt][e] = s[nt][e] == -INFINITY ? 0.f : __expf(s[nt][e] - mn0);
            s[nt][2 + e] = s[nt][2 + e] == -INFINITY ? 0.f : __expf(s[nt][2 + e] - mn1);
            ps0 += s[nt][e];
            ps1 += s[nt][2 + e];
          }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
          ps0 += __shfl_xor_sync(FULL, ps0, off);
          ps1 += __shfl_xor_sync(FULL, ps1, off);
        }
        l0 = l0 * al_0 + ps0;
        l1 = l1 * al_1 + ps1;
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          o[dt][0] *= al_0;
          o[dt][1] *= al_0;
          o[dt][2] *= al_1;
          o[dt][3] *= al_1;
        }
        // O += P V: P fragments come straight from the score fragments
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t ph0, pl0, ph1, pl1, ph2, pl2, ph3, pl3;
          split2(s[2 * kk][0], s[2 * kk][1], ph0, pl0);
          split2(s[2 * kk][2], s[2 * kk][3], ph1, pl1);
          split2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph2, pl2);
          split2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph3, pl3);
#pragma unroll
          for (int dt = 0; dt < NDT; ++dt) {
            uint32_t b0, b1;
            ldmatrix_x2_trans(b0, b1, Vs + (16 * kk + (lane & 15)) * ST + 8 * dt);
            mma_bf16(o[dt], ph0, ph1, ph2, ph3, b0, b1);
            mma_bf16(o[dt], pl0, pl1, pl2, pl3, b0, b1);
          }
        }
      }
      __syncthreads();
    }
    cp_async_wait<0>();

    // write this split's partial (or the final output when there is one split)
    if (warp < QT) {
      const int rows[2] = {r0, r1};
      const float mm[2] = {m0, m1}, ll[2] = {l0, l1};
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int q = rows[h2];
        if (q >= QN) continue;
        const int i = q / G, gg = q % G;
        const int m = b * a.R + i, h = kvh * G + gg;
        if (a.n_split == 1) {
          const float inv = ll[h2] > 0.f ? 1.f / ll[h2] : 0.f;
          float* out = a.out + (size_t)m * a.nq * HD + h * HD;
#pragma unroll
          for (int dt = 0; dt < NDT; ++dt) {
            out[8 * dt + 2 * c] = o[dt][2 * h2] * inv;
            out[8 * dt + 2 * c + 1] = o[dt][2 * h2 + 1] * inv;
          }
        } else {
          const size_t pidx = ((size_t)m * a.nq + h) * a.n_split + split;
          float* po = a.part_o + pidx * HD;
#pragma unroll
          for (int dt = 0; dt < NDT; ++dt) {
            po[8 * dt + 2 * c] = o[dt][2 * h2];
            po[8 * dt + 2 * c + 1] = o[dt][2 * h2 + 1];
          }
          if (c == 0) {
            a.part_ml[pidx * 2] = mm[h2];
            a.part_ml[pidx * 2 + 1] = ll[h2];
          }
        }
      }
    }
    if (a.n_split == 1) return;

    // the last split CTA of (b, KV head) merges
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned int done = atomicAdd(counters + blockIdx.x, 1u);
      s_last = done == gridDim.y - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // split weights w[q][s] = e^(m_s - M_q) / L_q, computed once per query in
    // shared memory (the page buffers are free now), then a parallel sum
    float* wts = reinterpret_cast<float*>(smem);            // [QN][n_split]
    for (int t = threadIdx.x; t < QN * a.n_split; t += blockDim.x) {
      const int q = t / a.n_split, sp = t % a.n_split, i = q / G, gg = q % G;
      const size_t pi = ((size_t)(b * a.R + i) * a.nq + kvh * G + gg) * a.n_split + sp;
      wts[t] = __ldcg(a.part_ml + pi * 2);
    }
    __syncthreads();
    for (int q = threadIdx.x; q < QN; q += blockDim.x) {
      const int i = q / G, gg = q % G;
      const size_t base_i = ((size_t)(b * a.R + i) * a.nq + kvh * G + gg) * a.n_split;
      float M = -INFINITY;
      for (int sp = 0; sp < a.n_split; ++sp) M = fmaxf(M, wts[q * a.n_split + sp]);
      float L = 0.f;
      for (int sp = 0; sp < a.n_split; ++sp) {
        const float ms = wts[q * a.n_split + sp];
        const float w = ms == -INFINITY ? 0.f : __expf(ms - M);
        wts[q * a.n_split + sp] = w;
        L += __ldcg(a.part_ml + (base_i + sp) * 2 + 1) * w;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int sp = 0; sp < a.n_split; ++sp) wts[q * a.n_split + sp] *= inv;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < QN * HD; t += blockDim.x) {
      const int q = t / HD, d = t % HD, i = q / G, gg = q % G;
      const int m = b * a.R + i, h = kvh * G + gg;
      const float* po = a.part_o + ((size_t)m * a.nq + h) * a.n_split * HD + d;
      const float* w = wts + q * a.n_split;
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      int sp = 0;
      for (; sp + 4 <= a.n_split; sp += 4) {
        acc0 = fmaf(w[sp], __ldcg(po + (size_t)sp * HD), acc0);
        acc1 = fmaf(w[sp + 1], __ldcg(po + (size_t)(sp + 1) * HD), acc1);
        acc2 = fmaf(w[sp + 2], __ldcg(po + (size_t)(sp + 2) * HD), acc2);
        acc3 = fmaf(w[sp + 3], __ldcg(po + (size_t)(sp + 3) * HD), acc3);
      }
      for (; sp < a.n_split; ++sp) acc0 = fmaf(w[sp], __ldcg(po + (size_t)sp * HD), acc0);
      a.out[(size_t)m * a.nq * HD + h * HD + d] = (acc0 + acc1) + (acc2 + acc3);
    }
    if (threadIdx.x == 0) counters[blockIdx.x] = 0u;
  }
};

template <int HD>
__global__ void __launch_bounds__(256) attn_tc_kernel(AttnArgs a, int pps, unsigned int* counters) {
  extern __shared__ __align__(16) unsigned char smem[];
  AttnTc<HD>::run(a, pps, counters, smem);
}

}  // namespace

size_t attention_tc_smem(int hd, int qn) {
  const int qt = (qn + 15) / 16, st = hd + 8;
  return (size_t)(2 * qt * 16 * st + 4 * PAGE * st) * 2;
}

void setup_attn_tc_attributes() {
  cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

// Splits of the page range: about one CTA per SM, at most 32 splits (the
// merge reads every split's partial).
int attention_tc_splits(int B, int nkv, int max_pages, int* pps) {
  const int target = std::max(1, num_sms() / std::max(1, B * nkv));
  const int n = std::min(std::min(max_pages, target), 32);
  *pps = (max_pages + n - 1) / n;
  return (max_pages + *pps - 1) / *pps;
}

int attention_tc(const AttnArgs& a, unsigned int* counters, int pps, cudaStream_t st) {
  const int QN = a.R * (a.nq / a.nkv);
  const int qt = (QN + 15) / 16;
  const size_t smem = attention_tc_smem(a.hd, QN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.nkv, a.n_split);
  cfg.blockDim = dim3(qt > 4 ? 256 : 128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.hd == 128) e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<128>, a, pps, counters);
  else if (a.hd == 64) e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<64>, a, pps, counters);
  else return -2;
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace spec
