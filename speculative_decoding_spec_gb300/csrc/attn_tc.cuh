// attn_tc.cuh -- causal attention of the verified rows over a bf16 paged KV
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
// A split (sequence b, KV head, page range) walks its pages in
// rounds of cp.async loads (the first round in one burst with the queries). All rows x GQA-group queries of the sequence
// form 16-query tiles, one warp per tile: S = Q K^T (scores), online softmax,
// O += P V with V fragments from ldmatrix.trans. Q and P enter the MMAs as
// bf16 hi + lo pairs (two MMAs each), so scores and outputs carry fp32-level
// accuracy against the exact bf16 keys and values. Each split writes an
// unnormalised partial (max, sum, O); the last CTA of (b, KV head) to finish
// merges the splits with log-sum-exp weights -- no CTA waits for another.
#pragma once
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"

namespace spec {
namespace atc {

constexpr int PAGE = 64;
constexpr int PGS_MAX = 256;  // page ids of a split cached in shared memory

static SPEC_DEV void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

static SPEC_DEV uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// hi = bf16(x), lo = bf16(x - hi), for a pair
static SPEC_DEV void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = pack2(x0, x1);
  lo = pack2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

static SPEC_DEV void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
static SPEC_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
static SPEC_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

static SPEC_DEV void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, const void* smem) {
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

  // prefetch.global.L2 of the K and V planes of the pages split `by` reads
  static SPEC_DEV void prefetch(const AttnArgs& a, int pps, int bx, int by) {
    const int b = bx / a.nkv, kvh = bx % a.nkv;
    const int slot = a.seq_ids[b];
    const int lmax = a.seq_len[slot] + a.R - 1 + a.key_extra;
    const int npages = min((lmax + PAGE - 1) / PAGE, a.max_pages);
    const int p0 = by * pps, p1 = min(p0 + pps, npages);
    const __nv_bfloat16* base = (const __nv_bfloat16*)a.pool + (size_t)a.layer * a.layer_elems;
    constexpr int LINES = PAGE * HD * 2 / 128;  // 128-byte lines per K (or V) plane
    for (int i = threadIdx.x; i < (p1 - p0) * 2 * LINES; i += blockDim.x) {
      const int p = p0 + i / (2 * LINES), r = i % (2 * LINES), plane = r / LINES, ln = r % LINES;
      const int pg = a.block_table[(size_t)slot * a.max_pages + p];
      if (pg >= 0 && pg < a.n_pages)
        prefetch_l2(base + (((size_t)pg * 2 + plane) * a.nkv + kvh) * PAGE * HD + ln * 64);
    }
  }

  // Warp roles: QT 16-query tiles x PW page slots x KG key groups of a page.
  static SPEC_DEV int key_groups(int QT) { return QT == 1 ? 4 : 1; }
  static SPEC_DEV int page_slots(int QT, int NW) {
    const int ps = NW / (QT * key_groups(QT));
    return ps > 0 ? ps : 1;
  }

  // S = Q K^T over NT*8 keys of a page starting at key kb, online softmax,
  // O += P V. Rows r0 = 16*qt + g and r1 = r0 + 8 of the query tile.
  template <int NT>
  static SPEC_DEV void page_tile(const __nv_bfloat16* Qh, const __nv_bfloat16* Ql, const __nv_bfloat16* Ks,
                                 const __nv_bfloat16* Vs, int r0, int kb, int key0, int nk0, int nk1,
                                 unsigned int tm0, unsigned int tm1, int L0, float scale,
                                 float& m0, float& m1, float& l0, float& l1, float (&o)[NDT][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
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
      for (int nt = 0; nt < NT; ++nt) {
        const __nv_bfloat16* kr = Ks + (kb + 8 * nt + g) * ST + 16 * ks + 2 * c;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 8);
        mma_bf16(s[nt], ah0, ah1, ah2, ah3, b0, b1);
        mma_bf16(s[nt], al0, al1, al2, al3, b0, b1);
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + kb + 8 * nt + 2 * c + e;
        s[nt][e] = key < nk0 && tree_visible(tm0, L0, key) ? s[nt][e] * scale : -INFINITY;
        s[nt][2 + e] = key < nk1 && tree_visible(tm1, L0, key) ? s[nt][2 + e] * scale : -INFINITY;
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
    for (int nt = 0; nt < NT; ++nt)
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
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      uint32_t ph0, pl0, ph1, pl1, ph2, pl2, ph3, pl3;
      split2(s[2 * kk][0], s[2 * kk][1], ph0, pl0);
      split2(s[2 * kk][2], s[2 * kk][3], ph1, pl1);
      split2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph2, pl2);
      split2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph3, pl3);
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt) {
        uint32_t b0, b1;
        ldmatrix_x2_trans(b0, b1, Vs + (kb + 16 * kk + (lane & 15)) * ST + 8 * dt);
        mma_bf16(o[dt], ph0, ph1, ph2, ph3, b0, b1);
        mma_bf16(o[dt], pl0, pl1, pl2, pl3, b0, b1);
      }
    }
  }

  // bx = sequence * n_kv + KV head, by = split (of a.n_split); the split covers
  // pages [by*pps, (by+1)*pps), pps a multiple of the page slots. standalone:
  // own launch (PDL waits) rather than a step of the persistent pass kernel.
  // pw_cap > 0 caps the page slots (and so the shared memory) below what the
  // CTA's warps could fill.
  static SPEC_DEV void run(const AttnArgs& a, int pps, unsigned int* counters, unsigned char* smem, int bx,
                           int by, bool standalone, size_t smem_bytes, int pw_cap = 0) {
    const int b = bx / a.nkv;
    const int slot = a.seq_ids[b];
    const int lmax = a.seq_len[slot] + a.R - 1 + a.key_extra;
    const int npages = min((lmax + PAGE - 1) / PAGE, a.max_pages);
    const int p0 = by * pps, p1 = min(p0 + pps, npages);
    if (standalone) prefetch(a, pps, bx, by);
    run_split(a, bx, p0, p1, by, a.n_split, counters, smem, standalone, smem_bytes, pw_cap);
  }

  // Balanced stand-alone launch for batches: each (sequence, KV head) pair
  // gets one CTA plus a share of the remaining CTAs proportional to its pages
  // (lengths read on the device, so the grid is fixed for graph capture),
  // capped so that a CTA has at least a round of page slots; CTA j of a pair
  // takes pages [np*j/k, np*(j+1)/k) as split j of k. Each CTA has one piece,
  // and the longest sequences get the most CTAs.
  static SPEC_DEV void run_balanced(const AttnArgs& a, unsigned int* counters, unsigned char* smem,
                                    size_t smem_bytes) {
    __shared__ int s_np[64];   // pages of each sequence
    __shared__ int s_k[64];    // CTAs per pair of each sequence
    __shared__ int s_kb[65];   // first CTA of each sequence's pairs
    const int nkv = a.nkv, B = a.B;
    const int G = a.nq / nkv, QT = (a.R * G + 15) / 16;
    const int PW = page_slots(QT, blockDim.x >> 5);
    if ((int)threadIdx.x < B) {
      const int lmax = a.seq_len[a.seq_ids[threadIdx.x]] + a.R - 1 + a.key_extra;
      s_np[threadIdx.x] = min((lmax + PAGE - 1) / PAGE, a.max_pages);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      long long P = 0;
      for (int b = 0; b < B; ++b) P += (long long)s_np[b] * nkv;
      const long long extra = (long long)gridDim.x - (long long)B * nkv;  // CTAs beyond one per pair
      int acc = 0;
      for (int b = 0; b < B; ++b) {
        int k = 1;
        if (extra > 0 && P > 0) k += (int)(((long long)s_np[b] * extra) / P);
        k = min(k, max(1, s_np[b] / PW));
        s_k[b] = k;
        s_kb[b] = acc;
        acc += k * nkv;
      }
      s_kb[B] = acc;
    }
    __syncthreads();
    const int cta = blockIdx.x;
    if (cta >= s_kb[B]) {
      grid_dep_wait();
      grid_dep_launch();
      return;
    }
    int b = 0;
    while (b + 1 < B && s_kb[b + 1] <= cta) ++b;
    const int k = s_k[b], np = s_np[b];
    const int kvh = (cta - s_kb[b]) / k, j = (cta - s_kb[b]) - kvh * k;
    const int p0 = (int)(((long long)np * j) / k), p1 = (int)(((long long)np * (j + 1)) / k);
    // pages do not depend on the previous kernel: pull this piece's K and V
    // planes towards L2 (one bulk prefetch per 16 KB plane) before the wait
    {
      const __nv_bfloat16* base = (const __nv_bfloat16*)a.pool + (size_t)a.layer * a.layer_elems;
      for (int i = threadIdx.x; i < (p1 - p0) * 2; i += blockDim.x) {
        const int pg = a.block_table[(size_t)a.seq_ids[b] * a.max_pages + p0 + (i >> 1)];
        if (pg >= 0 && pg < a.n_pages)
          prefetch_l2_bulk(base + (((size_t)pg * 2 + (i & 1)) * nkv + kvh) * PAGE * HD, PAGE * HD * 2);
      }
    }
    run_split(a, b * nkv + kvh, p0, p1, j, k, counters, smem, true, smem_bytes, 0);
  }

  // One split of (sequence, KV head) bx: pages [p0, p1) as split `split` of
  // `nsplit`; partials are indexed with stride a.n_split (>= nsplit).
  static SPEC_DEV void run_split(const AttnArgs& a, int bx, int p0, int p1, int split, int nsplit,
                                 unsigned int* counters, unsigned char* smem, bool standalone, size_t smem_bytes,
                                 int pw_cap) {
    const int b = bx / a.nkv, kvh = bx % a.nkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
    const int NW = blockDim.x >> 5;
    const int G = a.nq / a.nkv, QN = a.R * G, QT = (QN + 15) / 16;
    const int KG = key_groups(QT);
    const int PW = pw_cap > 0 && page_slots(QT, NW) > pw_cap ? pw_cap : page_slots(QT, NW);
    const int qt = warp % QT, rest = warp / QT, kg = rest % KG, pslot = rest / KG;
    const bool active = warp < QT * KG * PW;
    __nv_bfloat16* Qh = reinterpret_cast<__nv_bfloat16*>(smem);
    __nv_bfloat16* Ql = Qh + QT * 16 * ST;
    float* qf = reinterpret_cast<float*>(Ql + QT * 16 * ST);  // [QN][HD] fp32 query rows
    float* rf = qf + (size_t)QN * HD;                          // [R][HD] cos/sin rows
    __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(rf + (size_t)a.R * HD);  // [PW][64][ST]
    __nv_bfloat16* Vb = Kb + PW * PAGE * ST;                   // [PW][64][ST]
    __shared__ int s_last;

    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int lmax = L0 + a.R - 1 + a.key_extra;  // keys of the last row
    const __nv_bfloat16* base = (const __nv_bfloat16*)a.pool + (size_t)a.layer * a.layer_elems;
    // the split's page ids (the block table does not change within a pass):
    // read in parallel and checked before the dependency wait
    __shared__ int s_pgs[PGS_MAX];
    __shared__ int s_bad;
    const bool ids_cached = p1 - p0 <= PGS_MAX;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int p = p0 + (int)threadIdx.x; p < p1; p += blockDim.x) {
      const int pg = a.block_table[(size_t)slot * a.max_pages + p];
      if (pg < 0 || pg >= a.n_pages) s_bad = 1;
      if (ids_cached) s_pgs[p - p0] = pg;
    }
    if (standalone) {
      grid_dep_wait();
      grid_dep_launch();
    }
    __syncthreads();
    const bool pages_ok = s_bad == 0;
    if (!pages_ok && threadIdx.x == 0) set_error(a.err, SPEC_ERR_CAPACITY);
    const int pend = pages_ok ? p1 : p0;

    // K and V of pages [rb, rb + nr) into the page slots (rows past the keys zeroed)
    constexpr int CPR = HD / 8;
    auto issue_pages = [&](int rb, int nr) {
      for (int t = threadIdx.x; t < nr * PAGE * CPR; t += blockDim.x) {
        const int ps = t / (PAGE * CPR), rr = (t / CPR) % PAGE, ch = t % CPR;
        const int p = rb + ps;
        const int pg = ids_cached ? s_pgs[p - p0] : a.block_table[(size_t)slot * a.max_pages + p];
        const int nk = min(PAGE, lmax - p * PAGE);
        __nv_bfloat16* Ks = Kb + (size_t)ps * PAGE * ST;
        __nv_bfloat16* Vs = Vb + (size_t)ps * PAGE * ST;
        if (rr < nk) {
          const __nv_bfloat16* kp = base + (((size_t)pg * 2 + 0) * a.nkv + kvh) * PAGE * HD;
          const __nv_bfloat16* vp = base + (((size_t)pg * 2 + 1) * a.nkv + kvh) * PAGE * HD;
          cp_async16(Ks + rr * ST + ch * 8, kp + rr * HD + ch * 8);
          cp_async16(Vs + rr * ST + ch * 8, vp + rr * HD + ch * 8);
        } else {
          *reinterpret_cast<uint4*>(Ks + rr * ST + ch * 8) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(Vs + rr * ST + ch * 8) = make_uint4(0, 0, 0, 0);
        }
      }
    };

    // queries: q = i*G + gg is head kvh*G + gg of row b*R + i. The fp32 rows
    // (and RoPE rows when asked) come to shared memory in one burst with the
    // first round's pages (L2 only: they come from other CTAs or the previous
    // kernel), then are split into bf16 hi/lo with RoPE applied.
    for (int t = threadIdx.x; t < QN * (HD / 4); t += blockDim.x) {
      const int q = t / (HD / 4), c4 = t % (HD / 4), i = q / G, gg = q % G;
      cp_async16(qf + (size_t)q * HD + 4 * c4, a.q + (size_t)(b * a.R + i) * a.ldq + (kvh * G + gg) * HD + 4 * c4);
    }
    if (a.rope_cs)
      for (int t = threadIdx.x; t < a.R * (HD / 4); t += blockDim.x) {
        const int i = t / (HD / 4), c4 = t % (HD / 4);
        cp_async16(rf + (size_t)i * HD + 4 * c4, a.rope_cs + (size_t)(b * a.R + i) * HD + 4 * c4);
      }
    if (p0 < pend) issue_pages(p0, min(PW, pend - p0));
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int t = threadIdx.x; t < QT * 16 * (HD / 2); t += blockDim.x) {
      const int q = t / (HD / 2), d2 = (t % (HD / 2)) * 2;
      float x0 = 0.f, x1 = 0.f;
      if (q < QN) {
        const float* qr = qf + (size_t)q * HD;
        if (a.rope_cs) {
          const float* cs = rf + (size_t)(q / G) * HD;
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

    const int r0 = 16 * qt + g, r1 = r0 + 8;
    const int nk0 = r0 < QN ? L0 + r0 / G + a.key_extra : 0;
    const int nk1 = r1 < QN ? L0 + r1 / G + a.key_extra : 0;
    const unsigned int tm0 = a.tree_mask && r0 < QN ? a.tree_mask[b * a.R + r0 / G] : ~0u;
    const unsigned int tm1 = a.tree_mask && r1 < QN ? a.tree_mask[b * a.R + r1 / G] : ~0u;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[NDT][4];
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    const float scale = rsqrtf((float)HD);

    // rounds of up to PW pages: all loads of a round in flight, then compute
    // (the first round's loads went with the queries)
    for (int rb = p0; rb < pend; rb += PW) {
      const int nr = min(PW, pend - rb);
      __syncthreads();
      if (rb != p0) {
        issue_pages(rb, nr);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
      }
      if (active && pslot < nr) {
        const __nv_bfloat16* Ks = Kb + (size_t)pslot * PAGE * ST;
        const __nv_bfloat16* Vs = Vb + (size_t)pslot * PAGE * ST;
        const int key0 = (rb + pslot) * PAGE;
        if (KG == 4)
          page_tile<2>(Qh, Ql, Ks, Vs, r0, 16 * kg, key0, nk0, nk1, tm0, tm1, L0, scale, m0, m1, l0, l1, o);
        else
          page_tile<8>(Qh, Ql, Ks, Vs, r0, 0, key0, nk0, nk1, tm0, tm1, L0, scale, m0, m1, l0, l1, o);
      }
    }
    __syncthreads();

    // combine the warps of each query tile (shared memory, fixed warp order)
    constexpr int RS = HD + 2;  // o[HD], m, l per row
    float* scr = reinterpret_cast<float*>(Kb);  // [active warps][16][RS]
    float* mrow = scr + (size_t)QT * KG * PW * 16 * RS;  // [QT*16] combined max per query row
    if (active) {
      float* w0 = scr + ((size_t)warp * 16 + g) * RS;
      float* w1 = w0 + 8 * RS;
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt) {
        w0[8 * dt + 2 * c] = o[dt][0];
        w0[8 * dt + 2 * c + 1] = o[dt][1];
        w1[8 * dt + 2 * c] = o[dt][2];
        w1[8 * dt + 2 * c + 1] = o[dt][3];
      }
      if (c == 0) {
        w0[HD] = m0; w0[HD + 1] = l0;
        w1[HD] = m1; w1[HD + 1] = l1;
      }
    }
    __syncthreads();
    // per (tile, row): the warps' weights e^(m_j - M) and the combined sum L,
    // written over each warp's m slot (weight) and the first warp's l slot (L)
    const int nw_tile = KG * PW;
    for (int t = threadIdx.x; t < QT * 16; t += blockDim.x) {
      const int qq = t / 16, row = t % 16;
      float M = -INFINITY;
      for (int j = 0; j < nw_tile; ++j) M = fmaxf(M, scr[((size_t)(qq + j * QT) * 16 + row) * RS + HD]);
      float L = 0.f;
      for (int j = 0; j < nw_tile; ++j) {
        float* r = scr + ((size_t)(qq + j * QT) * 16 + row) * RS;
        const float wgt = r[HD] == -INFINITY ? 0.f : __expf(r[HD] - M);
        L += r[HD + 1] * wgt;
        r[HD] = wgt;
      }
      scr[((size_t)qq * 16 + row) * RS + HD + 1] = L;
      mrow[t] = M;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < QN * HD; t += blockDim.x) {
      const int q = t / HD, d = t % HD, qq = q / 16, row = q % 16;
      float acc = 0.f;
      for (int j = 0; j < nw_tile; ++j) {
        const float* r = scr + ((size_t)(qq + j * QT) * 16 + row) * RS;
        acc = fmaf(r[HD], r[d], acc);
      }
      const float L = scr[((size_t)qq * 16 + row) * RS + HD + 1];
      const int i = q / G, gg = q % G;
      const int m = b * a.R + i, h = kvh * G + gg;
      if (nsplit == 1) {
        a.out[(size_t)m * a.nq * HD + h * HD + d] = L > 0.f ? acc / L : 0.f;
      } else {
        const size_t pidx = ((size_t)m * a.nq + h) * a.n_split + split;
        a.part_o[pidx * HD + d] = acc;
        if (d == 0) {
          a.part_ml[pidx * 2] = mrow[qq * 16 + row];
          a.part_ml[pidx * 2 + 1] = L;
        }
      }
    }
    if (nsplit == 1) return;

    // the last split CTA of (b, KV head) merges: the arrival is a release
    // (this CTA's partials, ordered by the barrier) and an acquire (the other
    // splits' partials) in one atomic
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned int done = atomic_add_acq_rel(counters + bx, 1u);
      s_last = done == (unsigned int)nsplit - 1;
    }
    __syncthreads();
    if (!s_last) return;
    // split weights w[q][s] = e^(m_s - M_q) / L_q in shared memory; the split
    // partials of all queries are first copied to shared memory in one burst
    // (every request in flight) when they fit
    float* wts = reinterpret_cast<float*>(smem);                  // [QN][n_split]
    float* pst = wts + ((QN * nsplit + 3) & ~3);               // [QN][n_split][HD]
    const size_t pbytes = (size_t)QN * nsplit * HD * 4;
    const bool staged = (size_t)((unsigned char*)pst - smem) + pbytes <= smem_bytes;
    if (staged) {
      for (int t = threadIdx.x; t < QN * nsplit * (HD / 4); t += blockDim.x) {
        const int q = t / (nsplit * (HD / 4)), r = t % (nsplit * (HD / 4));
        const int sp = r / (HD / 4), c4 = r % (HD / 4), i = q / G, gg = q % G;
        const size_t pi = ((size_t)(b * a.R + i) * a.nq + kvh * G + gg) * a.n_split + sp;
        cp_async16(pst + ((size_t)q * nsplit + sp) * HD + 4 * c4, a.part_o + pi * HD + 4 * c4);
      }
      cp_async_commit();
    }
    float* lsp = pst + (staged ? (size_t)QN * nsplit * HD : 0);   // [QN][n_split] split sums
    const bool lsm = (size_t)((unsigned char*)(lsp + QN * nsplit) - smem) <= smem_bytes;
    for (int t = threadIdx.x; t < QN * nsplit; t += blockDim.x) {
      const int q = t / nsplit, sp = t % nsplit, i = q / G, gg = q % G;
      const size_t pi = ((size_t)(b * a.R + i) * a.nq + kvh * G + gg) * a.n_split + sp;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + pi);
      wts[t] = ml.x;
      if (lsm) lsp[t] = ml.y;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < QN; q += blockDim.x) {
      const int i = q / G, gg = q % G;
      const size_t base_i = ((size_t)(b * a.R + i) * a.nq + kvh * G + gg) * a.n_split;
      float M = -INFINITY;
      for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, wts[q * nsplit + sp]);
      float L = 0.f;
      for (int sp = 0; sp < nsplit; ++sp) {
        const float ms = wts[q * nsplit + sp];
        const float w = ms == -INFINITY ? 0.f : __expf(ms - M);
        wts[q * nsplit + sp] = w;
        L += (lsm ? lsp[q * nsplit + sp] : __ldcg(a.part_ml + (base_i + sp) * 2 + 1)) * w;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int sp = 0; sp < nsplit; ++sp) wts[q * nsplit + sp] *= inv;
    }
    if (staged) cp_async_wait<0>();
    __syncthreads();
    for (int t = threadIdx.x; t < QN * HD; t += blockDim.x) {
      const int q = t / HD, d = t % HD, i = q / G, gg = q % G;
      const int m = b * a.R + i, h = kvh * G + gg;
      const float* w = wts + q * nsplit;
      float acc0 = 0.f, acc1 = 0.f;
      if (staged) {
        const float* po = pst + (size_t)q * nsplit * HD + d;
        int sp = 0;
        for (; sp + 2 <= nsplit; sp += 2) {
          acc0 = fmaf(w[sp], po[(size_t)sp * HD], acc0);
          acc1 = fmaf(w[sp + 1], po[(size_t)(sp + 1) * HD], acc1);
        }
        if (sp < nsplit) acc0 = fmaf(w[sp], po[(size_t)sp * HD], acc0);
      } else {
        // 8 splits' loads in flight at a time; even splits to acc0 and odd
        // ones to acc1 in order, as in the staged branch
        const float* po = a.part_o + ((size_t)m * a.nq + h) * a.n_split * HD + d;
        for (int sp = 0; sp < nsplit; sp += 8) {
          float u[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) u[i] = __ldcg(po + (size_t)min(sp + i, nsplit - 1) * HD);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            if (sp + i < nsplit) acc0 = fmaf(w[sp + i], u[i], acc0);
            if (sp + i + 1 < nsplit) acc1 = fmaf(w[sp + i + 1], u[i + 1], acc1);
          }
        }
      }
      a.out[(size_t)m * a.nq * HD + h * HD + d] = acc0 + acc1;
    }
    if (threadIdx.x == 0) counters[bx] = 0u;
  }
};

}  // namespace atc
}  // namespace spec
