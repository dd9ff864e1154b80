// attn_flash.cu -- paged attention of the verified rows (and of the drafter's
// cross-attention) on the fifth-generation tensor cores: head_dim 128, bf16
// cache, up to 32 query rows per (sequence, KV head).
//
// Row i of sequence b sits at position seq_len + i and attends keys
// 0 .. seq_len + i (its own key and those of earlier rows of the same pass
// included): the target checks every drafted position in one pass ("Gemma 4's
// MTP drafter explained" (molayo1419.me), section "How does speculative
// decoding work?"). The drafter's cross-attention runs the same kernel on the
// target's last-layer pages with keys 0 .. seq_len - 1 ("Accelerating Gemini
// Nano on Pixel with frozen multi-token prediction" (ai-news-spoon), section
// "Zero-copy architecture").
//
// Shape. The queries of one (sequence, KV head) pair are few -- R rows times
// the GQA group, 6 to 30 -- while the keys are thousands, so the keys take the
// MMA's M side: a block is two pages (128 keys), and
//   S^T[key][q] = K_block . Q^T     (M = 128 keys, N = 2 x QNP, K = head_dim)
//   O^T[d][q]  += V_block^T . P^T   (M = 128 dims, N = 2 x QNP, K = 128 keys)
// with the queries (and the probabilities) entering as bf16 hi + lo column
// halves of the N side, so scores and outputs carry fp32-level accuracy
// against the exact bf16 keys and values. Both accumulators live in tensor
// memory. K and V pages arrive by TMA in the 128-byte swizzle layout: K is a
// K-major A operand, V (stored [key][dim]) an MN-major one, the same bytes.
//
// Roles (one CTA per SM): warp 0 issues the TMA loads (K ring of 2 blocks, V
// ring of 3: a V tile is needed a whole softmax later than the K tile of the
// same block), warp 1 the MMAs, warps 2-9 run the softmax in two groups of
// four (one warp per TMEM lane quarter, each group half of the query columns):
// thread = key of the block, so a column (query) maximum is a transposing warp
// reduction plus a 4-warp combine in shared memory. The running maximum is
// only raised when some score exceeds it by 2^8 (one OR-reducing barrier per
// block decides; then O^T is rescaled in tensor memory), so probabilities stay
// below 256 and the column reductions are rare. Each thread keeps its own
// partial sums; they are reduced once per split. The probabilities are written
// as an MN-major operand (one 128-byte row per key, two tiles alternating).
//
// Work split. When the pairs are fewer than the SMs, each pair gets one CTA
// plus a share of the others in proportion to its blocks (computed on the
// device from the lengths, so the grid is fixed), and the CTAs of a pair
// write unnormalised partials (O, max, sum), arrive on the pair's counter, wait
// (bounded) until all have arrived and then each merges a slice of the query
// rows with log-sum-exp weights. The plan is a warp-wide prefix sum over the
// pairs; the partials are written CTA-major (32 rows a CTA), one compact block
// the pair's CTAs read back. All CTAs of the grid are resident at once (grid
// <= SMs, one CTA per SM by its shared memory), and a dependent kernel is only
// launched once every CTA of this grid has started, so the wait cannot block
// on a CTA that never runs. A wait that runs out records SPEC_ERR_TIMEOUT and
// skips the merge; every CTA still departs, and the last to depart resets the
// pair's counters. Every mbarrier wait is bounded too.
//
// The merged rows can also be written as the O projection's bf16 (or fp16)
// hi + lo activation planes (AttnArgs.planes), so that projection needs no
// preparation kernel.
//
// The code after the last block runs once per CTA, out of a cold instruction
// cache and at the same moment on every SM, so it is kept short: an unrolled
// loop with per-column index divisions there cost about 8 us a launch, and a
// serial plan loop with 64-bit divisions another 9 us at 64 pairs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "mbar.cuh"

namespace spec {
namespace fa {

constexpr int HD = 128;
constexpr int PAGE = 64;
constexpr int BK = 128;                       // keys per block (two pages)
constexpr int NTHR = 320;                     // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr int SM0 = 64;                       // first softmax thread
constexpr int NSM = 256;                      // softmax threads: 2 column groups x 4 lane quarters
constexpr int KSLOTS = 2, VSLOTS = 3;
constexpr int HALF_BYTES = BK * 128;          // one 64-dim half of a block: 128 rows x 128 B
constexpr int TILE_BYTES = 2 * HALF_BYTES;    // K (or V) of a block: 32 KB
constexpr int BOX_BYTES = PAGE * 128;         // one TMA box: 64 rows x 64 dims
constexpr int PGS_CACHE = 256;                // page ids of a CTA's range kept in shared memory
constexpr int MAX_PAIRS = 1024;
constexpr int MERGE_MAX = 256;                // (query row, split) pairs one CTA merges at most
constexpr int TMEM_COLS = 256;                // S^T x 2 buffers + O^T, each 2 x QNP <= 64 columns
constexpr float TAU = 8.f;                    // raise the running maximum past 2^8 growth
constexpr unsigned SPIN_LIMIT = 1u << 26;
constexpr unsigned long long MERGE_WAIT_NS = 1000000000ull;  // 1 s

struct Plan {
  int npairs, grid, R, G, QN;
  float scale2;                               // log2(e) / sqrt(head_dim)
  int wait_extra;                             // added to the merge's arrival target (test hook)
};

SPEC_DEV void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SPEC_DEV void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory descriptors, 128-byte swizzle (bits 61-63 = 2, bits 46-48 =
// 0b001). K-major: 8-row groups 1024 B apart (stride offset), leading offset
// unused. MN-major: the 64-element halves of the M side `lbo` bytes apart
// (leading offset), 8-row groups of the K side 1024 B apart (stride offset).
SPEC_DEV uint64_t desc_k(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
SPEC_DEV uint64_t desc_mn(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, N >> 3 at
// bit 17, M >> 4 at bit 24; bit 15 = A is MN-major, bit 16 = B is MN-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

SPEC_DEV void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
SPEC_DEV void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(bar))
               : "memory");
}
SPEC_DEV void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          sa(dst)),
      "l"(map), "r"(x), "r"(y), "r"(sa(bar))
      : "memory");
}
// With an L2 cache policy: the target's own layers read each layer's pages
// once per pass, so they go first when L2 needs room (the drafter re-reads the
// last layer's pages at every step and keeps the default).
SPEC_DEV void tma_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(sa(dst)),
      "l"(map), "r"(x), "r"(y), "r"(sa(bar)), "l"(policy)
      : "memory");
}
SPEC_DEV uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
SPEC_DEV void ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
SPEC_DEV void ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
SPEC_DEV void st8(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
SPEC_DEV void ld4(uint32_t taddr, float* v) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
SPEC_DEV void st4(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3]))
               : "memory");
}
SPEC_DEV void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
SPEC_DEV void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// N (4, 8 or a multiple of 16) consecutive columns of this warp's 32 lanes.
template <int N>
SPEC_DEV void ldn(uint32_t taddr, float* v) {
  if constexpr (N % 16 == 0) {
#pragma unroll
    for (int i = 0; i < N / 16; ++i) ld16(taddr + 16 * i, v + 16 * i);
  } else if constexpr (N == 8) {
    ld8(taddr, v);
  } else {
    ld4(taddr, v);
  }
}
template <int N>
SPEC_DEV void stn(uint32_t taddr, const float* v) {
  if constexpr (N % 8 == 0) {
#pragma unroll
    for (int i = 0; i < N / 8; ++i) st8(taddr + 8 * i, v + 8 * i);
  } else {
    st4(taddr, v);
  }
}

// Named barrier of the 4 softmax warps.
SPEC_DEV void sm_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

SPEC_DEV bool wait_phase(uint64_t* b, unsigned parity, volatile int* abort_s, int* err) {
  for (unsigned it = 0; it < SPIN_LIMIT; ++it) {
    if (mbar_test(b, parity)) return true;
    if (*abort_s) return false;
  }
  *abort_s = 1;
  set_error(err, SPEC_ERR_TIMEOUT);
  return false;
}
SPEC_DEV void drain_phase(uint64_t* b, unsigned parity) {
  for (unsigned it = 0; it < SPIN_LIMIT; ++it)
    if (mbar_test(b, parity)) return;
}

// Byte offset of element (row, col) of a K-major operand region of 128-byte
// rows in the 128-byte swizzle layout (16-byte chunk c of row r at c ^ (r % 8)).
SPEC_DEV uint32_t swz(int row, int col_bytes) {
  return (uint32_t)(row * 128 + ((((col_bytes >> 4) ^ (row & 7)) << 4) | (col_bytes & 15)));
}

// Transposing warp reduction: v[0..N) per lane -> lane l holds the reduction
// of column (l % N) over all 32 lanes (N a power of two <= 32).
template <int N, bool MAX>
SPEC_DEV float col_reduce(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = N / 2; o >= 1; o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      const float got = __shfl_xor_sync(FULL, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = N; o < 32; o <<= 1) {
    const float got = __shfl_xor_sync(FULL, r, o);
    r = MAX ? fmaxf(r, got) : r + got;
  }
  return r;
}

// Shared memory of a CTA. The query planes and probability tiles always have
// 64 columns on the N side (queries' hi parts in columns 0-31, lo parts in
// 32-63), so every MMA has N = 64 whatever the number of queries.
struct Smem {
  static constexpr int QP_HALF = 64 * 128;             // one 64-dim half of the query planes
  static constexpr int P_BYTES = BK * 128;             // probability tile: one 128-byte row per key
  static constexpr size_t K_OFF = 0;
  static constexpr size_t V_OFF = K_OFF + (size_t)KSLOTS * TILE_BYTES;
  static constexpr size_t Q_OFF = V_OFF + (size_t)VSLOTS * TILE_BYTES;
  static constexpr size_t P_OFF = Q_OFF + 2 * QP_HALF;
  static constexpr size_t X_OFF = P_OFF + 2 * P_BYTES;  // small items (below)
  // barriers: kfull[3] kempty[3] vfull[2] vempty[2] sfull[2] pfull[2] pvdone[2] drain
  static constexpr int NBAR = 2 * KSLOTS + 2 * VSLOTS + 2 + 2 + 2 + 1;
  static constexpr size_t BAR_OFF = X_OFF;
  static constexpr size_t RED_OFF = BAR_OFF + NBAR * 8;          // float [8][32]
  static constexpr size_t MU_OFF = RED_OFF + 8 * 32 * 4;         // float [32] running max (log2 units)
  static constexpr size_t AL_OFF = MU_OFF + 32 * 4;              // float [32] rescale factors
  static constexpr size_t L_OFF = AL_OFF + 32 * 4;               // float [32] final sums
  static constexpr size_t PG_OFF = L_OFF + 32 * 4;               // int [PGS_CACHE]
  static constexpr size_t ML_OFF = PG_OFF + PGS_CACHE * 4;       // float2 [MERGE_MAX] merge weights
  static constexpr size_t MISC_OFF = ML_OFF + MERGE_MAX * 8;     // int [16]
  static constexpr size_t COFF_OFF = MISC_OFF + 16 * 4;          // int [32] output offset of each query column
  static constexpr size_t BYTES = COFF_OFF + 32 * 4;
  static constexpr size_t ALLOC = BYTES + 1024;                  // base alignment slack
};

struct Work {
  int b, kvh, j, np, blk0, blk1, npages;
};

SPEC_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Barrier 1 over the 8 softmax warps, returning the OR of `v` over them.
SPEC_DEV bool sm_any(bool v) {
  unsigned r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, 1, 256, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((unsigned)v)
      : "memory");
  return r != 0;
}

template <int QNP>
struct Cta {
  using S = Smem;
  const AttnArgs& a;
  const Plan& p;
  const CUtensorMap* tm;
  unsigned int* cnt;
  unsigned char* sm;
  uint64_t *kfull, *kempty, *vfull, *vempty, *sfull, *pfull, *pvdone, *drain;
  float *red, *mu, *alpha, *lfin;
  int* coff;                 // [32] offset of query column c's head in `out` (row-major [M][nq*HD])
  int* pgs;
  int* misc;                 // [0] merge ok, [2] tmem base, [3] abort
  volatile int* abort_s;
  uint32_t tmem;
  Work w;
  int slot, L0;
  int kpre, vpre;  // K and V blocks the producer issued before the dependency wait

  SPEC_DEV int nblocks() const { return w.blk1 - w.blk0; }
  // A merged output value (offset `at` in out [M][nq*HD]), and the same as
  // the hi + lo activation planes of the projection that follows.
  SPEC_DEV void put_out(size_t at, float v) const {
    a.out[at] = v;
    if (!a.planes) return;
    const size_t lo = at + (size_t)a.planes_mp * a.nq * HD;
    if (a.planes_f16) {
      const __half h = __float2half_rn(v), l = __float2half_rn(v - __half2float(h));
      a.planes[at] = __half_as_ushort(h);
      a.planes[lo] = __half_as_ushort(l);
    } else {
      const __nv_bfloat16 h = __float2bfloat16_rn(v), l = __float2bfloat16_rn(v - __bfloat162float(h));
      a.planes[at] = __bfloat16_as_ushort(h);
      a.planes[lo] = __bfloat16_as_ushort(l);
    }
  }
  SPEC_DEV int page_id(int pidx) const {
    const int local = pidx - 2 * w.blk0;
    if (local >= 0 && local < PGS_CACHE) return pgs[local];
    const int pg = a.block_table[(size_t)slot * a.max_pages + pidx];
    if (pg >= 0 && pg < a.n_pages) return pg;
    set_error(a.err, SPEC_ERR_CAPACITY);
    return 0;
  }
  // first pool row of (page, plane) for this KV head
  SPEC_DEV int row_of(int page, int plane) const { return ((page * 2 + plane) * a.nkv + w.kvh) * PAGE; }

  // ---- warp 0, one thread ----
  SPEC_DEV void load_tile(unsigned char* dst, int blk, int plane, uint64_t* bar, bool hint, uint64_t pol) {
    const int p0 = 2 * blk, p1 = min(2 * blk + 1, w.npages - 1);  // a missing second page repeats the first
    const int r0 = row_of(page_id(p0), plane), r1 = row_of(page_id(p1), plane);
    mbar_expect_tx(bar, TILE_BYTES);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (hint) {
        tma_2d_hint(dst + h * HALF_BYTES, tm, 64 * h, r0, bar, pol);
        tma_2d_hint(dst + h * HALF_BYTES + BOX_BYTES, tm, 64 * h, r1, bar, pol);
      } else {
        tma_2d(dst + h * HALF_BYTES, tm, 64 * h, r0, bar);
        tma_2d(dst + h * HALF_BYTES + BOX_BYTES, tm, 64 * h, r1, bar);
      }
    }
  }
  // Before the dependency wait: the first ring slots for blocks whose keys are
  // all committed positions (below seq_len), which the previous kernels of
  // this pass do not write. The drafter's keys are all committed.
  SPEC_DEV void preissue() {
    const int nb = nblocks();
    const bool hint = a.key_extra != 0;
    const uint64_t pol = l2_evict_first();
    auto safe = [&](int n) { return a.key_extra == 0 || BK * (w.blk0 + n + 1) <= L0; };
    kpre = 0;
    vpre = 0;
    while (kpre < min(KSLOTS, nb) && safe(kpre)) {
      load_tile(sm + S::K_OFF + (size_t)kpre * TILE_BYTES, w.blk0 + kpre, 0, &kfull[kpre], hint, pol);
      ++kpre;
    }
    while (vpre < min(VSLOTS, nb) && safe(vpre)) {
      load_tile(sm + S::V_OFF + (size_t)vpre * TILE_BYTES, w.blk0 + vpre, 1, &vfull[vpre], hint, pol);
      ++vpre;
    }
  }
  SPEC_DEV void producer() {
    const int nb = nblocks();
    const bool hint = a.key_extra != 0;  // the target's rows (not the drafter's)
    const uint64_t pol = l2_evict_first();
    int kn = kpre, vn = vpre;
    for (int n = 0; n <= nb; ++n) {
      if (n < nb && n >= kpre) {
        const int s = n % KSLOTS;
        if (n >= KSLOTS && !wait_phase(&kempty[s], ((n / KSLOTS) - 1) & 1, abort_s, a.err)) break;
        load_tile(sm + S::K_OFF + (size_t)s * TILE_BYTES, w.blk0 + n, 0, &kfull[s], hint, pol);
        kn = n + 1;
      }
      if (n >= 1 && n - 1 >= vpre) {
        const int m = n - 1, s = m % VSLOTS;
        if (m >= VSLOTS && !wait_phase(&vempty[s], ((m / VSLOTS) - 1) & 1, abort_s, a.err)) break;
        load_tile(sm + S::V_OFF + (size_t)s * TILE_BYTES, w.blk0 + m, 1, &vfull[s], hint, pol);
        vn = m + 1;
      }
    }
    // every copy issued here lands before the CTA's shared memory is released
    // (in a normal run they were all consumed already)
    for (int n = max(0, kn - KSLOTS); n < kn; ++n) drain_phase(&kfull[n % KSLOTS], (n / KSLOTS) & 1);
    for (int n = max(0, vn - VSLOTS); n < vn; ++n) drain_phase(&vfull[n % VSLOTS], (n / VSLOTS) & 1);
  }

  // ---- warp 1, one thread ----
  // S^T(j) = K_j . [Q_hi; Q_lo]^T into tensor-memory buffer j & 1
  SPEC_DEV bool issue_s(int j) {
    const int s = j % KSLOTS;
    if (!wait_phase(&kfull[s], (j / KSLOTS) & 1, abort_s, a.err)) return false;
    fence_after();
    const uint32_t kb = sa(sm + S::K_OFF + (size_t)s * TILE_BYTES), qb = sa(sm + S::Q_OFF);
    const uint32_t d = tmem + (uint32_t)((j & 1) * 64);
    const uint32_t id = idesc(BK, 64, false, false);
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const uint32_t h = ks >> 2, off = 32 * (ks & 3);
      mma(d, desc_k(kb + h * HALF_BYTES + off), desc_k(qb + h * S::QP_HALF + off), id, ks > 0 ? 1u : 0u);
    }
    commit(&kempty[s]);
    commit(&sfull[j & 1]);
    return true;
  }
  // O^T += V_j^T . P_j: both operands MN-major (V stored [key][dim], P [key][query])
  SPEC_DEV void mma_loop() {
    const int nb = nblocks();
    bool ok = nb == 0 || issue_s(0);
    for (int j = 0; ok && j < nb; ++j) {
      if (j + 1 < nb && !issue_s(j + 1)) break;
      const int s = j % VSLOTS;
      if (!wait_phase(&pfull[j & 1], (j >> 1) & 1, abort_s, a.err) ||
          !wait_phase(&vfull[s], (j / VSLOTS) & 1, abort_s, a.err))
        break;
      fence_after();
      const uint32_t vb = sa(sm + S::V_OFF + (size_t)s * TILE_BYTES);
      const uint32_t pb = sa(sm + S::P_OFF + (size_t)(j & 1) * S::P_BYTES);
      const uint32_t id = idesc(HD, 64, true, true);
#pragma unroll
      for (int ks = 0; ks < BK / 16; ++ks)  // 16 keys = two 8-key groups (2048 B) per step
        mma(tmem + 128u, desc_mn(vb + 2048u * ks, HALF_BYTES), desc_mn(pb + 2048u * ks, S::P_BYTES), id,
            (j > 0 || ks > 0) ? 1u : 0u);
      commit(&vempty[s]);
      commit(&pvdone[j & 1]);
    }
    // every MMA of this CTA complete before its tensor memory is freed
    commit(drain);
    drain_phase(drain, 0);
  }

  // ---- warps 2-9 (thread = TMEM lane: a key of the block, or a dimension) ----
  // Two groups of 4 warps, one warp per TMEM lane quarter each: group g takes
  // the query columns [g*QG, (g+1)*QG). Waits never make these warps diverge:
  // a wait that gives up sets the abort flag, later waits return at once, and
  // the warps run on (results are then not used), so every named barrier is
  // passed by all of them.
  static constexpr int QG = QNP / 2;
  SPEC_DEV int lane_base() const { return ((threadIdx.x >> 5) & 3) * 32; }
  SPEC_DEV int key_lane() const { return lane_base() + (threadIdx.x & 31); }
  SPEC_DEV int group() const { return (threadIdx.x - SM0) >> 7; }

  // query planes: row q (< QN) = rotated query i*G + g as bf16 hi, row 32 + q
  // its lo part; the other rows zero
  SPEC_DEV void build_q() {
    const int t = threadIdx.x - SM0;
    const int b = w.b;
    if (t < p.QN) {
      const int i = t / p.G, gg = t - i * p.G;
      coff[t] = (b * a.R + i) * a.nq * HD + (w.kvh * p.G + gg) * HD;
    }
    for (int u = t; u < 32 * 8; u += NSM) {
      const int q = u >> 3, c8 = u & 7;  // dims 8*c8 .. +7 and 64 + 8*c8 .. +7
      float x0[8], x1[8];
      if (q < p.QN) {
        const int i = q / p.G, g = q - i * p.G;
        const float* src = a.q + (size_t)(b * a.R + i) * a.ldq + (w.kvh * p.G + g) * HD;
        const float4 u0 = __ldcg(reinterpret_cast<const float4*>(src + 8 * c8));
        const float4 u1 = __ldcg(reinterpret_cast<const float4*>(src + 8 * c8 + 4));
        const float4 v0 = __ldcg(reinterpret_cast<const float4*>(src + 64 + 8 * c8));
        const float4 v1 = __ldcg(reinterpret_cast<const float4*>(src + 64 + 8 * c8 + 4));
        const float a0[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float a1[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        if (a.rope_cs) {
          const float* cs = a.rope_cs + (size_t)(b * a.R + i) * HD + 16 * c8;  // (cos, sin) of pair 8*c8 + e
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float co = __ldcg(cs + 2 * e), si = __ldcg(cs + 2 * e + 1);
            x0[e] = a0[e] * co - a1[e] * si;
            x1[e] = a1[e] * co + a0[e] * si;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x0[e] = a0[e];
            x1[e] = a1[e];
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x0[e] = x1[e] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float* x = h ? x1 : x0;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_pair(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
        unsigned char* base = sm + S::Q_OFF + h * S::QP_HALF;
        *reinterpret_cast<uint4*>(base + swz(q, 16 * c8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(base + swz(32 + q, 16 * c8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }

  // x = hi + lo with hi, lo bf16, for a pair (packed low element first)
  static SPEC_DEV void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(hh);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&hh);
    lo = *reinterpret_cast<const uint32_t*>(&ll);
  }

  SPEC_DEV bool poll(uint64_t* b, unsigned parity) { return wait_phase(b, parity, abort_s, a.err); }

  // Column reduction of this group's QG columns over all 128 keys of the
  // block: the 4 warps' results -> red, then thread c < QNP combines column c.
  template <bool MAX>
  SPEC_DEV float group_combine(float (&v)[QG], int c) {
    const int t = threadIdx.x - SM0, lane = t & 31, wi = (t >> 5) & 3, g = group();
    const float r = col_reduce<QG, MAX>(v);
    if (lane < QG) red[(g * 4 + wi) * 32 + lane] = r;
    sm_sync();
    float out = 0.f;
    if (c < QNP) {
      const int gc = c / QG, lc = c - gc * QG;
      const float* rr = red + gc * 128 + lc;
      out = MAX ? fmaxf(fmaxf(rr[0], rr[32]), fmaxf(rr[64], rr[96])) : (rr[0] + rr[32]) + (rr[64] + rr[96]);
    }
    return out;
  }

  SPEC_DEV void softmax_loop(float (&lsum)[QG]) {
    const int t = threadIdx.x - SM0, kl = key_lane(), g = group();
    const int c0 = g * QG;  // this thread's first query column
    const uint32_t lanes = (uint32_t)lane_base() << 16;
    const int nb = nblocks();
    if (t < 32) mu[t] = -INFINITY;
    float mreg[QG];
    int lim[QG];
    unsigned int tmk[QG];
#pragma unroll
    for (int q = 0; q < QG; ++q) {
      lsum[q] = 0.f;
      mreg[q] = -INFINITY;
      lim[q] = c0 + q < p.QN ? L0 + (c0 + q) / p.G + a.key_extra : 0;
      tmk[q] = a.tree_mask && c0 + q < p.QN ? a.tree_mask[w.b * a.R + (c0 + q) / p.G] : ~0u;
    }
    const int key_end = L0 + p.R - 1 + a.key_extra;
    for (int j = 0; j < nb; ++j) {
      poll(&sfull[j & 1], (j >> 1) & 1);
      fence_after();
      float s[QG], lo[QG];
      const uint32_t sb = tmem + lanes + (uint32_t)((j & 1) * 64 + c0);
      ldn<QG>(sb, s);
      ldn<QG>(sb + 32, lo);
      wait_ld();
      const int key = (w.blk0 + j) * BK + kl;
      bool over = false;
#pragma unroll
      for (int q = 0; q < QG; ++q) {
        s[q] = key < lim[q] && tree_visible(tmk[q], L0, key) ? (s[q] + lo[q]) * p.scale2 : -INFINITY;
        over |= s[q] > mreg[q] + TAU;
      }
      // the running maximum moves (rarely: the first block, or a score 2^8
      // above it): column maxima, new maxima, and O^T and the sums rescaled
      if (sm_any(over)) {
        float v[QG];
#pragma unroll
        for (int q = 0; q < QG; ++q) v[q] = s[q];
        const float bm = group_combine<true>(v, t);
        if (t < QNP) {
          const float m = mu[t];
          float f = 1.f;
          if (bm > m + TAU || (m == -INFINITY && bm > -INFINITY)) {
            f = m == -INFINITY ? 0.f : ex2(m - bm);
            mu[t] = bm;
          }
          alpha[t] = f;
        }
        sm_sync();
        float al[QG];
        bool any_o = false;
#pragma unroll
        for (int q = 0; q < QG; ++q) {
          al[q] = alpha[c0 + q];
          mreg[q] = mu[c0 + q];
          lsum[q] *= al[q];
          any_o |= al[q] != 1.f;
        }
        if (j > 0 && sm_any(any_o)) {
          // after PV(j-1): this thread's dimension row of O^T, its group's hi
          // and lo columns
          poll(&pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1);
          fence_after();
          const uint32_t ob = tmem + lanes + 128u + (uint32_t)c0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float o[QG];
            ldn<QG>(ob + 32 * h, o);
            wait_ld();
#pragma unroll
            for (int e = 0; e < QG; ++e) o[e] *= al[e];
            stn<QG>(ob + 32 * h, o);
          }
          wait_st();
        }
      }
      // probabilities of this key -> row `kl` of P tile j & 1 (hi columns
      // 0-31, lo columns 32-63), once PV(j-2) has read that tile
      if (j >= 2) poll(&pvdone[j & 1], ((j - 2) >> 1) & 1);
      uint32_t hi[QG / 2], lw[QG / 2];
#pragma unroll
      for (int q = 0; q < QG; q += 2) {
        const float p0 = s[q] == -INFINITY ? 0.f : ex2(s[q] - mreg[q]);
        const float p1 = s[q + 1] == -INFINITY ? 0.f : ex2(s[q + 1] - mreg[q + 1]);
        lsum[q] += p0;
        lsum[q + 1] += p1;
        split_pair(p0, p1, hi[q / 2], lw[q / 2]);
      }
      unsigned char* prow = sm + S::P_OFF + (size_t)(j & 1) * S::P_BYTES;
      if constexpr (QG >= 8) {
#pragma unroll
        for (int c = 0; c < QG / 8; ++c) {
          *reinterpret_cast<uint4*>(prow + swz(kl, 2 * c0 + 16 * c)) =
              make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
          *reinterpret_cast<uint4*>(prow + swz(kl, 64 + 2 * c0 + 16 * c)) =
              make_uint4(lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
        }
      } else {
        *reinterpret_cast<uint2*>(prow + swz(kl, 2 * c0)) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2*>(prow + swz(kl, 64 + 2 * c0)) = make_uint2(lw[0], lw[1]);
      }
      // keys past the last row's limit hold whatever the cache has there
      // (zero, stale or uncommitted rows); their probabilities are exact
      // zeros, and their values are zeroed too, so that nothing non-finite
      // there can reach O^T through 0 x value
      if ((w.blk0 + j + 1) * BK > key_end) {
        poll(&vfull[j % VSLOTS], (j / VSLOTS) & 1);
        if (key >= key_end) {
          unsigned char* vr = sm + S::V_OFF + (size_t)(j % VSLOTS) * TILE_BYTES + (size_t)kl * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vr + g * HALF_BYTES + 16 * c) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_before();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&pfull[j & 1]);
    }
  }

  // After the last block: reduce the sums, read O^T, write the final rows or
  // this split's partials.
  SPEC_DEV void finish(float (&lsum)[QG]) {
    const int t = threadIdx.x - SM0, d = key_lane(), g = group(), c0 = g * QG;
    const int nb = nblocks();
    if (nb > 0) poll(&pvdone[(nb - 1) & 1], ((nb - 1) >> 1) & 1);
    fence_after();
    const float l = group_combine<false>(lsum, t);
    if (t < QNP) lfin[t] = l;
    sm_sync();
    float o[QG];
    if (nb > 0) {
      float hi[QG], lo[QG];
      const uint32_t ob = tmem + ((uint32_t)lane_base() << 16) + 128u + (uint32_t)c0;
      ldn<QG>(ob, hi);
      ldn<QG>(ob + 32, lo);
      wait_ld();
#pragma unroll
      for (int q = 0; q < QG; ++q) o[q] = hi[q] + lo[q];
    } else {
#pragma unroll
      for (int q = 0; q < QG; ++q) o[q] = 0.f;
    }
    const int nv = min(QG, p.QN - c0);  // this group's columns that are queries
    if (w.np == 1) {
#pragma unroll
      for (int q = 0; q < QG; ++q)
        if (q < nv) {
          const float lc = lfin[c0 + q];
          put_out((size_t)coff[c0 + q] + d, lc > 0.f ? o[q] / lc : 0.f);
        }
    } else {
      // partials CTA-major: rows blockIdx.x * 32 + column
      float* po = a.part_o + ((size_t)blockIdx.x * 32 + c0) * HD + d;
#pragma unroll
      for (int q = 0; q < QG; ++q)
        if (q < nv) __stcg(po + q * HD, o[q]);
      if (d < nv)
        __stcg(reinterpret_cast<float2*>(a.part_ml) + (size_t)blockIdx.x * 32 + c0 + d,
               make_float2(mu[c0 + d], lfin[c0 + d]));
    }
  }

  // The CTAs of a pair merge after all have written their partials: CTA j of
  // the pair takes query rows [QN*j/np, QN*(j+1)/np). The (max, sum) pairs of
  // those rows' splits are read in one parallel round and turned into
  // weights; then each half of the threads takes half of the rows, one
  // dimension per thread, with up to 8 partial loads in flight at a time.
  SPEC_DEV void merge(bool arrived_ok) {
    const int t = threadIdx.x - SM0, d = t & 127, half = t >> 7;
    unsigned int* arrive = cnt + (w.b * a.nkv + w.kvh);
    unsigned int* depart = arrive + p.npairs;
    float2* ml = reinterpret_cast<float2*>(sm + S::ML_OFF);
    if (t == 0) {
      __threadfence();
      int ok = 0;
      if (arrived_ok) {
        atomic_add_acq_rel(arrive, 1u);
        const unsigned target = (unsigned)(w.np + p.wait_extra);
        const unsigned long long t0 = globaltimer();
        for (;;) {
          if (ld_acquire(arrive) >= target) {
            ok = 1;
            break;
          }
          if (globaltimer() - t0 > MERGE_WAIT_NS) break;
          __nanosleep(100);
        }
        if (!ok) set_error(a.err, SPEC_ERR_TIMEOUT);
      }
      misc[0] = ok;
    }
    sm_sync();
    const int np = w.np, q0 = (p.QN * w.j) / np, q1 = (p.QN * (w.j + 1)) / np;
    const int rows = q1 - q0, n = rows * np;
    const bool go = misc[0] != 0 && n <= MERGE_MAX;
    if (misc[0] && n > MERGE_MAX && t == 0) set_error(a.err, SPEC_ERR_CAPACITY);
    const size_t first = (size_t)(blockIdx.x - w.j) * 32 + q0;  // row q0 of the pair's first CTA
    if (go)
      for (int k = t; k < n; k += NSM) {
        const int r = k / np, sp = k - r * np;
        ml[k] = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + first + (size_t)sp * 32 + r);
      }
    sm_sync();
    if (go && t < rows) {
      float M = -INFINITY, L = 0.f;
      for (int sp = 0; sp < np; ++sp) M = fmaxf(M, ml[t * np + sp].x);
      for (int sp = 0; sp < np; ++sp) {
        const float2 v = ml[t * np + sp];
        const float wt = v.x == -INFINITY ? 0.f : ex2(v.x - M);
        L += wt * v.y;
        ml[t * np + sp].x = wt;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int sp = 0; sp < np; ++sp) ml[t * np + sp].x *= inv;
    }
    sm_sync();
    if (go) {
      // thread = dimension d; the two halves of the threads take alternate
      // rows, two rows at a time; each row's splits are added in order, with
      // up to eight loads in flight
      constexpr size_t SP = 32 * HD;  // distance between two splits of a row
      for (int r = half; r < rows; r += 4) {
        const bool two = r + 2 < rows;
        const float* s0 = a.part_o + (first + r) * HD + d;
        const float* s1 = two ? s0 + 2 * HD : s0;
        const float2* w0 = ml + r * np;
        const float2* w1 = two ? w0 + 2 * np : w0;
        float acc0 = 0.f, acc1 = 0.f;
        int sp = 0;
        for (; sp + 4 <= np; sp += 4) {
          float u[4], v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            u[i] = __ldcg(s0 + (sp + i) * SP);
            v[i] = __ldcg(s1 + (sp + i) * SP);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc0 = fmaf(w0[sp + i].x, u[i], acc0);
            acc1 = fmaf(w1[sp + i].x, v[i], acc1);
          }
        }
        for (; sp < np; ++sp) {
          const float u = __ldcg(s0 + sp * SP), v = __ldcg(s1 + sp * SP);
          acc0 = fmaf(w0[sp].x, u, acc0);
          acc1 = fmaf(w1[sp].x, v, acc1);
        }
        put_out((size_t)coff[q0 + r] + d, acc0);
        if (two) put_out((size_t)coff[q0 + r + 2] + d, acc1);
      }
    }
    sm_sync();
    if (t == 0) {
      // the last CTA of the pair to leave resets both counters
      if (atomic_add_acq_rel(depart, 1u) == (unsigned)np - 1) {
        *arrive = 0u;
        *depart = 0u;
        __threadfence();
      }
    }
  }
};

// Device-side plan: which pair, which of its CTAs and which blocks this CTA
// takes. Pairs get CTAs in proportion to their blocks (at least one each).
SPEC_DEV bool plan_work(const AttnArgs& a, const Plan& p, int* s_nb, int* misc, Work& w) {
  const int tid = threadIdx.x;
  __shared__ int s_tot;
  __shared__ int s_pair, s_j, s_np, s_nbp;
  if (p.grid <= p.npairs) {
    // one CTA per pair: no split, no merge
    const int pr = blockIdx.x;
    w.b = pr / a.nkv;
    w.kvh = pr % a.nkv;
    w.j = 0;
    w.np = 1;
    const int L = a.seq_len[a.seq_ids[w.b]];
    const int keys = L + a.R - 1 + a.key_extra;
    int pages = keys > 0 ? (keys + PAGE - 1) / PAGE : 0;
    if (pages > a.max_pages) {
      if (tid == 0) set_error(a.err, SPEC_ERR_CAPACITY);
      pages = a.max_pages;
    }
    w.npages = pages;
    w.blk0 = 0;
    w.blk1 = (pages + 1) / 2;
    __syncthreads();
    return pr < p.npairs;
  }
  if (tid == 0) {
    s_tot = 0;
    s_pair = -1;
  }
  __syncthreads();
  for (int pr = tid; pr < p.npairs; pr += blockDim.x) {
    const int b = pr / a.nkv;
    const int L = a.seq_len[a.seq_ids[b]];
    const int keys = L + a.R - 1 + a.key_extra;
    int pages = keys > 0 ? (keys + PAGE - 1) / PAGE : 0;
    if (pages > a.max_pages) {
      set_error(a.err, SPEC_ERR_CAPACITY);
      pages = a.max_pages;
    }
    s_nb[pr] = (pages + 1) / 2;
    atomicAdd(&s_tot, s_nb[pr]);
  }
  __syncthreads();
  if (tid < 32) {
    // warp 0: each pair's CTA count, and an exclusive prefix sum over the
    // pairs (32 at a time) that places this CTA
    const int extra = p.grid - p.npairs, tot = s_tot;
    int run = 0;
    for (int base = 0; base < p.npairs; base += 32) {
      const int pr = base + tid;
      int nb = 0, np = 0;
      if (pr < p.npairs) {
        nb = s_nb[pr];
        np = 1;
        if (extra > 0 && tot > 0) np += (int)(((long long)extra * nb) / tot);
        np = min(np, max(nb, 1));
      }
      int incl = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += v;
      }
      const int c0 = run + incl - np;
      if (np > 0 && (int)blockIdx.x >= c0 && (int)blockIdx.x < c0 + np) {
        s_pair = pr;
        s_j = (int)blockIdx.x - c0;
        s_np = np;
        s_nbp = nb;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  if (s_pair < 0) return false;
  w.b = s_pair / a.nkv;
  w.kvh = s_pair % a.nkv;
  w.j = s_j;
  w.np = s_np;
  const int nb = s_nbp;
  w.blk0 = (int)(((long long)nb * w.j) / w.np);
  w.blk1 = (int)(((long long)nb * (w.j + 1)) / w.np);
  const int L = a.seq_len[a.seq_ids[w.b]];
  const int keys = L + a.R - 1 + a.key_extra;
  w.npages = min(keys > 0 ? (keys + PAGE - 1) / PAGE : 0, a.max_pages);
  (void)misc;
  return true;
}

template <int QNP>
__global__ void __launch_bounds__(NTHR, 1)
    attn_flash_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ Plan p,
                      const __grid_constant__ CUtensorMap tm, unsigned int* cnt) {
  using S = Smem;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_nb[MAX_PAIRS];
  const uint32_t mis = sa(smem_raw) & 1023u;
  unsigned char* sm = smem_raw + (mis ? 1024 - mis : 0);
  Cta<QNP> k{a, p, &tm, cnt, sm};
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::BAR_OFF);
  k.kfull = bars;
  k.kempty = bars + KSLOTS;
  k.vfull = bars + 2 * KSLOTS;
  k.vempty = k.vfull + VSLOTS;
  k.sfull = k.vempty + VSLOTS;
  k.pfull = k.sfull + 2;
  k.pvdone = k.pfull + 2;
  k.drain = k.pvdone + 2;
  k.red = reinterpret_cast<float*>(sm + S::RED_OFF);
  k.mu = reinterpret_cast<float*>(sm + S::MU_OFF);
  k.alpha = reinterpret_cast<float*>(sm + S::AL_OFF);
  k.lfin = reinterpret_cast<float*>(sm + S::L_OFF);
  k.coff = reinterpret_cast<int*>(sm + S::COFF_OFF);
  k.pgs = reinterpret_cast<int*>(sm + S::PG_OFF);
  k.misc = reinterpret_cast<int*>(sm + S::MISC_OFF);
  k.abort_s = reinterpret_cast<volatile int*>(k.misc + 3);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KSLOTS; ++s) {
      mbar_init(&k.kfull[s], 1);
      mbar_init(&k.kempty[s], 1);
    }
    for (int s = 0; s < VSLOTS; ++s) {
      mbar_init(&k.vfull[s], 1);
      mbar_init(&k.vempty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k.sfull[i], 1);
      mbar_init(&k.pfull[i], NSM);
      mbar_init(&k.pvdone[i], 1);
    }
    mbar_init(k.drain, 1);
    k.misc[0] = k.misc[1] = 0;
    *k.abort_s = 0;
    mbar_init_fence();
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     sa(reinterpret_cast<uint32_t*>(k.misc + 2))),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // The lengths, sequence ids and page tables are not written by the kernels
  // of a pass (the previous pass's commit wrote the lengths, and every earlier
  // kernel had completed before the one just before this launched it), so the
  // plan, the page ids and the first committed blocks come before the wait;
  // the queries and the pass's new keys and values come after it.
  const bool have = plan_work(a, p, s_nb, k.misc, k.w);  // contains __syncthreads
  fence_before();
  __syncthreads();
  fence_after();
  k.tmem = *reinterpret_cast<uint32_t*>(k.misc + 2);
  k.kpre = k.vpre = 0;
  if (have) {
    k.slot = a.seq_ids[k.w.b];
    k.L0 = a.seq_len[k.slot];
    // this range's page ids (checked: a bad id is skipped -- page 0 read instead -- and recorded)
    const int pa = 2 * k.w.blk0, pe = min(2 * k.w.blk1, k.w.npages);
    for (int pi = pa + (int)threadIdx.x; pi < pe && pi - pa < PGS_CACHE; pi += NTHR) {
      int pg = a.block_table[(size_t)k.slot * a.max_pages + pi];
      if (pg < 0 || pg >= a.n_pages) {
        set_error(a.err, SPEC_ERR_CAPACITY);
        pg = 0;
      }
      k.pgs[pi - pa] = pg;
    }
  }
  __syncthreads();
  if (have && threadIdx.x == 0) k.preissue();
  grid_dep_wait();
  if (have && warp >= 2) k.build_q();
  fence_before();
  __syncthreads();
  fence_after();
  // every CTA of this grid is resident past this point: the next kernel may be
  // scheduled (it waits for this grid's completion before reading its output)
  grid_dep_launch();

  if (have) {
    if (warp == 0) {
      if (lane == 0) k.producer();
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) k.mma_loop();
      __syncwarp();
    } else {
      float lsum[QNP / 2];
      k.softmax_loop(lsum);
      k.finish(lsum);
    }
  }
  fence_before();
  __syncthreads();
  const bool aborted = *k.abort_s != 0;
  // tensor memory is released once every MMA issued here has completed: the
  // softmax warps waited for the last PV commit (which covers every earlier
  // MMA) unless they gave up, in which case the MMA thread stopped issuing
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(k.tmem), "r"(TMEM_COLS) : "memory");
  }
  if (have && k.w.np > 1 && warp >= 2) k.merge(!aborted);
}

template <int QNP>
void set_attr() {
  cudaFuncSetAttribute(attn_flash_kernel<QNP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)Smem::ALLOC);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void init_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
}

// One layer of the pool as a 2-D bf16 tensor [rows][128] (rows = pages x 2
// planes x KV heads x 64 positions); boxes of 64 rows x 64 dims in the
// 128-byte swizzle layout.
bool encode_pool(CUtensorMap* m, const void* base, long long rows) {
  if (!g_encode || ((uintptr_t)base & 15) || rows <= 0 || rows > 0x7fffffffLL) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)HD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)HD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)PAGE};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fa

void setup_attn_flash_attributes() {
  fa::set_attr<8>();
  fa::set_attr<16>();
  fa::set_attr<32>();
}

bool attention_flash_ok(const AttnArgs& a) {
  const int G = a.nq / a.nkv, QN = a.R * G;
  return a.kv_dtype == DT_BF16 && a.hd == fa::HD && QN >= 1 && QN <= 32 && a.B * a.nkv <= fa::MAX_PAIRS &&
         (a.key_extra == 0 || a.key_extra == 1);
}

// counters: 2 x B x nkv words (arrivals, departures), zero between launches.
int attention_flash(const AttnArgs& a, unsigned int* counters, int wait_extra, cudaStream_t st) {
  using namespace fa;
  if (!attention_flash_ok(a)) return -2;
  std::call_once(g_once, init_encode);
  Plan p;
  p.npairs = a.B * a.nkv;
  // At least two blocks a CTA for the target's rows (fewer CTAs to merge on
  // short contexts: E2B b1 verify 1.58 -> 1.44 ms); one for the drafter's
  // single row, whose merges are cheap (two a CTA measured slower there).
  const int min_blocks = a.key_extra != 0 ? 2 : 1;
  p.grid = std::max(p.npairs, std::min(num_sms(), p.npairs * std::max(1, (a.max_pages + 1) / 2 / min_blocks)));
  // split CTAs write their partials CTA-major (32 rows each)
  if (p.grid > p.npairs && (size_t)p.grid * 32 > (size_t)ATTN_FLASH_PART_ROWS) return -2;
  p.R = a.R;
  p.G = a.nq / a.nkv;
  p.QN = a.R * p.G;
  p.scale2 = 1.4426950408889634f / sqrtf((float)HD);
  p.wait_extra = wait_extra;
  CUtensorMap tm;
  const __nv_bfloat16* base = (const __nv_bfloat16*)a.pool + (size_t)a.layer * a.layer_elems;
  if (!encode_pool(&tm, base, a.layer_elems / HD)) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(NTHR);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.standalone ? 0 : 1;
  cudaError_t e;
  if (p.QN <= 8) {
    cfg.dynamicSmemBytes = Smem::ALLOC;
    e = cudaLaunchKernelEx(&cfg, attn_flash_kernel<8>, a, p, tm, counters);
  } else if (p.QN <= 16) {
    cfg.dynamicSmemBytes = Smem::ALLOC;
    e = cudaLaunchKernelEx(&cfg, attn_flash_kernel<16>, a, p, tm, counters);
  } else {
    cfg.dynamicSmemBytes = Smem::ALLOC;
    e = cudaLaunchKernelEx(&cfg, attn_flash_kernel<32>, a, p, tm, counters);
  }
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace spec
