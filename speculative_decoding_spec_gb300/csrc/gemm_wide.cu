// gemm_wide.cu -- weight-streaming projection for 9..64 activation rows on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory,
// operands staged by TMA).
//
// Verification runs the k+1 positions of every sequence in one pass, so each
// weight is read once for all B*(k+1) rows ("Gemma 4's MTP drafter explained"
// (molayo1419.me), section "Why is generating one token at a time slow?"). With
// batch 4-8 and k = 4 that is 20-40 rows: too many for register-fragment MMAs
// to keep up with HBM, while a 128-row weight tile times a 16-64-row activation
// tile is a natural tcgen05 shape (M = 128 weight rows, N = rows padded to 16).
//
// Data flow per CTA (one CTA per SM: 6 warps, 10 with Q4_0 weights):
//  - warp 0 (one thread): TMA producer. A ring of stages, each one 128 x 64
//    bf16 weight tile and the matching 64 columns of the activation hi and lo
//    planes, both in the 128-byte-swizzled K-major layout the MMA reads.
//    Weights do not depend on earlier kernels, so the first stages' weight
//    loads are issued before the programmatic-launch wait.
//  - warp 1: owns the tensor memory; one thread issues, per stage, one MMA per
//    16-column k-step with N = 2 x rows (the hi and lo planes are consecutive
//    rows of the B operand, so each k-step is one instruction) and commits the
//    stage back to the producer and, at the end of a tile, the accumulator to
//    the epilogue. Even and odd k-steps go to two independent accumulator
//    chains: with a few dozen activation rows an MMA is short, and
//    back-to-back MMAs into one accumulator would wait on each other. Two
//    such accumulator sets alternate between tiles, so the epilogue of one
//    tile overlaps the MMAs of the next.
//  - warps 2-5: epilogue. tcgen05.ld gives thread r the tile's weight row r for
//    every activation row (the sum of the two chains' hi and lo columns);
//    they apply the RMSNorm factor and the operation's
//    epilogue (store, residual add, gated GELU, RoPE + KV append, argmax +
//    accept), which are the ones of the register-fragment kernel.
//
// The activations enter as bf16 hi + lo planes (x = hi + lo to 2^-17), written
// once per launch by a small preparation kernel that also applies the RMSNorm
// gain and computes each row's 1/rms; so a result equals an fp32-activation dot
// product of the bf16 weights, as in the register-fragment kernel. Q4_0
// weights: four more warps expand each stage's codes and block scales into
// fp16 hi + lo weight planes (exact), and the activation planes are fp16.
//
// Work split: units are (tile, 64-column chunk) pairs in tile-major order and
// CTA b owns the balanced range [U*b/G, U*(b+1)/G). A tile cut between CTAs is
// summed by the last CTA to arrive (arrival counter per tile), in CTA order, so
// results do not depend on timing. Matrices with few tiles run instead as one
// thread-block cluster of S CTAs per tile: each CTA streams a K-range and keeps
// its partial in shared memory; after a cluster barrier each CTA sums a slice
// of the activation rows over the cluster's CTAs in rank order (distributed
// shared memory) and finishes those rows.
//
// Inside a target pass two more arrangements remove work from a launch's
// tail. A residual-add launch whose next projection prepares its own planes
// may leave its cut tiles to that preparation (wide.defer): the CTAs only
// publish their partials, and the preparation adds them, in CTA order, into
// the residual rows before it normalises them. And a gated-GELU launch may
// write the next projection's activation planes itself (wide.out_xs), which
// then has no preparation (wide.ready).
//
// Every wait is bounded: on a timeout the CTA records SPEC_ERR_TIMEOUT, stops,
// drains its own copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "common.cuh"
#include "mbar.cuh"
#include "tail.cuh"

namespace spec {
namespace wide {

constexpr int TM = 128;              // weight rows per tile (MMA M)
constexpr int KC = 64;               // K columns per stage (one 128-byte swizzle row of bf16)
constexpr int NTHR = 192;            // 6 warps (bf16 weights)
constexpr int NTHR_Q4 = 320;         // + 4 dequantising warps (Q4_0 weights)
constexpr int EPI0 = 64;             // first epilogue thread
constexpr int DQ0 = 192;             // first dequantising thread (Q4_0)
constexpr int CODE_BYTES = TM * KC / 2;  // 4 KB of Q4_0 codes per stage
constexpr int W_BYTES = TM * KC * 2; // 16 KB weight tile per stage
constexpr int XCH_LD = TM + 1;       // exchange buffer row stride (floats): conflict-free both ways
constexpr int MAX_STAGES = 8;
// The preparation splits every row into blocks of PREP_COLS columns; with an
// RMSNorm each block leaves its sum of squares in rms[row][block] (at most
// RMS_PARTS blocks) and the projection adds them in block order.
constexpr int PREP_COLS = 1024, RMS_PARTS = 16;
constexpr int NBARS = 3 * MAX_STAGES + 6;  // full, empty, weights-ready, 2 acc-full, 2 acc-empty, drain, pad
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr unsigned SPIN_LIMIT = 1u << 26;
constexpr int TMEM_COLS = 512;       // 2 accumulator sets x 2 chains x (hi, lo) x up to 64 columns
constexpr int SET_COLS = 256;        // columns of one accumulator set
constexpr int CHAIN_COLS = 128;      // columns of one chain (hi columns, then lo columns)

enum { MAP_PLAIN = 0, MAP_PAIR = 1, MAP_ROPE = 2 };

struct Plan {
  int T, C, U, grid;
  int MP;        // activation rows padded to a multiple of 16 (MMA N)
  int map;
  int stages;
  int stage_bytes;
  int x_off;     // activation planes within a stage
  int c_off;     // Q4_0 codes within a stage (after the two dequantised weight planes)
  int tx_bytes;  // bytes the TMA loads of one stage bring
  int q4;        // Q4_0 weights, dequantised in shared memory
  int S;         // CTAs per tile in a thread-block cluster (1: balanced unit ranges, global fixups)
  int smem;      // dynamic shared memory requested (includes 1 KB alignment slack)
};

// ---- tcgen05 / TMA primitives ----------------------------------------------

SPEC_DEV void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SPEC_DEV void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8-row groups of 1024 bytes, stride-dimension offset 1024 bytes);
// bits 46-48 hold the fixed value 0b001, bits 61-63 the swizzle mode (2).
SPEC_DEV uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with fp16 A and B (type fields 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

SPEC_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
SPEC_DEV void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(bar))
               : "memory");
}

// 2-D tiled TMA load of box (x, y) -> shared memory, completion on `bar`.
SPEC_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          sa(dst)),
      "l"(map), "r"(x), "r"(y), "r"(sa(bar))
      : "memory");
}

// The same with an L2 cache policy (weights: evict first, so that the stream of
// bytes read once does not push out the lines that are read again -- the
// activation planes, the residual rows, the split-tile partials).
SPEC_DEV void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar, uint64_t policy) {
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

// 16 consecutive accumulator columns of this warp's 32 lanes (lane = tile row).
SPEC_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
SPEC_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Optional per-CTA timeline (globaltimer, ns): slot i of this CTA's 16.
SPEC_DEV void stamp(unsigned long long* tr, int i) {
  if (tr) tr[blockIdx.x * 16 + i] = globaltimer();
}

// Thread-block cluster: barrier over every thread of every CTA, this CTA's
// rank, and a load from the shared memory of CTA `rank` of the cluster.
SPEC_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
SPEC_DEV unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
SPEC_DEV float ld_peer(const float* p, unsigned rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(sa(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// Named barrier of the 4 epilogue warps.
SPEC_DEV void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded wait on an mbarrier phase; a timeout sets the abort flag and the
// error word, and every other wait then gives up too.
SPEC_DEV bool wait_phase(uint64_t* b, unsigned parity, volatile int* abort_s, int* err) {
  for (unsigned it = 0; it < SPIN_LIMIT; ++it) {
    if (mbar_test(b, parity)) return true;
    if (*abort_s) return false;
  }
  *abort_s = 1;
  set_error(err, SPEC_ERR_TIMEOUT);
  return false;
}
// The same without giving up on abort: used to drain this CTA's own copies
// and MMAs before it frees its shared and tensor memory.
SPEC_DEV void drain_phase(uint64_t* b, unsigned parity) {
  for (unsigned it = 0; it < SPIN_LIMIT; ++it)
    if (mbar_test(b, parity)) return;
}

// ---- plan ----------------------------------------------------------------

// First unit of CTA b. Cluster mode (S > 1): cluster t = b / S takes tile t,
// its CTA j the chunks [C*j/S, C*(j+1)/S). Otherwise balanced ranges of the
// tile-major unit list.
__host__ __device__ inline int unit_begin(int b, const Plan& p) {
  if (p.S > 1) return (b / p.S) * p.C + (p.C * (b % p.S)) / p.S;
  return (int)(((long long)b * p.U) / p.grid);
}

// CTA whose unit range holds unit u.
__host__ __device__ inline int cta_of(int u, const Plan& p) {
  int b = (int)((((long long)u + 1) * p.grid - 1) / p.U);
  if (b >= p.grid) b = p.grid - 1;
  while (b > 0 && unit_begin(b, p) > u) --b;
  while (b + 1 < p.grid && unit_begin(b + 1, p) <= u) ++b;
  return b;
}

// Segments of a unit range: maximal runs of units of one tile.
struct SegIter {
  int u, u1, C;
  SPEC_DEV bool next(int& t, int& c0, int& c1) {
    if (u >= u1) return false;
    t = u / C;
    const int e = min(u1, (t + 1) * C);
    c0 = u - t * C;
    c1 = e - t * C;
    u = e;
    return true;
  }
};

// v as hi + lo halves (hi = v rounded, lo = the rest rounded), the split the
// preparation kernel makes, stored at xs[hi_at] and xs[lo_at].
SPEC_DEV void put_planes(uint16_t* xs, size_t hi_at, size_t lo_at, float v, int f16) {
  if (f16) {
    const __half h = __float2half_rn(v), l = __float2half_rn(v - __half2float(h));
    xs[hi_at] = __half_as_ushort(h);
    xs[lo_at] = __half_as_ushort(l);
  } else {
    const __nv_bfloat16 h = __float2bfloat16_rn(v), l = __float2bfloat16_rn(v - __bfloat162float(h));
    xs[hi_at] = __bfloat16_as_ushort(h);
    xs[lo_at] = __bfloat16_as_ushort(l);
  }
}

// ---- one CTA ----------------------------------------------------------------

template <int MP, bool Q4>
struct Cta {
  const GemvArgs& a;
  const Plan& p;
  const CUtensorMap* tmw;
  const CUtensorMap* tmx;
  const float* inv_rms;
  float* fix;
  unsigned int* cnt;
  int* err;
  unsigned long long* trace;
  unsigned char* stages;   // p.stages x p.stage_bytes, 1024-byte aligned
  float* xch;              // [MP][XCH_LD]
  uint64_t *full, *empty, *wready, *accf, *acce, *drain;
  float* rms_s;            // [64]
  float* rope_s;           // MAP_ROPE: [M][128] the rows' RoPE (cos, sin) pairs
  int *pos_s, *page_s;     // MAP_ROPE: [64] each row's position and cache page
  uint32_t* tmem_slot;
  volatile int* abort_s;
  int* bc;                 // [4] broadcast words of the epilogue warps
  uint32_t tmem;
  int u0, u1;

  SPEC_DEV unsigned char* stage(int s) const { return stages + (size_t)s * p.stage_bytes; }

  SPEC_DEV void load_w(int s, int u, uint64_t pol) const {
    const int t = u / p.C, x = (u - t * p.C) * KC;
    if (Q4) {
      // 128 rows x 32 code bytes (64 values); the planes are built from them
      unsigned char* dst = stage(s) + p.c_off;
      if (p.map == MAP_PAIR) {
        tma_load_2d_hint(dst, tmw, x / 2, t * 64, &full[s], pol);
        tma_load_2d_hint(dst + CODE_BYTES / 2, tmw, x / 2, a.geglu_half + t * 64, &full[s], pol);
      } else {
        tma_load_2d_hint(dst, tmw, x / 2, t * TM, &full[s], pol);
      }
      return;
    }
    unsigned char* dst = stage(s);
    if (p.map == MAP_PAIR) {
      // rows 0-63: gate rows 64t.., rows 64-127: the matching up rows
      tma_load_2d_hint(dst, tmw, x, t * 64, &full[s], pol);
      tma_load_2d_hint(dst + W_BYTES / 2, tmw, x, a.geglu_half + t * 64, &full[s], pol);
    } else {
      tma_load_2d_hint(dst, tmw, x, t * TM, &full[s], pol);
    }
  }
  SPEC_DEV void load_x(int s, int u) const {
    const int t = u / p.C, x = (u - t * p.C) * KC;
    tma_load_2d(stage(s) + p.x_off, tmx, x, 0, &full[s]);
  }

  // warp 0, one thread
  SPEC_DEV void producer() {
    const int nu = u1 - u0, pre = min(nu, p.stages);
    const uint64_t pol = l2_evict_first();
    for (int n = 0; n < pre; ++n) {
      mbar_expect_tx(&full[n], (unsigned)p.tx_bytes);
      load_w(n, u0 + n, pol);
    }
    grid_dep_wait();  // the activation planes come from the preparation kernel
    stamp(trace, 2);
    for (int n = 0; n < pre; ++n) load_x(n, u0 + n);
    int issued = pre;
    for (int n = pre; n < nu; ++n) {
      const int s = n % p.stages;
      if (!wait_phase(&empty[s], ((n / p.stages) - 1) & 1, abort_s, err)) break;
      mbar_expect_tx(&full[s], (unsigned)p.tx_bytes);
      load_w(s, u0 + n, pol);
      load_x(s, u0 + n);
      issued = n + 1;
    }
    if (*abort_s)  // let this CTA's copies land before its shared memory is released
      for (int n = max(0, issued - p.stages); n < issued; ++n) drain_phase(&full[n % p.stages], (n / p.stages) & 1);
  }

  // warp 1, one thread
  SPEC_DEV void mma_loop() {
    const uint32_t idesc = Q4 ? idesc_f16(TM, 2 * MP) : idesc_bf16(TM, 2 * MP);
    SegIter it{u0, u1, p.C};
    int t, c0, c1, n = 0, i = 0;
    bool ok = true;
    while (ok && it.next(t, c0, c1)) {
      const int acc = i & 1;
      if (i >= 2 && !wait_phase(&acce[acc], ((i >> 1) - 1) & 1, abort_s, err)) break;
      fence_after();
      const uint32_t d = tmem + (uint32_t)(acc * SET_COLS);
      for (int c = c0; c < c1; ++c, ++n) {
        const int s = n % p.stages;
        if (!wait_phase(&full[s], (n / p.stages) & 1, abort_s, err) ||
            (Q4 && !wait_phase(&wready[s], (n / p.stages) & 1, abort_s, err))) {
          ok = false;
          break;
        }
        if (n == 0) stamp(trace, 3);
        fence_after();
        const uint32_t w = sa(stage(s)), x = w + (uint32_t)p.x_off;
        if (Q4) {
          // hi weight plane into chain 0, lo plane into chain 1
#pragma unroll
          for (int ks = 0; ks < KC / 16; ++ks) {
            const uint64_t xd = sw128_desc(x + 32 * ks);
            const uint32_t acc = (c > c0 || ks > 0) ? 1u : 0u;
            mma_bf16(d, sw128_desc(w + 32 * ks), xd, idesc, acc);
            mma_bf16(d + (uint32_t)CHAIN_COLS, sw128_desc(w + W_BYTES + 32 * ks), xd, idesc, acc);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < KC / 16; ++ks)
            mma_bf16(d + (uint32_t)((ks & 1) * CHAIN_COLS), sw128_desc(w + 32 * ks), sw128_desc(x + 32 * ks), idesc,
                     (c > c0 || ks > 1) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      if (!ok) break;
      mma_commit(&accf[acc]);
      ++i;
    }
    stamp(trace, 4);
    // every MMA of this CTA complete before its tensor memory is freed
    mma_commit(drain);
    drain_phase(drain, 0);
  }

  // warps 6-9 (Q4_0): thread r turns row r of a stage's codes into two fp16
  // weight planes with packed half2 arithmetic: 0x6400 | code is the fp16
  // 1024 + code, so subtracting 1032 leaves code - 8 exactly; hi = (code - 8)
  // * scale rounded and lo = fma(code - 8, scale, -hi), the exact remainder
  // (an 11-bit scale times a 4-bit integer; exact for every normal fp16
  // scale). Rows are written in the 128-byte swizzle layout the MMA reads
  // (16-byte chunk j of row r at chunk j ^ (r % 8)).
  SPEC_DEV void dequant() {
    const int r = threadIdx.x - DQ0, lane = threadIdx.x & 31;
    const int K32 = a.K / 32, nu = u1 - u0;
    const uint16_t* S = (const uint16_t*)a.W.scales;
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    for (int n = 0; n < nu; ++n) {
      const int u = u0 + n, t = u / p.C, c = u - t * p.C, s = n % p.stages;
      // this row's two block scales (zero past the matrix, whose codes read as zero)
      int grow;
      bool valid;
      if (p.map == MAP_PAIR) {
        const int j = t * 64 + (r & 63);
        valid = j < a.geglu_half;
        grow = (r < 64 ? 0 : a.geglu_half) + j;
      } else {
        grow = t * TM + r;
        valid = grow < a.N;
      }
      const unsigned int sw = valid ? __ldg(reinterpret_cast<const unsigned int*>(S + (size_t)grow * K32 + 2 * c)) : 0u;
      int ok = 1;
      if (lane == 0) ok = wait_phase(&full[s], (n / p.stages) & 1, abort_s, err) ? 1 : 0;
      ok = __shfl_sync(FULL, ok, 0);
      if (!ok) break;
      unsigned char* st = stage(s);
      const uint4 q0 = *reinterpret_cast<const uint4*>(st + p.c_off + r * 32);
      const uint4 q1 = *reinterpret_cast<const uint4*>(st + p.c_off + r * 32 + 16);
      const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      unsigned char* whi = st + r * 128;
      unsigned char* wlo = whi + W_BYTES;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)(blk ? sw >> 16 : sw & 0xFFFFu)));
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t w0 = words[blk * 4 + half * 2], w1 = words[blk * 4 + half * 2 + 1];
#pragma unroll
          for (int nib = 0; nib < 2; ++nib) {
            // values 32*blk + 16*nib + 8*half + i, i = 0..7: nibble `nib` of code byte 8*half + i
            const uint32_t n0 = (nib ? w0 >> 4 : w0) & 0x0F0F0F0Fu, n1 = (nib ? w1 >> 4 : w1) & 0x0F0F0F0Fu;
            const uint32_t e[4] = {__byte_perm(n0, 0x6464u, 0x5140), __byte_perm(n0, 0x6464u, 0x5342),
                                   __byte_perm(n1, 0x6464u, 0x5140), __byte_perm(n1, 0x6464u, 0x5342)};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half2 cv = __hsub2(*reinterpret_cast<const __half2*>(&e[i]), off);
              const __half2 h = __hmul2(cv, s2);
              const __half2 l = __hfma2(cv, s2, __hneg2(h));
              hi[i] = *reinterpret_cast<const uint32_t*>(&h);
              lo[i] = *reinterpret_cast<const uint32_t*>(&l);
            }
            const int chunk = blk * 4 + nib * 2 + half;
            const int offc = ((chunk ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(whi + offc) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(wlo + offc) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      // the planes are read by the tensor cores (async proxy)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&wready[s]);
    }
  }

  // ---- epilogue (warps 2-5; thread r of the tile is TMEM lane r) ----

  SPEC_DEV int row() const { return ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31); }

  // The finished tile goes through shared memory: xch[m][r] = row m of the
  // activations, weight row r of the tile, RMSNorm factor applied. The
  // operation's epilogue then runs as short loops over rows, so its code is
  // compact (it runs once per tile, with a cold instruction cache) and every
  // thread can take any (row, column) of the tile.
  SPEC_DEV void finish(int t, const float (&v)[MP], unsigned long long& mybest) {
    const int r = row();
#pragma unroll
    for (int m = 0; m < MP; ++m) xch[m * XCH_LD + r] = v[m] * rms_s[m];
    epi_sync();
    finish_rows(t, 0, a.M, mybest);
    epi_sync();  // xch is free for the next tile
  }

  // The operation's epilogue for activation rows [m0, m1) of the tile in xch.
  SPEC_DEV void finish_rows(int t, int m0, int m1, unsigned long long& mybest) {
    const int r = row(), e = threadIdx.x - EPI0;
    if (p.map == MAP_ROPE) rope(t, r, m0, m1);
    else if (p.map == MAP_PAIR) geglu(t, e, m0, m1);
    else if (a.epi == EPI_ARGMAX) argmax(t, r, e, m0, m1, mybest);
    else store_add(t, r, m0, m1);
  }

  // Cluster mode: each CTA of the cluster holds its K-range's partial tile in
  // xch (unscaled); CTA `rank` sums activation rows [M*rank/S, M*(rank+1)/S)
  // over the cluster's CTAs in rank order (distributed shared memory), scales
  // them and finishes those rows.
  SPEC_DEV void cluster_finish() {
    const int S = p.S, rank = (int)cluster_rank(), t = blockIdx.x / S, r = row();
    const int m0 = (a.M * rank) / S, m1 = (a.M * (rank + 1)) / S;
    if (threadIdx.x == EPI0) stamp(trace, 9);
    for (int m = m0; m < m1; ++m) {
      float u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) u[j] = ld_peer(xch + m * XCH_LD + r, (unsigned)min(j, S - 1));
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc += j < S ? u[j] : 0.f;
      xch[m * XCH_LD + r] = acc * rms_s[m];
    }
    epi_sync();
    if (threadIdx.x == EPI0) stamp(trace, 10);
    unsigned long long unused = 0ull;
    finish_rows(t, m0, m1, unused);
    if (threadIdx.x == EPI0) stamp(trace, 11);
  }

  SPEC_DEV void store_add(int t, int r, int ma, int mb) {
    const int n = t * TM + r;
    if (n >= a.N) return;
    if (a.epi == EPI_ADD) {
      // residual add, 32 rows at a time with the reads ahead of the writes
      for (int m0 = ma; m0 < mb; m0 += 32) {
        float old[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) old[i] = __ldcg(a.Y + (size_t)min(m0 + i, mb - 1) * a.ldy + n);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (m0 + i < mb) a.Y[(size_t)(m0 + i) * a.ldy + n] = old[i] + xch[(m0 + i) * XCH_LD + r];
      }
      return;
    }
#pragma unroll 4
    for (int m = ma; m < mb; ++m) a.Y[(size_t)m * a.ldy + n] = xch[m * XCH_LD + r];
  }

  SPEC_DEV void argmax(int t, int r, int e, int ma, int mb, unsigned long long& mybest) {
    const int n = t * TM + r;
    if (a.Y && n < a.N) {
#pragma unroll 4
      for (int m = ma; m < mb; ++m) a.Y[(size_t)m * a.ldy + n] = xch[m * XCH_LD + r];
    }
    if (e >= ma && e < mb) {
      const int nv = min(TM, a.N - t * TM);
      for (int j = 0; j < nv; ++j) {
        const unsigned long long key = pack_best(xch[e * XCH_LD + j], (uint32_t)(t * TM + j));
        mybest = key > mybest ? key : mybest;
      }
    }
  }

  // gated GELU: tile rows 0-63 are gate rows j = 64t + c, rows 64-127 the
  // matching up rows; thread e takes column c = e % 64 of every other row
  SPEC_DEV void geglu(int t, int e, int ma, int mb) {
    const int c = e & 63, j = t * 64 + c;
    if (j >= a.geglu_half) return;
#pragma unroll 2
    for (int m = ma + (e >> 6); m < mb; m += 2) {
      const float g = xch[m * XCH_LD + c];
      const float gl = 0.5f * g * (1.f + erff(g * 0.70710678118654752f));
      const float v = gl * xch[m * XCH_LD + 64 + c];
      a.Y[(size_t)m * a.ldy + j] = v;
      if (a.wide.out_xs)
        put_planes(a.wide.out_xs, (size_t)m * a.geglu_half + j, (size_t)(MP + m) * a.geglu_half + j, v,
                   a.wide.out_f16);
    }
  }

  // q, k, v head t (head_dim 128): rotate-half RoPE pairs element r with
  // r +- 64; q goes to Y, k and v to the row's slot of the paged cache.
  SPEC_DEV void rope(int t, int r, int ma, int mb) {
    const RopeEpi& E = a.rope;
    const int j = r & 63, h = t;
    const bool second = r >= 64, rot = h < E.nq + E.nkv, is_q = h < E.nq;
    const int plane = rot ? 0 : 1, kh = h - E.nq - plane * E.nkv;
    // the rows' tables were loaded into shared memory at the epilogue start
#pragma unroll 4
    for (int m = ma; m < mb; ++m) {
      const float self = xch[m * XCH_LD + r], part = xch[m * XCH_LD + (r ^ 64)];
      const float co = rope_s[m * TM + 2 * j], si = rope_s[m * TM + 2 * j + 1];
      const float x0 = second ? part : self, x1 = second ? self : part;
      const float y = rot ? (second ? x1 * co + x0 * si : x0 * co - x1 * si) : self;
      if (is_q) {
        a.Y[(size_t)m * a.ldy + h * E.hd + r] = y;
        continue;
      }
      const int page = page_s[m], pos = pos_s[m];
      if (page < 0 || page >= E.n_pages) {
        set_error(E.err, SPEC_ERR_CAPACITY);
        continue;
      }
      __nv_bfloat16* dst = (__nv_bfloat16*)E.pool + E.layer_off +
                           ((((size_t)page * 2 + plane) * E.nkv + kh) * 64 + pos % 64) * E.hd;
      dst[r] = __float2bfloat16_rn(y);
    }
  }

  // Per-launch tables of the RoPE epilogue, loaded while the weights stream.
  SPEC_DEV void load_rope_tables() {
    const RopeEpi& E = a.rope;
    const int e = threadIdx.x - EPI0;
    for (int idx = e; idx < a.M * (TM / 4); idx += 128) {
      const int m = idx / (TM / 4), q = idx - m * (TM / 4);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(E.rope_cs + (size_t)(a.m_base + m) * E.hd) + q);
      *reinterpret_cast<float4*>(rope_s + m * TM + 4 * q) = v;
    }
    if (e < a.M) {
      const int am = a.m_base + e, pos = __ldcg(E.pos + am), pidx = pos / 64;
      pos_s[e] = pos;
      page_s[e] = pidx < E.max_pages ? E.block_table[(size_t)E.seq_ids[am / E.R] * E.max_pages + pidx] : -1;
    }
  }

  // A tile shared with other CTAs: publish this CTA's partial sum; the last
  // CTA to arrive adds all of them in CTA order and finishes the tile.
  SPEC_DEV void partial(int t, int i, float (&v)[MP], unsigned long long& mybest) {
    const int r = row(), e = threadIdx.x - EPI0, b = blockIdx.x;
    const int slot = t == u0 / p.C ? 0 : 1;
    float* f = fix + (size_t)(b * 2 + slot) * MP * TM;
    // all MP rows (the padding rows' sums are exact zeros): no branch between
    // the stores here or the loads below
#pragma unroll
    for (int m = 0; m < MP; ++m) __stcg(f + m * TM + r, v[m]);
    if (a.wide.defer) return;  // the next projection's preparation adds the partials
    epi_sync();
    if (e == 0) stamp(trace, 8);
    if (e == 0) bc[2 + (i & 1)] = (int)atomic_add_acq_rel(cnt + t, 1u);
    epi_sync();
    if (e == 0) stamp(trace, 9);
    const int done = bc[2 + (i & 1)];
    const int bf = cta_of(t * p.C, p), bl = cta_of(t * p.C + p.C - 1, p);
    if (done != bl - bf) return;
#pragma unroll
    for (int m = 0; m < MP; ++m) v[m] = 0.f;
    // two contributors per round of loads, added in CTA order
    for (int bb = bf; bb <= bl; bb += 2) {
      const bool two = bb + 1 <= bl;
      const float* g0 = fix + (size_t)(bb * 2 + (t == unit_begin(bb, p) / p.C ? 0 : 1)) * MP * TM;
      const float* g1 = two ? fix + (size_t)((bb + 1) * 2 + (t == unit_begin(bb + 1, p) / p.C ? 0 : 1)) * MP * TM : g0;
      float u0[MP], u1[MP];
#pragma unroll
      for (int m = 0; m < MP; ++m) {
        u0[m] = __ldcg(g0 + m * TM + r);
        u1[m] = __ldcg(g1 + m * TM + r);
      }
#pragma unroll
      for (int m = 0; m < MP; ++m) {
        v[m] += u0[m];
        if (two) v[m] += u1[m];
      }
    }
    if (e == 0) cnt[t] = 0u;
    if (e == 0) stamp(trace, 10);
    finish(t, v, mybest);
    if (e == 0) stamp(trace, 11);
  }

  SPEC_DEV void epilogue() {
    const int e = threadIdx.x - EPI0;
    grid_dep_wait();
    grid_dep_launch();
    if (e < 64) {
      // 1/rms of each row from the preparation kernel; planes written by the
      // producer are never normalised
      float rv = 0.f;
      if (e < a.M) {
        rv = 1.f;
        if (!a.wide.ready && a.gain) {
          float tot = 0.f;
          for (int y = 0; y < (a.K + PREP_COLS - 1) / PREP_COLS; ++y) tot += __ldcg(inv_rms + e * RMS_PARTS + y);
          rv = rsqrtf(tot / (float)a.K + a.eps);
        }
      }
      rms_s[e] = rv;
    }
    if (p.map == MAP_ROPE) load_rope_tables();
    if (a.epi == EPI_ADD) {
      // the residual rows of this CTA's tiles towards L2 while the weights
      // stream (the finish reads them; they may be out of L2 by now)
      const int t0 = u0 / p.C, t1 = (u1 - 1) / p.C;
      for (int i = e; i < (t1 - t0 + 1) * a.M; i += 128) {
        const int t = t0 + i / a.M, m = i - (i / a.M) * a.M, n0 = t * TM;
        const int cols = min(TM, a.N - n0);
        if (cols > 0 && (cols & 3) == 0) prefetch_l2_bulk(a.Y + (size_t)m * a.ldy + n0, (unsigned)cols * 4);
      }
    }
    epi_sync();
    unsigned long long mybest = 0ull;
    SegIter it{u0, u1, p.C};
    int t, c0, c1, i = 0;
    while (it.next(t, c0, c1)) {
      const int acc = i & 1;
      if (e == 0) bc[i & 1] = wait_phase(&accf[acc], (i >> 1) & 1, abort_s, err) ? 1 : 0;
      epi_sync();
      if (!bc[i & 1]) break;
      if (e == 0) stamp(trace, i == 0 ? 12 : 5);
      fence_after();
      float v[MP];
      const uint32_t taddr = tmem + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)(acc * SET_COLS);
#pragma unroll
      for (int j = 0; j < MP / 16; ++j) {
        // (chain 0: hi + lo) + (chain 1: hi + lo)
        float h0[16], l0[16], h1[16], l1[16];
        tmem_ld16(taddr + 16 * j, h0);
        tmem_ld16(taddr + MP + 16 * j, l0);
        tmem_ld16(taddr + CHAIN_COLS + 16 * j, h1);
        tmem_ld16(taddr + CHAIN_COLS + MP + 16 * j, l1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * j + i] = (h0[i] + l0[i]) + (h1[i] + l1[i]);
      }
      fence_before();
      mbar_arrive(&acce[acc]);
      if (p.S > 1) {
        // cluster mode: this CTA's partial of its one tile stays in shared
        // memory for the cluster's reduction after the roles finish
        const int r = row();
#pragma unroll
        for (int m = 0; m < MP; ++m) xch[m * XCH_LD + r] = v[m];
        if (e == 0) stamp(trace, 8);
      } else if (c0 == 0 && c1 == p.C) {
        finish(t, v, mybest);
      } else {
        partial(t, i, v, mybest);
      }
      if (i == 0 && e == 0) stamp(trace, 13);
      ++i;
    }
    if (a.epi == EPI_ARGMAX && e < a.M && mybest) atomicMax(a.best + e, mybest);
    if (e == 0) stamp(trace, 6);
  }
};

template <int MP, bool Q4>
__global__ void __launch_bounds__(Q4 ? NTHR_Q4 : NTHR, 1)
    wide_kernel(const __grid_constant__ GemvArgs a, const __grid_constant__ Plan p,
                const __grid_constant__ CUtensorMap tmw,
                const __grid_constant__ CUtensorMap tmx, const float* inv_rms, float* fix, unsigned int* cnt,
                int* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t mis = sa(smem_raw) & 1023u;
  unsigned char* base = smem_raw + (mis ? 1024 - mis : 0);
  Cta<MP, Q4> k{a, p, &tmw, &tmx, inv_rms, fix, cnt, err, a.wide.trace};
  if (threadIdx.x == 0) stamp(k.trace, 0);
  k.stages = base;
  k.xch = reinterpret_cast<float*>(base + (size_t)p.stages * p.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(k.xch + MP * XCH_LD);
  k.full = bars;
  k.empty = bars + MAX_STAGES;
  k.wready = bars + 2 * MAX_STAGES;
  k.accf = bars + 3 * MAX_STAGES;
  k.acce = k.accf + 2;
  k.drain = k.acce + 2;
  k.rms_s = reinterpret_cast<float*>(bars + NBARS);
  k.pos_s = reinterpret_cast<int*>(k.rms_s + 64);
  k.page_s = k.pos_s + 64;
  // 16-byte aligned: the exchange tile, barrier block and row tables are multiples of 16 bytes
  k.rope_s = reinterpret_cast<float*>(k.page_s + 64);
  k.tmem_slot = reinterpret_cast<uint32_t*>(k.rope_s + (p.map == MAP_ROPE ? MP * TM : 0));
  k.abort_s = reinterpret_cast<volatile int*>(k.tmem_slot + 1);
  k.bc = const_cast<int*>(k.abort_s) + 1;
  k.u0 = unit_begin(blockIdx.x, p);
  k.u1 = unit_begin(blockIdx.x + 1, p);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&k.full[s], 1);
      mbar_init(&k.empty[s], 1);
      mbar_init(&k.wready[s], 4);  // one arrival per dequantising warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k.accf[i], 1);
      mbar_init(&k.acce[i], 128);
    }
    mbar_init(k.drain, 1);
    *k.abort_s = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sa(k.tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  k.tmem = *k.tmem_slot;
  if (threadIdx.x == 0) stamp(k.trace, 1);

  if (warp == 0) {
    if (lane == 0) k.producer();
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) k.mma_loop();
    __syncwarp();
  } else if (warp < 6) {
    k.epilogue();
  } else if (Q4) {
    k.dequant();
  }
  fence_before();
  __syncthreads();
  if (p.S > 1) {
    // every CTA of the cluster passes both barriers, whatever happened above
    cluster_sync();
    if (warp >= 2 && warp < 6 && !*k.abort_s) k.cluster_finish();
    cluster_sync();
  }
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(k.tmem), "r"(TMEM_COLS) : "memory");
    if (lane == 0) stamp(k.trace, 7);
  }
  if (a.epi != EPI_ARGMAX || a.tail.mode == TAIL_NONE) return;
  // the last CTA to finish runs the accept / commit / draft tail
  grid_dep_wait();
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) k.bc[0] = atomicAdd(a.tail.counter, 1u) == (unsigned)p.grid - 1;
  __syncthreads();
  if (!k.bc[0]) return;
  __threadfence();
  run_tail(a.tail);
}

// Activation rows -> bf16 (f16: fp16) hi/lo planes [2][MP][K] (gain applied) and 1/rms
// per row (1 without a gain, 0 for the padding rows, whose planes are zero).
// Split tiles of an EPI_ADD producer that deferred them: per tile, the first
// contributing CTA, their count and each one's partial-slot offset.
struct FixSrc {
  const float* fix;
  int U, grid, C, T, MP;
};
constexpr int FIX_MAX_T = 128, FIX_MAX_N = 16;

__global__ void __launch_bounds__(128) wide_prep_kernel(float* X, int ldx, int M, int K, const float* gain,
                                                        float eps, int MP, uint16_t* xs, float* rms, int f16,
                                                        FixSrc fx) {
  __shared__ float red[32];
  __shared__ int s_n[FIX_MAX_T];
  __shared__ int s_off[FIX_MAX_T][FIX_MAX_N];
  const int m = blockIdx.x;
  // blocks (m, y) split the row's columns: a fixed split for a given K, so a
  // row's sums do not depend on how many rows the launch has
  const int kb = blockIdx.y * PREP_COLS, ke = min(K, kb + PREP_COLS);
  // The projection that follows may start at once: it fetches only weights
  // until its own wait, which also covers everything this kernel waits for.
  grid_dep_launch();
  if (fx.fix && m < M) {
    Plan q = {};
    q.U = fx.U;
    q.grid = fx.grid;
    q.C = fx.C;
    q.S = 1;
    for (int t = threadIdx.x; t < fx.T; t += blockDim.x) {
      const int bf = cta_of(t * fx.C, q), bl = cta_of(t * fx.C + fx.C - 1, q);
      // a tile within one CTA's range was finished by that CTA
      s_n[t] = bf == bl ? 0 : bl - bf + 1;
      for (int bb = bf; bb <= bl && bb - bf < FIX_MAX_N; ++bb)
        s_off[t][bb - bf] = (bb * 2 + (t == unit_begin(bb, q) / fx.C ? 0 : 1)) * fx.MP * TM;
    }
    __syncthreads();
  }
  grid_dep_wait();
  uint16_t* hi = xs + (size_t)m * K;
  uint16_t* lo = xs + (size_t)(MP + m) * K;
  if (m >= M) {
    for (int c8 = kb + threadIdx.x * 8; c8 < ke; c8 += blockDim.x * 8) {
      *reinterpret_cast<uint4*>(hi + c8) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(lo + c8) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  float ss = 0.f;
  for (int c8 = kb + threadIdx.x * 8; c8 < ke; c8 += blockDim.x * 8) {
    float4 u0 = __ldcg(reinterpret_cast<const float4*>(X + (size_t)m * ldx + c8));
    float4 u1 = __ldcg(reinterpret_cast<const float4*>(X + (size_t)m * ldx + c8 + 4));
    if (fx.fix) {
      const int t = c8 / TM, n = s_n[t];
      if (n > 0) {
        // the tile's partials in CTA order, then the residual: the sum the
        // producer's last CTA would have made
        const int r0 = c8 - t * TM;
        float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
        for (int k0 = 0; k0 < n; k0 += 4) {
          // four contributors' loads in flight, added in order
          float4 p[4][2];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k0 + k < n) {
              const float* g = fx.fix + s_off[t][k0 + k] + (size_t)m * TM + r0;
              p[k][0] = __ldcg(reinterpret_cast<const float4*>(g));
              p[k][1] = __ldcg(reinterpret_cast<const float4*>(g + 4));
            }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k0 + k < n) {
              s0.x += p[k][0].x; s0.y += p[k][0].y; s0.z += p[k][0].z; s0.w += p[k][0].w;
              s1.x += p[k][1].x; s1.y += p[k][1].y; s1.z += p[k][1].z; s1.w += p[k][1].w;
            }
        }
        u0 = make_float4(u0.x + s0.x, u0.y + s0.y, u0.z + s0.z, u0.w + s0.w);
        u1 = make_float4(u1.x + s1.x, u1.y + s1.y, u1.z + s1.z, u1.w + s1.w);
        *reinterpret_cast<float4*>(X + (size_t)m * ldx + c8) = u0;
        *reinterpret_cast<float4*>(X + (size_t)m * ldx + c8 + 4) = u1;
      }
    }
    float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    if (gain) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss = fmaf(v[i], v[i], ss);
        v[i] *= gain[c8 + i];
      }
    }
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (f16) {
        const __half h0 = __float2half_rn(v[2 * i]), h1 = __float2half_rn(v[2 * i + 1]);
        const __half2 hh = __halves2half2(h0, h1);
        const __half2 ll = __floats2half2_rn(v[2 * i] - __half2float(h0), v[2 * i + 1] - __half2float(h1));
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
        l[i] = *reinterpret_cast<const uint32_t*>(&ll);
      } else {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
        const __nv_bfloat162 hh = __halves2bfloat162(h0, h1);
        const __nv_bfloat162 ll =
            __floats2bfloat162_rn(v[2 * i] - __bfloat162float(h0), v[2 * i + 1] - __bfloat162float(h1));
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
        l[i] = *reinterpret_cast<const uint32_t*>(&ll);
      }
    }
    *reinterpret_cast<uint4*>(hi + c8) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + c8) = make_uint4(l[0], l[1], l[2], l[3]);
  }
  if (gain) {
    const float tot = block_sum(ss, red);
    if (threadIdx.x == 0) rms[m * RMS_PARTS + blockIdx.y] = tot;
  }
}

// ---- host -------------------------------------------------------------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void init_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
}

// Row-major bf16 [rows][inner] as a 2-D tensor; boxes of box_rows x 64
// columns land in the 128-byte swizzle layout. Rows past the end read as zero.
bool encode(CUtensorMap* m, const void* base, int inner, int rows, int box_rows) {
  if (!g_encode || ((uintptr_t)base & 15) || (inner * 2) % 16) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)KC, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// shared memory besides the stages: exchange tile, barriers, per-row tables,
// the RoPE rows (RoPE epilogue only), tensor-memory slot, flags, 1 KB alignment
// Q4_0 codes [rows][inner bytes] as a 2-D uint8 tensor, boxes of box_rows x
// 32 bytes (64 values), no swizzle.
bool encode_codes(CUtensorMap* m, const void* base, int inner, int rows, int box_rows) {
  if (!g_encode || ((uintptr_t)base & 15) || inner % 16) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)inner};
  const cuuint32_t box[2] = {(cuuint32_t)(KC / 2), (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t fixed_smem(int MP, bool rope) {
  return (size_t)MP * XCH_LD * 4 + NBARS * 8 + 3 * 64 * 4 + (rope ? (size_t)MP * TM * 4 : 0) + 4 + 4 + 16 + 1024;
}

const void* kernel_of(int MP, bool q4) {
  switch (MP) {
    case 16: return q4 ? (const void*)wide_kernel<16, true> : (const void*)wide_kernel<16, false>;
    case 32: return q4 ? (const void*)wide_kernel<32, true> : (const void*)wide_kernel<32, false>;
    case 48: return q4 ? (const void*)wide_kernel<48, true> : (const void*)wide_kernel<48, false>;
    default: return q4 ? (const void*)wide_kernel<64, true> : (const void*)wide_kernel<64, false>;
  }
}

// Clusters of S CTAs of this kernel and shared memory that the GPU holds at
// once (cached).
int max_clusters(const Plan& p) {
  static std::mutex mu;
  static std::map<long long, int> cache;
  const long long key = ((long long)p.MP * 2 + p.q4) * 16 * (1 << 20) + (long long)p.S * (1 << 20) + p.smem;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.T * p.S);
  cfg.blockDim = dim3(p.q4 ? NTHR_Q4 : NTHR);
  cfg.dynamicSmemBytes = p.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel_of(p.MP, p.q4), &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

template <int MP>
cudaError_t launch_mp(const cudaLaunchConfig_t& cfg, const GemvArgs& a, const Plan& p, const CUtensorMap& tmw,
                      const CUtensorMap& tmx) {
  return p.q4 ? cudaLaunchKernelEx(&cfg, wide_kernel<MP, true>, a, p, tmw, tmx, (const float*)a.wide.rms, a.wide.fix,
                                   a.tc_cnt, a.wide.err)
              : cudaLaunchKernelEx(&cfg, wide_kernel<MP, false>, a, p, tmw, tmx, (const float*)a.wide.rms, a.wide.fix,
                                   a.tc_cnt, a.wide.err);
}

}  // namespace

bool make_plan(const GemvArgs& a, int nsm, Plan& p) {
  p.map = a.epi == EPI_GEGLU ? MAP_PAIR : a.epi == EPI_ROPE ? MAP_ROPE : MAP_PLAIN;
  if (a.K % KC || a.M < 1 || a.M > 64 || a.N < 1) return false;
  if (p.map == MAP_ROPE && (a.rope.hd != TM || a.N != (a.rope.nq + 2 * a.rope.nkv) * a.rope.hd)) return false;
  if (p.map == MAP_PAIR && (a.geglu_half < 1 || a.N != 2 * a.geglu_half)) return false;
  p.T = p.map == MAP_PAIR ? (a.geglu_half + 63) / 64 : (a.N + TM - 1) / TM;
  p.C = a.K / KC;
  p.U = p.T * p.C;
  // few tiles: a cluster of S CTAs per tile (reduced in distributed shared
  // memory); the launcher lowers S until every cluster is resident at once
  p.S = 1;
  if (a.epi != EPI_ARGMAX && 2 * p.T <= nsm) p.S = std::min(std::min(8, nsm / p.T), p.C);
  p.grid = p.S > 1 ? p.T * p.S : std::min(p.U, nsm);
  p.MP = (a.M + 15) / 16 * 16;
  p.q4 = a.W.dtype == DT_Q4_0;
  if (p.q4 && !a.W.scales) return false;
  const int xbytes = 2 * p.MP * KC * 2;
  if (p.q4) {
    // [hi plane | lo plane | activation planes | codes]
    p.x_off = 2 * W_BYTES;
    p.c_off = 2 * W_BYTES + xbytes;
    p.stage_bytes = 2 * W_BYTES + xbytes + CODE_BYTES;
    p.tx_bytes = xbytes + CODE_BYTES;
  } else {
    // [weights | activation planes]
    p.x_off = W_BYTES;
    p.c_off = 0;
    p.stage_bytes = W_BYTES + xbytes;
    p.tx_bytes = p.stage_bytes;
  }
  const size_t fixed = fixed_smem(p.MP, p.map == MAP_ROPE);
  p.stages = (int)std::min<size_t>(MAX_STAGES, (SMEM_LIMIT - fixed) / p.stage_bytes);
  if (p.stages < 2) return false;
  p.smem = (int)(p.stages * (size_t)p.stage_bytes + fixed);
  return true;
}

}  // namespace wide

using namespace wide;

void setup_gemv_wide_attributes() {
  cudaFuncSetAttribute(wide_kernel<16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<48, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<48, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  cudaFuncSetAttribute(wide_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
}

size_t gemv_wide_fix_bytes() { return (size_t)num_sms() * 2 * 64 * TM * sizeof(float); }

bool gemv_wide_ok(const GemvArgs& a) {
  Plan p;
  return (a.W.dtype == DT_BF16 || a.W.dtype == DT_Q4_0) && a.wide.xs && a.wide.rms && a.wide.fix && a.tc_cnt &&
         (!a.gain || (a.K + PREP_COLS - 1) / PREP_COLS <= RMS_PARTS) &&
         a.K <= a.wide.kmax && make_plan(a, num_sms(), p);
}

namespace {
// make_plan, then the launch's cluster decision and grid
bool final_plan(const GemvArgs& a, Plan& p) {
  std::call_once(g_once, init_encode);
  if (!make_plan(a, num_sms(), p)) return false;
  while (p.S > 1 && max_clusters(p) < p.T) --p.S;
  // The cluster reduction removes the split-tile tail (about 10 us) but leaves
  // nsm - T*S SMs idle: keep it only while the streaming time those SMs would
  // have saved (the weights at about 6 TB/s) stays under about 5 us, and only
  // for matrices of at most 64 MB (larger ones measured slower inside the
  // pipelined pass, where a cluster waits for S free SMs of one GPC).
  if (p.S > 1) {
    const double wbytes = (double)a.N * a.K * (p.q4 ? 0.5625 : 2.0);
    const double lost_us = wbytes / 6.0e6 * ((double)num_sms() / (p.T * p.S) - 1.0);
    if (lost_us > 5.0 || wbytes > 64.0 * (1 << 20)) p.S = 1;
  }
  if (p.S <= 1) {
    p.S = 1;
    p.grid = std::min(p.U, num_sms());
  } else {
    p.grid = p.T * p.S;
  }
  return true;
}
}  // namespace

WideSplit gemv_wide_split(const GemvArgs& a) {
  WideSplit w = {};
  Plan p;
  if (!final_plan(a, p)) return w;
  w.U = p.U;
  w.grid = p.grid;
  w.C = p.C;
  w.T = p.T;
  // CTAs on one tile: at most ceil(C / smallest range) + 1
  const int per = p.U / p.grid;
  const int most = per > 0 ? (p.C + per - 1) / per + 1 : p.grid;
  w.deferrable = p.S == 1 && p.map == MAP_PLAIN && p.T <= FIX_MAX_T && most <= FIX_MAX_N;
  return w;
}

// M in 1..64 rows, bf16 weights, K % 64 == 0 (gemv_wide_ok). Launches the
// activation preparation (unless the planes are ready) and the projection;
// returns the number of kernels, or -1 on an error.
int gemv_wide(const GemvArgs& a, cudaStream_t st) {
  Plan p;
  if (!final_plan(a, p)) return -1;
  if (a.wide.defer && (p.S != 1 || !gemv_wide_split(a).deferrable)) return -1;
  CUtensorMap tmw, tmx;
  const int box_rows = p.map == MAP_PAIR ? 64 : TM;
  const bool wok = p.q4 ? encode_codes(&tmw, a.W.data, a.K / 2, a.N, box_rows) : encode(&tmw, a.W.data, a.K, a.N, box_rows);
  if (!wok || !encode(&tmx, a.wide.xs, a.K, 2 * p.MP, 2 * p.MP)) return -1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pc = {};
  // PREP_COLS columns a block, a thread per 8 columns
  pc.gridDim = dim3(p.MP, (a.K + PREP_COLS - 1) / PREP_COLS);
  pc.blockDim = dim3(PREP_COLS / 8);
  pc.stream = st;
  pc.attrs = attr;
  pc.numAttrs = a.pdl ? 1 : 0;
  FixSrc fx = {};
  if (a.wide.fix_src) {
    fx.fix = a.wide.fix_src;
    fx.U = a.wide.fix_U;
    fx.grid = a.wide.fix_grid;
    fx.C = a.wide.fix_C;
    fx.T = a.wide.fix_T;
    fx.MP = p.MP;
    if (a.wide.ready || fx.T > FIX_MAX_T || a.K != fx.T * TM) return -1;
  }
  if (!a.wide.ready && cudaLaunchKernelEx(&pc, wide_prep_kernel, const_cast<float*>(a.X), a.ldx, a.M, a.K,
                                          a.gain, a.eps, p.MP, a.wide.xs, a.wide.rms, p.q4, fx) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = pc;
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.q4 ? NTHR_Q4 : NTHR);
  cfg.dynamicSmemBytes = p.smem;
  cudaLaunchAttribute attr2[2];
  attr2[0] = attr[0];
  attr2[1].id = cudaLaunchAttributeClusterDimension;
  attr2[1].val.clusterDim.x = p.S;
  attr2[1].val.clusterDim.y = 1;
  attr2[1].val.clusterDim.z = 1;
  cfg.attrs = a.pdl ? attr2 : attr2 + 1;
  cfg.numAttrs = (a.pdl ? 1 : 0) + (p.S > 1 ? 1 : 0);
  cudaError_t e;
  switch (p.MP) {
    case 16: e = launch_mp<16>(cfg, a, p, tmw, tmx); break;
    case 32: e = launch_mp<32>(cfg, a, p, tmw, tmx); break;
    case 48: e = launch_mp<48>(cfg, a, p, tmw, tmx); break;
    default: e = launch_mp<64>(cfg, a, p, tmw, tmx); break;
  }
  return e == cudaSuccess ? (a.wide.ready ? 1 : 2) : -1;
}

}  // namespace spec
