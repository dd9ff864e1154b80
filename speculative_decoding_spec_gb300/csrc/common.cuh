// common.cuh -- device helpers shared by the sm_103a kernels of the
// speculative-decoding hot path.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

#define SPEC_DEV __device__ __forceinline__

namespace spec {

constexpr unsigned FULL = 0xffffffffu;

SPEC_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
SPEC_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

SPEC_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
SPEC_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024). `red` holds 32 floats.
SPEC_DEV float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
SPEC_DEV uint32_t ord_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
SPEC_DEV float ord_val(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Packed (score, index) key: the larger score wins, then the LOWER index.
SPEC_DEV unsigned long long pack_best(float v, uint32_t idx) {
  return ((unsigned long long)ord_key(v) << 32) | (unsigned long long)(0xffffffffu - idx);
}
SPEC_DEV uint32_t best_index(unsigned long long k) { return 0xffffffffu - (uint32_t)(k & 0xffffffffu); }
SPEC_DEV float best_value(unsigned long long k) { return ord_val((uint32_t)(k >> 32)); }

SPEC_DEV unsigned long long volatile_load(const unsigned long long* p) {
  return *(const volatile unsigned long long*)p;
}

// Device-scope add with acquire-release ordering: the warp's earlier writes
// (ordered to lane 0 by a __syncwarp) are visible to whoever observes the new
// count, and reads after it see every write released before earlier adds.
SPEC_DEV unsigned int atomic_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

SPEC_DEV unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
SPEC_DEV void st_release(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

SPEC_DEV void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch: a kernel launched with the PDL attribute may
// start before its predecessor finishes; it must not read the predecessor's
// outputs before grid_dep_wait(). Weights do not depend on earlier kernels, so
// they may be fetched before the wait.
SPEC_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SPEC_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Prefetch one 128-byte line into L2 (no register or shared-memory cost).
SPEC_DEV void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
// Prefetch a contiguous range into L2 with one bulk (TMA) request; p 16-byte
// aligned, bytes a multiple of 16.
SPEC_DEV void prefetch_l2_bulk(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 128-bit streaming load of weights: read once, do not keep in L1.
SPEC_DEV uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
SPEC_DEV uint2 ldg_stream8(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

SPEC_DEV float load_kv(const float* p) { return *p; }
SPEC_DEV float load_kv(const __nv_bfloat16* p) { return __bfloat162float(*p); }
SPEC_DEV void store_kv(float* p, float v) { *p = v; }
SPEC_DEV void store_kv(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

}  // namespace spec
