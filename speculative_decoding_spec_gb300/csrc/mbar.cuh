// mbar.cuh -- shared-memory mbarrier and bulk asynchronous copy primitives
// (PTX mbarrier.*, cp.async.bulk.*) used by the kernels that stream weights
// through shared-memory rings.
#pragma once
#include <stdint.h>

#include "common.cuh"

namespace spec {

// 32-bit shared-memory address of a generic pointer into shared memory.
SPEC_DEV uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

SPEC_DEV void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(count) : "memory");
}
// Makes barrier initialisation visible to the async proxy and the cluster.
SPEC_DEV void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// One arrival that also expects `bytes` of asynchronous copies to complete.
SPEC_DEV void mbar_expect_tx(uint64_t* b, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
}
SPEC_DEV void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
// Non-blocking test: true once the phase with parity `parity` has completed.
SPEC_DEV bool mbar_test(uint64_t* b, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Global -> this CTA's shared memory, completion counted on `bar` in bytes.
SPEC_DEV void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   sa(dst)),
               "l"(src), "r"(bytes), "r"(sa(bar))
               : "memory");
}

SPEC_DEV unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace spec
