// gemv_tc.cu -- launcher of the tensor-core weight-streaming projection
// (body in gemv_tc.cuh).
#include "gemv_tc.cuh"

namespace spec {
namespace tc {

// Q4: Q4_0 weights (exact codes in fp16 fragments, block scales in fp32); else bf16.
template <bool Q4>
__global__ void __launch_bounds__(TW_DEFAULT * 32, 1) gemv_tc_kernel(GemvArgs a, SkPlan p, int map, float* fix,
                                                             unsigned int* cnt) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Sk<TW_DEFAULT, Q4> k{a, p, map};
  sk_bind(k, smem_raw, fix, cnt, blockIdx.x, true);
  k.trace = a.tc_trace ? a.tc_trace + (size_t)blockIdx.x * 16 : nullptr;
  k.run();
}

}  // namespace tc

using namespace tc;

void setup_gemv_tc_attributes() {
  cudaFuncSetAttribute(gemv_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
  cudaFuncSetAttribute(gemv_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
}

// bf16 weights with K % 32 == 0, or Q4_0 weights with K % 128 == 0; M <= 8.
// Returns 1 on launch, -2 when the shape is not handled here (the caller uses
// the CUDA-core kernel), -1 on a launch error. fix / cnt: fixup scratch of at
// least gemv_tc_fixup_bytes() and a zeroed counter array of at least
// gemv_tc_counters() entries.
int gemv_tc(const GemvArgs& a, float* fix, unsigned int* cnt, cudaStream_t st) {
  const int map = a.epi == EPI_GEGLU ? MAP_PAIR : a.epi == EPI_ROPE ? MAP_ROPE : MAP_PLAIN;
  if (map == MAP_ROPE && (a.rope.hd % 16 || a.N != (a.rope.nq + 2 * a.rope.nkv) * a.rope.hd)) return -1;
  const bool q4 = a.W.dtype == DT_Q4_0;
  if (!q4 && a.W.dtype != DT_BF16) return -2;
  if (q4 && (a.K % 128 || !a.W.scales)) return -2;
  if (a.K % 32 || a.M > 8 || a.M < 1 || !fix || !cnt) return -2;
  const SkPlan p = plan<TW_DEFAULT>(a, map, num_sms());
  if (p.smem > (size_t)SMEM_MAX) return -2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(TW_DEFAULT * 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  const cudaError_t e = q4 ? cudaLaunchKernelEx(&cfg, gemv_tc_kernel<true>, a, p, map, fix, cnt)
                           : cudaLaunchKernelEx(&cfg, gemv_tc_kernel<false>, a, p, map, fix, cnt);
  return e == cudaSuccess ? 1 : -1;
}

size_t gemv_tc_fixup_bytes() { return (size_t)num_sms() * 2 * 32 * 16; }

}  // namespace spec
