// attn_tc.cu -- launcher of the tensor-core paged attention (body in
// attn_tc.cuh).
#include "attn_tc.cuh"

namespace spec {
namespace atc {

template <int HD>
__global__ void __launch_bounds__(256) attn_tc_kernel(AttnArgs a, int pps, unsigned int* counters, size_t smem_bytes) {
  extern __shared__ __align__(16) unsigned char smem[];
  AttnTc<HD>::run(a, pps, counters, smem, blockIdx.x, blockIdx.y, true, smem_bytes);
}

// Balanced launch: one CTA per SM over the flattened pages of every
// (sequence, KV head) pair.
template <int HD>
__global__ void __launch_bounds__(256) attn_tc_bal_kernel(AttnArgs a, unsigned int* counters, size_t smem_bytes) {
  extern __shared__ __align__(16) unsigned char smem[];
  AttnTc<HD>::run_balanced(a, counters, smem, smem_bytes);
}

}  // namespace atc

using namespace atc;

// warps per attention CTA (stand-alone and persistent launches alike)
constexpr int ATT_WARPS = 8;

static int host_qt(int qn) { return (qn + 15) / 16; }
static int host_page_slots(int qn) {
  const int qt = host_qt(qn), kg = qt == 1 ? 4 : 1;
  const int ps = ATT_WARPS / (qt * kg);
  return ps > 0 ? ps : 1;
}

// Query hi/lo tiles, the fp32 query rows and the r RoPE rows, then the page
// slots or, after the rounds, the warp combine.
size_t attention_tc_smem(int hd, int qn, int r) {
  const int qt = host_qt(qn), st = hd + 8, pw = host_page_slots(qn);
  const size_t pages = (size_t)2 * pw * PAGE * st * 2;
  const size_t combine = (size_t)ATT_WARPS * 16 * (hd + 2) * 4 + (size_t)qt * 16 * 4;
  const size_t qstage = (size_t)(qn + r) * hd * 4;
  return (size_t)2 * qt * 16 * st * 2 + qstage + std::max(pages, combine);
}

// Shared memory of a CTA running the attention with `pw` page slots.
size_t attention_tc_smem_slots(int hd, int qn, int r, int pw) {
  const int qt = host_qt(qn), st = hd + 8, kg = qt == 1 ? 4 : 1;
  const size_t pages = (size_t)2 * pw * PAGE * st * 2;
  const size_t combine = (size_t)qt * kg * pw * 16 * (hd + 2) * 4 + (size_t)qt * 16 * 4;
  const size_t qstage = (size_t)(qn + r) * hd * 4;
  return (size_t)2 * qt * 16 * st * 2 + qstage + std::max(pages, combine);
}

void setup_attn_tc_attributes() {
  cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(attn_tc_bal_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(attn_tc_bal_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

// Splits of the page range: about one CTA per SM, at most 32 splits (the
// merge reads every split's partial); a split is a whole number of rounds of
// the CTA's page slots.
int attention_tc_splits(int B, int nkv, int max_pages, int* pps, int qn) {
  const int pw = host_page_slots(qn);
  const int target = std::max(1, num_sms() / std::max(1, B * nkv));
  const int n = std::max(1, std::min(std::min((max_pages + pw - 1) / pw, target), 32));
  int p = (max_pages + n - 1) / n;
  p = (p + pw - 1) / pw * pw;
  *pps = p;
  return (max_pages + p - 1) / p;
}

int attention_tc(const AttnArgs& a0, unsigned int* counters, int pps, cudaStream_t st) {
  AttnArgs a = a0;
  const int QN = a.R * (a.nq / a.nkv);
  const int qt = (QN + 15) / 16;
  // Batches (up to 64 sequences): the balanced launch, where each (sequence,
  // KV head) pair gets CTAs in proportion to its pages, so ragged contexts do
  // not leave the longest sequences with the most rounds per CTA; one
  // sequence: fixed splits of the page capacity. The partials of a balanced
  // launch have one slot per page of a sequence (the callers' buffers hold
  // max_pages splits per row and head).
  const bool balanced = a.B > 1 && a.B <= 64;
  if (balanced) a.n_split = a.max_pages;
  size_t smem = attention_tc_smem(a.hd, QN, a.R);
  if (smem > 200 * 1024) return -2;
  // room for staging every split partial in the merge, when it fits: a pair's
  // splits in the balanced launch are at most one per round of page slots of
  // its pages, plus one
  const int pw = host_page_slots(QN);
  const int nsplit_max = balanced ? std::min(a.max_pages, (a.max_pages + pw - 1) / pw + 1) : a.n_split;
  const size_t merge = ((size_t)QN * nsplit_max + 4) * 4 + (size_t)QN * nsplit_max * a.hd * 4;
  if (merge <= 200 * 1024) smem = std::max(smem, merge);
  cudaLaunchConfig_t cfg = {};
  // balanced: one CTA per SM, and at least one per (sequence, KV head) pair
  const int nbal = std::max(num_sms(), a.B * a.nkv);
  cfg.gridDim = balanced ? dim3(nbal) : dim3(a.B * a.nkv, a.n_split);
  cfg.blockDim = dim3(ATT_WARPS * 32);
  (void)qt;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.hd == 128)
    e = balanced ? cudaLaunchKernelEx(&cfg, attn_tc_bal_kernel<128>, a, counters, smem)
                 : cudaLaunchKernelEx(&cfg, attn_tc_kernel<128>, a, pps, counters, smem);
  else if (a.hd == 64)
    e = balanced ? cudaLaunchKernelEx(&cfg, attn_tc_bal_kernel<64>, a, counters, smem)
                 : cudaLaunchKernelEx(&cfg, attn_tc_kernel<64>, a, pps, counters, smem);
  else return -2;
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace spec
