// linear_noalloc.cu -- spec_linear for callers that cannot allocate device
// memory.
//
// Some hosts of this library own every device allocation themselves: an
// inference server with a fixed device-memory budget carved up at start-up, a
// plugin loaded into a framework whose allocator must account for all memory,
// or code that must never reach cudaMalloc because it may synchronise the
// device. Such callers cannot hand spec_linear a workspace of their own. This
// entry point runs the same projection kernel with its scratch (split-tile
// partial sums and per-tile arrival counters) in a fixed-size array that lives
// in the library's own device image: the array is created when the library is
// loaded on a device and stays until the process exits.
//
// The first call on each device looks up the array's device address with that
// device current (cudaGetSymbolAddress); make that first call before any
// stream capture. Every call shares the one array, so calls that overlap on the
// GPU (different streams, or different host threads) race on it: serialise
// them. The counters must start at zero; each call clears them on its stream
// before the launch.
#include <mutex>

#include "../../include/spec.h"
#include "kernels.h"

namespace {

constexpr size_t FIX_BYTES = 256 * 1024;   // split-tile partials: 1 KiB per SM, up to 256 SMs
constexpr size_t CNT_BYTES = 256 * 1024;   // per-tile arrival counters (4 B per 8 output rows, + 64)
constexpr size_t SCRATCH_BYTES = FIX_BYTES + CNT_BYTES;

static __device__ __align__(256) unsigned char g_linear_scratch[SCRATCH_BYTES];

using spec::MAX_DEVICES;
std::mutex g_mu;
void* g_addr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_linear_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool mat_ok(const spec_matrix& m, int K) {
  if (!m.data) return false;
  if (m.dtype == SPEC_Q4_0) return m.scales && K % 32 == 0;
  if (m.dtype == SPEC_F32 || m.dtype == SPEC_BF16) return K % 8 == 0;
  return false;
}

}  // namespace

extern "C" spec_status spec_linear_noalloc(const spec_matrix* w, int32_t N, int32_t K, const float* x, int32_t M,
                                           const float* gain, float eps, float* y, void* stream) {
  if (!w || !x || !y || N <= 0 || K <= 0 || M <= 0 || M > 64 || !mat_ok(*w, K)) return SPEC_EINVAL;
  if (N > SPEC_LINEAR_NOALLOC_MAX_ROWS) return SPEC_ECAPACITY;
  const size_t cnt_bytes = ((size_t)N / 8 + 64) * sizeof(unsigned int);
  if (spec::gemv_tc_fixup_bytes() > FIX_BYTES || cnt_bytes > CNT_BYTES) return SPEC_ECAPACITY;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return SPEC_ECUDA;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned int* cnt = (unsigned int*)((char*)base + FIX_BYTES);
  if (cudaMemsetAsync(cnt, 0, cnt_bytes, st) != cudaSuccess) return SPEC_ECUDA;
  spec::setup_device_attributes();
  spec::GemvArgs g = {};
  g.X = x; g.ldx = K; g.M = M; g.N = N; g.K = K;
  g.W = spec::Mat{w->dtype, w->data, w->scales};
  g.gain = gain; g.eps = eps;
  g.epi = spec::EPI_STORE; g.Y = y; g.ldy = N; g.pdl = 0; g.prefetch = 0;
  g.tc_fix = (float*)base;
  g.tc_cnt = cnt;
  if (spec::gemv(g, st) < 0) return SPEC_ECUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
