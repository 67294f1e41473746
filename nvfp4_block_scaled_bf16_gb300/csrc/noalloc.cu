// nvfp4_gemm_noalloc: nvfp4_gemm whose split-K scratch is a static device array of the
// library, for callers that cannot hand over a workspace (see the declaration in nvfp4.h).
//
// The array lives in this translation unit alone, so with lazy module loading (the CUDA
// default) its 20 MiB are taken only by processes that call this entry point.  Its address is
// looked up once per device with cudaGetSymbolAddress; nothing here allocates device memory.
#include <mutex>

#include "host.h"

namespace {

// Scratch of the stream-K split: arrival counters first, then the fp32 partial-tile slots.
// 20 MiB holds the workspace of every plan nvfp4_gemm picks on a GPU of up to 160 SMs (at most
// 2 slots of 128 x 128 fp32 per CTA plus the counters); larger needs are refused.
constexpr size_t kScratchBytes = size_t(20) << 20;
__device__ __align__(256) unsigned char g_gemm_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  bool looked_up = false;
  cudaError_t err = cudaSuccess;
  void *ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_mu;

// Device address of the scratch on the current device (looked up once per device).
nvfp4_status_t scratch_address(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nvfp4::fail(NVFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return nvfp4::fail(NVFP4_ERR_UNSUPPORTED_DEVICE, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot &s = g_slots[dev];
  if (!s.looked_up) {
    s.err = cudaGetSymbolAddress(&s.ptr, g_gemm_scratch);
    if (s.err != cudaSuccess) cudaGetLastError();
    s.looked_up = true;
  }
  if (s.err != cudaSuccess)
    return nvfp4::fail(NVFP4_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(s.err));
  *out = s.ptr;
  return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status_t nvfp4_gemm_noalloc(const uint8_t *a, const uint8_t *sfa, const uint8_t *b,
                                             const uint8_t *sfb, const float *alpha, void *d, int64_t m,
                                             int64_t n, int64_t k, uint32_t flags, nvfp4_stream_t stream) {
  nvfp4::clear_error();
  size_t need = 0;
  if (m > 0 && n > 0 && k > 0 && nvfp4_gemm_workspace_size(m, n, k, &need) != NVFP4_OK) return NVFP4_ERR_INVALID_ARG;
  if (need == 0)  // no tile is split (or the arguments are invalid): nvfp4_gemm reports the rest
    return nvfp4_gemm(a, sfa, b, sfb, alpha, d, m, n, k, nullptr, 0, flags, stream);
  if (need > kScratchBytes)
    return nvfp4::fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                       "nvfp4_gemm_noalloc: m=%lld n=%lld k=%lld needs %zu bytes of split-K scratch, the static "
                       "scratch holds %zu; use nvfp4_gemm with a workspace",
                       (long long)m, (long long)n, (long long)k, need, kScratchBytes);
  // nvfp4_gemm's argument checks, made here too so that nothing is enqueued for a call it
  // would refuse (the counter clearing below goes on the stream first)
  if (k % 32 || n % 32 || m >= (1LL << 31) || n >= (1LL << 31) || k >= (1LL << 31))
    return nvfp4_gemm(a, sfa, b, sfb, alpha, d, m, n, k, nullptr, 0, flags, stream);
  if (!a || !sfa || !b || !sfb || !alpha || !d || !nvfp4::aligned(a, 32) || !nvfp4::aligned(b, 32) ||
      !nvfp4::aligned(d, 32) || !nvfp4::aligned(sfa, 16) || !nvfp4::aligned(sfb, 16) || !nvfp4::aligned(alpha, 4) ||
      (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT | NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD | NVFP4_FLAG_SF_SM103)))
    return nvfp4_gemm(a, sfa, b, sfb, alpha, d, m, n, k, nullptr, 0, flags, stream);
  nvfp4::DeviceInfo dev;
  nvfp4_status_t st = nvfp4::current_device(&dev);
  if (st != NVFP4_OK) return st;
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != NVFP4_OK) return st;
  // The per-tile arrival counters at the head of the scratch must read zero when the kernel
  // starts.  Every call that completes leaves them zero, but one that timed out may not, so they
  // are cleared on the stream before each launch (the partial-tile slots need no clearing).
  nvfp4_gemm_plan_t plan;
  st = nvfp4_gemm_plan(m, n, k, &plan);
  if (st != NVFP4_OK) return st;
  const size_t counter_bytes = (static_cast<size_t>(plan.sk_tiles) * 4 + 255) / 256 * 256;
  cudaError_t e = cudaMemsetAsync(scratch, 0, counter_bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return nvfp4::fail(NVFP4_ERR_CUDA, "nvfp4_gemm_noalloc: clearing the counters: %s", cudaGetErrorString(e));
  }
  return nvfp4_gemm(a, sfa, b, sfb, alpha, d, m, n, k, scratch, kScratchBytes, flags, stream);
}
