// nvfp4_gemm_noalloc: nvfp4_gemm whose split-K scratch is a static device array of the
// library, for callers that cannot hand over a workspace (see the declaration in nvfp4.h).
//
// The array lives in this translation unit alone, so with lazy module loading (the CUDA
// default) its memory is taken only by processes that call this entry point.  Its address is
// looked up with cudaGetSymbolAddress once per device and context; nothing here allocates
// device memory.
#include <mutex>

#include "ptx.cuh"
#include "host.h"

namespace {

// Scratch of the stream-K split: arrival counters first, then the fp32 partial-tile slots.
// Sized for every plan nvfp4_gemm picks on a GPU of up to kMaxSms SMs: stream-K plans run one
// CTA per SM on 128-wide tiles and split at most sm_count / 2 tiles.  Larger needs are refused.
constexpr int kMaxSms = 160;
constexpr size_t kScratchBytes = (size_t(20) << 20) + 4096;
static_assert(kScratchBytes >= nvfp4::stream_k_workspace_bytes(kMaxSms / 2, kMaxSms, 128),
              "the static scratch must hold the largest stream-K workspace");
__device__ __align__(256) unsigned char g_gemm_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx = 0;  // context the address was looked up in (0: not yet)
  void *ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_mu;

// Device address of the scratch on the current device.  The lookup is made on the first call
// on each device, and again whenever the device has a new context (after a device reset the
// module is loaded anew and the array may sit elsewhere).
nvfp4_status_t scratch_address(int dev, void **out) {
  if (dev < 0 || dev >= kMaxDevices) return nvfp4::fail(NVFP4_ERR_UNSUPPORTED_DEVICE, "device %d out of range", dev);
  const unsigned long long ctx = nvfp4::current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot &s = g_slots[dev];
  if (ctx == 0 || s.ctx != ctx) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_gemm_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      s.ctx = 0;
      return nvfp4::fail(NVFP4_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    }
    s.ptr = p;
    s.ctx = ctx;
  }
  *out = s.ptr;
  return NVFP4_OK;
}

// Zeroes the arrival counters at the head of the scratch.  Launched with the GEMM's own PDL
// setting, it lets the GEMM launch at once (the GEMM only touches the counters after its own
// dependency wait) and itself clears only once the preceding kernel -- possibly an earlier GEMM
// on the same scratch -- has completed, so a chain producer -> GEMM keeps its overlap.
__global__ void __launch_bounds__(256) clear_counters_kernel(unsigned int *counters, int words) {
  nvfp4::pdl_trigger();
  nvfp4::pdl_wait();
  for (int i = threadIdx.x; i < words; i += blockDim.x) counters[i] = 0u;
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
  st = scratch_address(dev.device, &scratch);
  if (st != NVFP4_OK) return st;
  // The per-tile arrival counters at the head of the scratch must read zero when the kernel
  // starts.  Every call that completes leaves them zero, but one that timed out may not, so they
  // are cleared on the stream before each launch (the partial-tile slots need no clearing).
  nvfp4_gemm_plan_t plan;
  st = nvfp4_gemm_plan(m, n, k, &plan);
  if (st != NVFP4_OK) return st;
  const int words = plan.sk_tiles;
  const cudaError_t e = nvfp4::launch(clear_counters_kernel, dim3(1), dim3(256), 0, (cudaStream_t)stream,
                                      (flags & NVFP4_FLAG_PDL) != 0, 1, static_cast<unsigned int *>(scratch), words);
  if (e != cudaSuccess) return nvfp4::check_launch(e, "nvfp4_gemm_noalloc (clearing the counters)");
  return nvfp4_gemm(a, sfa, b, sfb, alpha, d, m, n, k, scratch, kScratchBytes, flags, stream);
}
