// Library-wide host state: error messages, device checks, the device status word, tensor
// maps, and the size queries of the C ABI.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "host.h"

namespace nvfp4 {

// Set by kernels whose bounded pipeline wait gave up; read and cleared by nvfp4_check_status.
__device__ unsigned int g_status_word;

namespace {
thread_local char t_msg[512] = "";

constexpr int kMaxDevices = 64;
struct DevState {
  // context the fields below were filled in for (0: not yet); set (release) after them
  std::atomic<unsigned long long> ctx{0};
  bool ok = false;
  DeviceInfo info{};
  char why[200] = "";
};
DevState g_dev[kMaxDevices];
std::mutex g_mu;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

struct SmemEntry {
  const void *fn;
  int device;
  unsigned long long ctx;  // the attribute belongs to the context it was set in
  int bytes;
};
SmemEntry g_smem[256];
int g_smem_n = 0;
}  // namespace

nvfp4_status_t fail(nvfp4_status_t code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { t_msg[0] = '\0'; }

unsigned long long current_context_id() {
  std::call_once(g_ctx_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx ||
      g_ctx_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

nvfp4_status_t current_device(DeviceInfo *out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
  DevState &st = g_dev[dev];
  // The status word's address belongs to the context it was looked up in: after a device reset
  // (a new primary context) the module is loaded again, possibly elsewhere, so the cached
  // address is looked up again.  cudaGetDevice above has made the context current.
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || st.ctx.load(std::memory_order_acquire) != ctx) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (ctx == 0 || st.ctx.load(std::memory_order_relaxed) != ctx) {
      st.ok = false;
      st.why[0] = '\0';
      int major = 0, minor = 0, sms = 0;
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      void *status = nullptr;
      cudaError_t se = cudaSuccess;
      if (major == 10 && minor == 3) se = cudaGetSymbolAddress(&status, g_status_word);
      if (major != 10 || minor != 3) {
        snprintf(st.why, sizeof(st.why), "device %d is sm_%d%d; this library runs on sm_103 only",
                 dev, major, minor);
      } else if (se != cudaSuccess) {
        snprintf(st.why, sizeof(st.why), "cudaGetSymbolAddress(status word): %s",
                 cudaGetErrorString(se));
      } else {
        st.ok = true;
        st.info.device = dev;
        st.info.sm_count = sms;
        st.info.status = static_cast<unsigned int *>(status);
      }
      st.ctx.store(ctx, std::memory_order_release);
      if (!st.ok) return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, "%s", st.why);
      *out = st.info;
      return NVFP4_OK;
    }
  }
  if (!st.ok) return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, "%s", st.why);
  *out = st.info;
  return NVFP4_OK;
}

long long wait_limit(uint32_t flags) {
  // clock64 counts SM cycles (at most about 2.1 GHz on this part)
  return (flags & NVFP4_FLAG_DEBUG_TIMEOUT) ? 40000000LL : 20000000000LL;
}

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime (no -lcuda needed).
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

nvfp4_status_t encode_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes,
                                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                                 uint32_t box_rows, bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (!encode) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llu x %llu bytes",
                static_cast<int>(r), static_cast<unsigned long long>(rows),
                static_cast<unsigned long long>(inner_bytes));
  return NVFP4_OK;
}

nvfp4_status_t encode_tmap_stages_u8(CUtensorMap *map, const void *base, uint64_t k_bytes, uint64_t rows,
                                     uint32_t box_rows, uint32_t box_stages) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (!encode) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  if (k_bytes % 128 != 0) return fail(NVFP4_ERR_INVALID_ARG, "stage view needs K %% 256 == 0");
  cuuint64_t dims[3] = {128, rows, k_bytes / 128};
  cuuint64_t strides[2] = {k_bytes, 128};
  cuuint32_t box[3] = {128, box_rows, box_stages};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (stage view) failed (%d) for %llu x %llu bytes",
                static_cast<int>(r), static_cast<unsigned long long>(rows), static_cast<unsigned long long>(k_bytes));
  return NVFP4_OK;
}

int resident_blocks(const void *fn, int threads) {
  struct Entry {
    const void *fn;
    int threads, blocks;
  };
  static Entry cache[64];
  static int n = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].fn == fn && cache[i].threads == threads) return cache[i].blocks;
  }
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, threads, 0) != cudaSuccess || blocks < 1) {
    cudaGetLastError();  // consume the error so later calls do not see it
    return 1;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (n < 64) cache[n++] = Entry{fn, threads, blocks};
  return blocks;
}

nvfp4_status_t allow_smem(const void *fn, int bytes, int device) {
  const unsigned long long ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_smem_n; ++i)
      if (g_smem[i].fn == fn && g_smem[i].device == device && g_smem[i].ctx == ctx && g_smem[i].bytes >= bytes)
        return NVFP4_OK;
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();  // consume the error this call raised so later calls do not see it
    return fail(NVFP4_ERR_CUDA, "cudaFuncSetAttribute(smem=%d): %s", bytes, cudaGetErrorString(e));
  }
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_smem_n; ++i)
    if (g_smem[i].fn == fn && g_smem[i].device == device) {  // a newer context or a larger size
      g_smem[i] = SmemEntry{fn, device, ctx, bytes};
      return NVFP4_OK;
    }
  if (g_smem_n < 256) g_smem[g_smem_n++] = SmemEntry{fn, device, ctx, bytes};
  return NVFP4_OK;
}

nvfp4_status_t check_launch(cudaError_t e, const char *what) {
  if (e != cudaSuccess) {
    cudaGetLastError();  // a failed launch also records itself as the runtime's last error
    return fail(NVFP4_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  }
  return NVFP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" const char *nvfp4_last_error(void) { return t_msg; }

extern "C" size_t nvfp4_sf_bytes(int64_t rows, int64_t k, int sf_vec) {
  if (rows < 0 || k < 0 || (sf_vec != 16 && sf_vec != 32) || k % sf_vec) return 0;
  return static_cast<size_t>(round_up(rows, 128) * round_up(k / sf_vec, 4));
}

extern "C" size_t mxfp4_grouped_sf_bytes(int64_t total_rows, int num_experts, int64_t k) {
  if (total_rows < 0 || num_experts < 1 || k < 0 || k % 32) return 0;
  return static_cast<size_t>((round_up(total_rows, 128) + 128 * static_cast<int64_t>(num_experts)) *
                             round_up(k / 32, 4));
}

extern "C" nvfp4_status_t nvfp4_check_status(nvfp4_stream_t stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  unsigned int word = 0;
  e = cudaMemcpy(&word, dev.status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (word) {
    const unsigned int zero = 0;
    cudaMemcpy(dev.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (word & 2u)
      return fail(NVFP4_ERR_INVALID_ARG, "a grouped kernel found malformed row offsets and did no work (status 0x%x)", word);
    if (word & 8u)
      return fail(NVFP4_ERR_INVALID_ARG, "a MoE step found an expert id or row index out of range and skipped it (status 0x%x)", word);
    if (word & 4u)
      return fail(NVFP4_ERR_CUDA, "internal: a split tile had more partials than the fix-up buffer holds (status 0x%x)", word);
    static const char *const kSites[7] = {"load/free-slot", "mma/accumulator", "mma/stage", "mma/scales",
                                          "scales/slot", "scales/stage", "epilogue/accumulator"};
    char sites[160] = "";
    for (int i = 0; i < 7; ++i)
      if (word & (1u << (8 + i))) {
        strncat(sites, sites[0] ? ", " : "", sizeof(sites) - strlen(sites) - 1);
        strncat(sites, kSites[i], sizeof(sites) - strlen(sites) - 1);
      }
    return fail(NVFP4_ERR_TIMEOUT, "a kernel gave up a bounded pipeline wait (status 0x%x; waits: %s)", word, sites);
  }
  return NVFP4_OK;
}
