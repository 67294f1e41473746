// Row-major scale matrix <-> 128x4 swizzled scale layout (weight-load time, not per token).
// Layout: vLLM fork compare view "add pdl", nvfp4_quant_kernels.cu, "Scale factor layout
// conversion: SM100 <-> SM103" (SM100 in-tile offset) and nvfp4_utils.cuh (512-byte tiles of
// 128 rows x 4 scale columns); nvfp4_utils.py swizzle_blockscale pads to (128, 4) with zeros.
#include "host.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

__device__ __forceinline__ int64_t swz_offset(int64_t r, int64_t j, int64_t cp) {
  return ((r >> 7) * (cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// One thread per position of the padded [rp, cp] matrix (writes every destination byte).
__global__ void __launch_bounds__(256) swizzle_kernel(const uint8_t *__restrict__ src,
                                                      uint8_t *__restrict__ dst, int64_t rows,
                                                      int64_t cols, int64_t cp, int64_t total) {
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int64_t r = idx / cp, j = idx - (idx / cp) * cp;
    dst[swz_offset(r, j, cp)] = (r < rows && j < cols) ? src[r * cols + j] : 0;
  }
}

// One thread per element of the unpadded [rows, cols] destination.
__global__ void __launch_bounds__(256) unswizzle_kernel(const uint8_t *__restrict__ src,
                                                        uint8_t *__restrict__ dst, int64_t rows,
                                                        int64_t cols, int64_t cp) {
  pdl_wait();
  const int64_t total = rows * cols;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int64_t r = idx / cols, j = idx - (idx / cols) * cols;
    dst[idx] = src[swz_offset(r, j, cp)];
  }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status_t sf_swizzle(const uint8_t *src, uint8_t *dst, int64_t rows, int64_t cols,
                                     int to_swizzled, nvfp4_stream_t stream) {
  clear_error();
  if (rows < 0 || cols < 0) return fail(NVFP4_ERR_INVALID_ARG, "sf_swizzle: rows=%lld cols=%lld", (long long)rows, (long long)cols);
  if (to_swizzled != 0 && to_swizzled != 1) return fail(NVFP4_ERR_INVALID_ARG, "sf_swizzle: to_swizzled=%d", to_swizzled);
  if (rows == 0 || cols == 0) {
    if (to_swizzled && rows > 0 && cols == 0) { /* nothing: zero scale columns pad to zero bytes */ }
    return NVFP4_OK;
  }
  if (!src || !dst) return fail(NVFP4_ERR_INVALID_ARG, "sf_swizzle: null pointer");
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t cp = round_up(cols, 4);
  const int64_t total = to_swizzled ? round_up(rows, 128) * cp : rows * cols;
  int64_t blocks = ceil_div(total, 256);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
  const int grid = static_cast<int>(blocks < cap ? blocks : cap);
  cudaError_t e;
  if (to_swizzled)
    e = launch(swizzle_kernel, dim3(grid), dim3(256), 0, (cudaStream_t)stream, false, 1, src, dst,
               rows, cols, cp, total);
  else
    e = launch(unswizzle_kernel, dim3(grid), dim3(256), 0, (cudaStream_t)stream, false, 1, src, dst,
               rows, cols, cp);
  return check_launch(e, "sf_swizzle");
}
