// Row-major scale matrix <-> 128x4 swizzled scale layout, and the SM100 <-> SM103 re-arrangement
// of a swizzled buffer (weight-load time, not per token).
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

// SM100 <-> SM103 layout of a swizzled scale buffer (vLLM fork compare view "add pdl",
// nvfp4_quant_kernels.cu, "Scale factor layout conversion: SM100 <-> SM103").  Both layouts
// keep the 4 scale columns of a tile row as 4 adjacent bytes, so a tile is 128 32-bit words,
// word w of a row m at:
//   SM100: w = (m % 32) * 4 + (m / 32) % 4
//   SM103: w = ((m / 16) % 8) * 4 + ((m / 4) % 4) * 32 + m % 4
// One warp per 512-byte tile: it loads the tile with 16-byte loads into shared memory, then each
// lane assembles 16 bytes of the destination tile from the words they come from.
__device__ __forceinline__ int word_sm100(int m) { return (m & 31) * 4 + ((m >> 5) & 3); }
__device__ __forceinline__ int word_sm103(int m) { return ((m >> 4) & 7) * 4 + ((m >> 2) & 3) * 32 + (m & 3); }
__device__ __forceinline__ int row_of_sm100_word(int w) { return (w >> 2) + 32 * (w & 3); }
__device__ __forceinline__ int row_of_sm103_word(int w) { return (w & 3) + 4 * ((w >> 5) & 3) + 16 * ((w >> 2) & 7); }

constexpr int kConvWarps = 8;

__global__ void __launch_bounds__(kConvWarps * 32) convert_layout_kernel(const uint8_t *__restrict__ src,
                                                                          uint8_t *__restrict__ dst,
                                                                          int64_t tiles, int to_sm103) {
  __shared__ __align__(16) uint32_t buf[kConvWarps][128];
  pdl_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kConvWarps + warp; t < tiles;
       t += static_cast<int64_t>(gridDim.x) * kConvWarps) {
    const uint4 v = *reinterpret_cast<const uint4 *>(src + t * 512 + lane * 16);
    *reinterpret_cast<uint4 *>(&buf[warp][lane * 4]) = v;
    __syncwarp();
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int dw = lane * 4 + i;  // destination word
      const int sw = to_sm103 ? word_sm100(row_of_sm103_word(dw)) : word_sm103(row_of_sm100_word(dw));
      w[i] = buf[warp][sw];
    }
    *reinterpret_cast<uint4 *>(dst + t * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    __syncwarp();  // the next tile overwrites buf
  }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status_t nvfp4_sf_convert_layout(const uint8_t *src, uint8_t *dst, int64_t rows, int64_t cols,
                                                  int to_sm103, nvfp4_stream_t stream) {
  clear_error();
  if (rows < 0 || cols < 0 || rows >= (1LL << 40) || cols >= (1LL << 31))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_sf_convert_layout: rows=%lld cols=%lld", (long long)rows, (long long)cols);
  if (to_sm103 != 0 && to_sm103 != 1)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_sf_convert_layout: to_sm103=%d", to_sm103);
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (!src || !dst) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_sf_convert_layout: null pointer");
  if (!aligned(src, 16) || !aligned(dst, 16))
    return fail(NVFP4_ERR_MISALIGNED, "nvfp4_sf_convert_layout: src and dst need 16-B alignment");
  const int64_t bytes = round_up(rows, 128) * round_up(cols, 4);
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + static_cast<uintptr_t>(bytes) && d0 < s0 + static_cast<uintptr_t>(bytes))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_sf_convert_layout: src and dst overlap");
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t tiles = bytes / 512;
  const int64_t blocks = ceil_div(tiles, kConvWarps);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
  const int grid = static_cast<int>(blocks < cap ? blocks : cap);
  cudaError_t e = launch(convert_layout_kernel, dim3(grid), dim3(kConvWarps * 32), 0, (cudaStream_t)stream, false, 1,
                         src, dst, tiles, to_sm103);
  return check_launch(e, "nvfp4_sf_convert_layout");
}

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
