// Host-side helpers shared by the entry points: error reporting, device checks, launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <utility>

#include "nvfp4.h"

namespace nvfp4 {

// Records a formatted message for nvfp4_last_error() and returns `code`.
nvfp4_status_t fail(nvfp4_status_t code, const char *fmt, ...);
void clear_error();

struct DeviceInfo {
  int device;
  int sm_count;
  unsigned int *status;  // device status word (address of a __device__ variable)
};
// Checks that the current device is sm_103 and returns its properties, cached per device for
// as long as its context lives (a device reset makes a new context: they are looked up again).
nvfp4_status_t current_device(DeviceInfo *out);

// Unique id of the calling thread's current CUDA context (cuCtxGetId); 0 if there is none.
unsigned long long current_context_id();

// Bytes of the stream-K workspace: one arrival counter per split tile (rounded up to 256 bytes),
// then two fp32 partial-tile slots of 128 x bn per CTA.
constexpr size_t stream_k_workspace_bytes(int sk_tiles, int ctas, int bn) {
  return (static_cast<size_t>(sk_tiles) * 4 + 255) / 256 * 256 + static_cast<size_t>(ctas) * 2 * 128 * bn * 4;
}

// Wait limit (SM clock cycles) for the bounded pipeline waits.
long long wait_limit(uint32_t flags);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda needed).
nvfp4_status_t encode_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes,
                                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                                 uint32_t box_rows, bool swizzle128);

// 3-D view of a K-major FP4 operand [rows, K/2 bytes] for loading a run of K stages in one copy:
// dims {128 bytes, rows, K/256 stages}, strides {row stride, 128}, box {128, box_rows, box_stages},
// 128-byte swizzle.  The box lands as box_stages consecutive (box_rows x 128-byte) tiles.
// Needs K % 256 == 0 (otherwise the last stage would run into the next row).
nvfp4_status_t encode_tmap_stages_u8(CUtensorMap *map, const void *base, uint64_t k_bytes, uint64_t rows,
                                     uint32_t box_rows, uint32_t box_stages);

// Raises the dynamic shared-memory limit of `fn` on the current device (once per device).
nvfp4_status_t allow_smem(const void *fn, int bytes, int device);

// Blocks of `threads` threads (no dynamic shared memory) of kernel `fn` resident on one SM, by
// the occupancy calculator; cached per kernel, since it depends only on the compiled code.
// 1 if the query fails.
int resident_blocks(const void *fn, int threads);

inline bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
inline int64_t round_up(int64_t x, int64_t y) { return (x + y - 1) / y * y; }
inline int64_t ceil_div(int64_t x, int64_t y) { return (x + y - 1) / y; }
// A grid-stride loop over `total` positions may count in 32-bit signed integers only when the
// last position plus one stride still fits: then no step wraps.
inline bool fits_i32_loop(int64_t total, int64_t grid_threads) { return total + grid_threads < (1LL << 31); }

// cudaLaunchKernelEx with optional programmatic-dependent-launch and cluster attributes.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   bool pdl, int cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  unsigned n = 0;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

nvfp4_status_t check_launch(cudaError_t e, const char *what);

}  // namespace nvfp4
