// bf16 -> NVFP4 and bf16 -> MXFP4 quantisers (bandwidth-bound, CUDA cores).
//
// NVFP4 follows vLLM fork compare view "add pdl", nvfp4_quant_kernels.cu, "SM103 (B300)
// activation quantization kernel": one fp32 global scale, one e4m3 scale per 16 elements of a
// row written straight into the 128x4 swizzled layout, packed e2m1 output, padded scale rows and
// columns written as if quantised from zeros.  MXFP4 ("e8m0 scale per 32", vLLM PR 51158,
// "Changes", mxfp4_experts_quant.cu) uses a power-of-two scale rounded up and, for MoE input,
// one zero-padded 128-row scale block per expert.
//
// Work mapping: one thread per (scale row, scale column) position of the padded scale matrix.
// A warp covers 32 consecutive positions of one scale row, so its data loads are contiguous;
// four neighbouring threads gather their scale bytes into one 32-bit store (the 4 scale
// columns of a 512-byte tile row are adjacent bytes).
#include <cuda_bf16.h>

#include "host.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t j, int64_t cp) {
  return ((r >> 7) * (cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}
// The SM103 layout (same tiles; inside a tile row m = m4b + 4*m4a + 16*m8 sits at
// m8*16 + m4a*128 + m4b*4): vLLM fork compare view "add pdl", nvfp4_utils.cuh, SM103 swizzled
// SF offset, written by that page's SM103 quantisation kernel.
__device__ __forceinline__ int64_t sf_offset_sm103(int64_t r, int64_t j, int64_t cp) {
  const int64_t m = r & 127;
  return ((r >> 7) * (cp >> 2) + (j >> 2)) * 512 + ((m >> 4) & 7) * 16 + ((m >> 2) & 3) * 128 + (m & 3) * 4 + (j & 3);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// 4 lanes (j % 4 == 0 .. 3) -> one little-endian 32-bit word held by the first of them.
__device__ __forceinline__ uint32_t gather4(uint32_t code) {
  const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, code, 1);
  const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, code, 2);
  const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, code, 3);
  return code | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

// total = round_up(m,128) * cp, a multiple of 512, so every warp runs the same trip count.
// SM103: scales in the SM103 layout instead of the 128x4 one.  I: the position type (32-bit
// when total plus one grid stride < 2^31: its division is several times cheaper than the
// 64-bit one).
template <bool SM103, typename I>
__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const __nv_bfloat16 *__restrict__ x,
                                                          int64_t m, int64_t kb, int64_t ldx,
                                                          const float *__restrict__ gs_ptr,
                                                          uint8_t *__restrict__ q,
                                                          uint8_t *__restrict__ sf, int64_t total_,
                                                          int64_t cp_) {
  const I total = static_cast<I>(total_), cp = static_cast<I>(cp_);
  // Let the next kernel launch at once (it waits for this grid's completion before it reads
  // our outputs), then wait for our own predecessor before reading x.
  pdl_trigger();
  pdl_wait();
  const float gs = __ldg(gs_ptr);
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  I idx = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x;
  // (row, scale column) of idx, stepped by the grid stride instead of a division per position
  I r = idx / cp, j = idx - (idx / cp) * cp;
  const I dr = stride / cp, dj = stride - dr * cp;
  for (; idx < total; idx += stride, r += dr, j += dj) {
    if (j >= cp) {
      j -= cp;
      ++r;
    }
    uint32_t code = 0;
    if (r < m && j < kb) {
      const uint4 *src = reinterpret_cast<const uint4 *>(x + r * ldx + j * 16);
      float f[16];
      bf16x16_to_f32(__ldg(src), __ldg(src + 1), f);
      *reinterpret_cast<uint2 *>(q + r * (kb * 8) + j * 8) = nvfp4_block16(f, gs, code);
    }
    const uint32_t word = gather4(code);
    if ((j & 3) == 0) *reinterpret_cast<uint32_t *>(sf + (SM103 ? sf_offset_sm103(r, j, cp) : sf_offset(r, j, cp))) = word;
  }
}

constexpr int kMaxExperts = 1024;
// 128-row scale blocks whose owning expert the grouped quantiser tabulates in shared memory
// (8 KB; 512K scale rows); beyond that it searches the scale-row prefix per position.
constexpr int kExpertBlockTable = 4096;

// Scale rows of the (optionally expert-grouped) MXFP4 layout: expert e owns scale rows
// sfr[e] .. sfr[e+1]-1, sfr[e+1] - sfr[e] = round_up(M_e, 128).
template <typename I>
__global__ void __launch_bounds__(256) mxfp4_quant_kernel(const __nv_bfloat16 *__restrict__ x,
                                                          int64_t t, int64_t kb, int64_t ldx,
                                                          const int64_t *__restrict__ row_offsets,
                                                          int experts, uint8_t *__restrict__ q,
                                                          uint8_t *__restrict__ sf,
                                                          int64_t cap_rows, int64_t cp) {
  __shared__ int64_t s_ro[kMaxExperts + 1];
  __shared__ int64_t s_sfr[kMaxExperts + 1];
  __shared__ uint16_t s_blk[kExpertBlockTable];
  // Let the next kernel launch at once (it waits for this grid's completion before it reads
  // our outputs), then wait for our own predecessor before reading x.
  pdl_trigger();
  pdl_wait();
  if (row_offsets == nullptr) {
    if (threadIdx.x == 0) {
      s_ro[0] = 0;
      s_ro[1] = t;
      s_sfr[0] = 0;
      s_sfr[1] = (t + 127) / 128 * 128;
    }
    experts = 1;
  } else {
    for (int e = threadIdx.x; e <= experts; e += blockDim.x) s_ro[e] = row_offsets[e];
    __syncthreads();
    if (threadIdx.x < 32) {  // scale-row prefix: a warp scan over the experts, 32 at a time
      const int lane = threadIdx.x;
      int64_t carry = 0;
      for (int base = 0; base < experts; base += 32) {
        const int e = base + lane;
        int64_t v = 0;
        if (e < experts) {
          const int64_t cnt = s_ro[e + 1] - s_ro[e];
          v = (cnt > 0 ? cnt + 127 : 0) / 128 * 128;
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t n = __shfl_up_sync(0xFFFFFFFFu, v, o);
          if (lane >= o) v += n;
        }
        if (e < experts) s_sfr[e + 1] = carry + v;
        carry += __shfl_sync(0xFFFFFFFFu, v, 31);
      }
      if (lane == 0) s_sfr[0] = 0;
    }
  }
  __syncthreads();
  // Every expert owns whole 128-row blocks of scale rows: with at most kExpertBlockTable of them
  // a table filled by one search per entry gives a position's expert in one lookup.
  const int64_t nblk = s_sfr[experts] >> 7;
  const bool table = experts > 1 && nblk >= 0 && nblk <= kExpertBlockTable;
  if (table) {
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
      const int64_t row0 = static_cast<int64_t>(b) << 7;
      int lo = 0, hi = experts - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_sfr[mid] <= row0) lo = mid;
        else hi = mid - 1;
      }
      s_blk[b] = static_cast<uint16_t>(lo);
    }
    __syncthreads();
  }
  const int64_t rows = s_sfr[experts] < cap_rows ? s_sfr[experts] : cap_rows;
  const I total = static_cast<I>(rows > 0 ? rows * cp : 0), cpi = static_cast<I>(cp);
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  I idx = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x;
  // (scale row, scale column) of idx, stepped by the grid stride instead of a division each
  I s = idx / cpi, j = idx - (idx / cpi) * cpi;
  const I ds = stride / cpi, dj = stride - ds * cpi;
  for (; idx < total; idx += stride, s += ds, j += dj) {
    if (j >= cpi) {
      j -= cpi;
      ++s;
    }
    int lo;  // expert owning scale row s: the largest e with s_sfr[e] <= s
    if (table) {
      lo = s_blk[s >> 7];  // s < rows <= 128 * nblk; every entry holds an expert in range
    } else {
      lo = 0;
      int hi = experts - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_sfr[mid] <= s) lo = mid;
        else hi = mid - 1;
      }
    }
    const int64_t local = s - s_sfr[lo];
    const int64_t r = s_ro[lo] + local;
    uint32_t code = 0;
    if (local < s_ro[lo + 1] - s_ro[lo] && r >= 0 && r < t && j < kb) {
      const uint4 *src = reinterpret_cast<const uint4 *>(x + r * ldx + j * 32);
      float f[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) bf16x8_to_f32(__ldg(src + i), f + 8 * i);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
      code = ue8m0_code_up(__fdiv_rn(amax, 6.0f));
      const float inv = ue8m0_inverse(code);
      uint4 out;
      uint32_t *o = &out.x;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(f[8 * g + i], inv);
        o[g] = e2m1x8(y);
      }
      *reinterpret_cast<uint4 *>(q + r * (kb * 16) + j * 16) = out;
    }
    const uint32_t word = gather4(code);
    if ((j & 3) == 0) *reinterpret_cast<uint32_t *>(sf + sf_offset(s, j, cp)) = word;
  }
}

// At most the blocks of `kern` resident on every SM at once: a block walks its share of the
// positions, and its prologue runs once.
int quant_grid(int64_t total_threads, int sm_count, const void *kern) {
  const int64_t blocks = ceil_div(total_threads, 256);
  const int64_t cap = static_cast<int64_t>(sm_count) * resident_blocks(kern, 256);
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status_t nvfp4_quantize(const void *x, int64_t m, int64_t k, int64_t ldx,
                                         const float *gs, uint8_t *q, uint8_t *sf, uint32_t flags,
                                         nvfp4_stream_t stream) {
  clear_error();
  if (m < 0 || k <= 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize: m=%lld k=%lld", (long long)m, (long long)k);
  if (k % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "nvfp4_quantize: k=%lld is not a multiple of 16", (long long)k);
  if (ldx < k || ldx % 8) return fail(NVFP4_ERR_MISALIGNED, "nvfp4_quantize: ldx=%lld (need ldx >= k, ldx %% 8 == 0)", (long long)ldx);
  if (m == 0) return NVFP4_OK;
  if (!x || !gs || !q || !sf) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize: null pointer");
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(sf, 16) || !aligned(gs, 4))
    return fail(NVFP4_ERR_MISALIGNED, "nvfp4_quantize: x needs 16-B, q 8-B, sf 16-B, gs 4-B alignment");
  if (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT | NVFP4_FLAG_SF_SM103))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize: unknown flags 0x%x", flags);
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t cp = round_up(k / 16, 4);
  const int64_t total = round_up(m, 128) * cp;
  const bool sm103 = (flags & NVFP4_FLAG_SF_SM103) != 0;
  auto kern = sm103 ? nvfp4_quant_kernel<true, int> : nvfp4_quant_kernel<false, int>;
  int grid = quant_grid(total, dev.sm_count, reinterpret_cast<const void *>(kern));
  if (!fits_i32_loop(total, static_cast<int64_t>(grid) * 256)) {
    kern = sm103 ? nvfp4_quant_kernel<true, int64_t> : nvfp4_quant_kernel<false, int64_t>;
    grid = quant_grid(total, dev.sm_count, reinterpret_cast<const void *>(kern));
  }
  cudaError_t e = launch(kern, dim3(grid), dim3(256), 0, (cudaStream_t)stream,
                         (flags & NVFP4_FLAG_PDL) != 0, 1, (const __nv_bfloat16 *)x, m, k / 16,
                         ldx, gs, q, sf, total, cp);
  return check_launch(e, "nvfp4_quantize");
}

extern "C" nvfp4_status_t mxfp4_quantize(const void *x, int64_t t, int64_t k, int64_t ldx,
                                         const int64_t *row_offsets, int num_experts, uint8_t *q,
                                         uint8_t *sf, size_t sf_bytes, uint32_t flags,
                                         nvfp4_stream_t stream) {
  clear_error();
  if (t < 0 || k <= 0) return fail(NVFP4_ERR_INVALID_ARG, "mxfp4_quantize: t=%lld k=%lld", (long long)t, (long long)k);
  if (k % 32) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "mxfp4_quantize: k=%lld is not a multiple of 32", (long long)k);
  if (ldx < k || ldx % 8) return fail(NVFP4_ERR_MISALIGNED, "mxfp4_quantize: ldx=%lld (need ldx >= k, ldx %% 8 == 0)", (long long)ldx);
  if (row_offsets && (num_experts < 1 || num_experts > kMaxExperts))
    return fail(NVFP4_ERR_INVALID_ARG, "mxfp4_quantize: num_experts=%d (1..%d)", num_experts, kMaxExperts);
  const size_t need = row_offsets ? mxfp4_grouped_sf_bytes(t, num_experts, k) : nvfp4_sf_bytes(t, k, 32);
  if (sf_bytes < need)
    return fail(NVFP4_ERR_INVALID_ARG, "mxfp4_quantize: sf_bytes=%zu < %zu", sf_bytes, need);
  if (t == 0) return NVFP4_OK;
  if (!x || !q || !sf) return fail(NVFP4_ERR_INVALID_ARG, "mxfp4_quantize: null pointer");
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(sf, 16) || (row_offsets && !aligned(row_offsets, 8)))
    return fail(NVFP4_ERR_MISALIGNED, "mxfp4_quantize: x, q, sf need 16-B and row_offsets 8-B alignment");
  if (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT))
    return fail(NVFP4_ERR_INVALID_ARG, "mxfp4_quantize: unknown flags 0x%x", flags);
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t cp = round_up(k / 32, 4);
  const int64_t cap_rows = static_cast<int64_t>(sf_bytes) / cp / 128 * 128;
  const int64_t total = (row_offsets ? round_up(t, 128) + 128LL * num_experts : round_up(t, 128)) * cp;
  // (the kernel's positions cover at most `total`: 32-bit when that plus one grid stride fits)
  auto kern = mxfp4_quant_kernel<int>;
  int grid = quant_grid(total, dev.sm_count, reinterpret_cast<const void *>(kern));
  if (!fits_i32_loop(total, static_cast<int64_t>(grid) * 256)) {
    kern = mxfp4_quant_kernel<int64_t>;
    grid = quant_grid(total, dev.sm_count, reinterpret_cast<const void *>(kern));
  }
  cudaError_t e = launch(kern, dim3(grid), dim3(256), 0, (cudaStream_t)stream,
                         (flags & NVFP4_FLAG_PDL) != 0, 1, (const __nv_bfloat16 *)x, t, k / 32,
                         ldx, row_offsets, row_offsets ? num_experts : 1, q, sf, cap_rows, cp);
  return check_launch(e, "mxfp4_quantize");
}
