// NVFP4 dense GEMM entry point and its M-based tile selector.
//
// Selector (the role of "SM103 Dispatch" in vLLM fork compare view "add pdl",
// nvfp4_scaled_mm_kernels.cu, which buckets M into [1,16], (16,256], (256,inf); and of the
// narrow output tiles FlashInfer PR 4865's "Reviewer Notes" credit for small-M speed):
//   M <= 256  swap A and B: the weight's rows fill the 128-row MMA slot and the tokens the
//             N slot (N = 32, 64, 128 or 256, the smallest that holds M), so no MMA row is
//             wasted on padding; K is split over a thread-block cluster of up to 8 CTAs until the
//             grid covers the SMs, and the partial tiles are reduced through distributed
//             shared memory (decode shapes are weight-streaming, so every SM must pull).
//   M >  256  128 x 256 tiles (128 x 128 when N is not a multiple of 256... or fewer tiles
//             than SMs), persistent over the SMs, double-buffered accumulators where tensor
//             memory allows.
#include "gemm.cuh"
#include "host.h"

namespace nvfp4 {
namespace {

struct Plan {
  int swap, bn, splits, stages, ctas, m_tiles, n_tiles, k_tiles;
};

Plan select_plan(int64_t m, int64_t n, int64_t k, int sm_count) {
  Plan pl{};
  pl.k_tiles = static_cast<int>(ceil_div(k, 256));
  if (m <= 256) {
    pl.swap = 1;
    pl.bn = m <= 32 ? 32 : m <= 64 ? 64 : m <= 128 ? 128 : 256;
    pl.m_tiles = static_cast<int>(ceil_div(n, 128));  // weight rows
    pl.n_tiles = static_cast<int>(ceil_div(m, pl.bn));
    const int tiles = pl.m_tiles * pl.n_tiles;
    int s = sm_count / (tiles > 0 ? tiles : 1);
    s = s < 1 ? 1 : (s > 8 ? 8 : s);
    if (s > pl.k_tiles) s = pl.k_tiles;
    pl.splits = s;
    pl.ctas = tiles * s;
  } else {
    pl.swap = 0;
    pl.bn = (n % 256 == 0 && ceil_div(m, 128) * (n / 256) >= sm_count) ? 256 : 128;
    pl.m_tiles = static_cast<int>(ceil_div(m, 128));
    pl.n_tiles = static_cast<int>(ceil_div(n, pl.bn));
    pl.splits = 1;
    const int tiles = pl.m_tiles * pl.n_tiles;
    pl.ctas = tiles < sm_count ? tiles : sm_count;
  }
  // Rings as deep as shared memory allows: a swap-AB CTA then has its whole K slice in flight
  // from the start (the decode GEMM is bound by load latency, not by shared memory).
  switch (pl.bn) {
    case 32: pl.stages = 8; break;
    case 64: pl.stages = 7; break;
    case 128: pl.stages = 6; break;
    default: pl.stages = 4; break;
  }
  return pl;
}

template <int BN, int STAGES, bool MULTI_TILE>
nvfp4_status_t run(const Plan &pl, const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args,
                   const DeviceInfo &dev, uint32_t flags, cudaStream_t s) {
  using C = GemmCfg<BN, STAGES, false, MULTI_TILE>;
  auto kern = bs_gemm_kernel<C, false>;
  nvfp4_status_t st = allow_smem(reinterpret_cast<const void *>(kern), C::smem_bytes(false), dev.device);
  if (st != NVFP4_OK) return st;
  cudaError_t e = launch(kern, dim3(pl.ctas), dim3(C::THREADS), C::smem_bytes(false), s,
                         (flags & NVFP4_FLAG_PDL) != 0, pl.splits, ta, tb, args);
  return check_launch(e, "nvfp4_gemm");
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status_t nvfp4_gemm_plan(int64_t m, int64_t n, int64_t k, nvfp4_gemm_plan_t *plan) {
  clear_error();
  if (!plan || m < 0 || n <= 0 || k <= 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gemm_plan: bad arguments");
  int sms = 152;
  DeviceInfo dev;
  int cur = -1;
  if (cudaGetDevice(&cur) == cudaSuccess && current_device(&dev) == NVFP4_OK) sms = dev.sm_count;
  clear_error();
  const Plan pl = select_plan(m, n, k, sms);
  plan->swap_ab = pl.swap;
  plan->tile_m = 128;
  plan->tile_n = pl.bn;
  plan->splits = pl.splits;
  plan->stages = pl.stages;
  plan->ctas = pl.ctas;
  return NVFP4_OK;
}

extern "C" nvfp4_status_t nvfp4_gemm(const uint8_t *a, const uint8_t *sfa, const uint8_t *b,
                                     const uint8_t *sfb, const float *alpha, void *d, int64_t m,
                                     int64_t n, int64_t k, uint32_t flags, nvfp4_stream_t stream) {
  clear_error();
  if (m < 0 || n <= 0 || k <= 0 || m >= (1LL << 31) || n >= (1LL << 31) || k >= (1LL << 31))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gemm: m=%lld n=%lld k=%lld", (long long)m, (long long)n, (long long)k);
  if (k % 32 || n % 32)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "nvfp4_gemm: need k %% 32 == 0 and n %% 32 == 0 (k=%lld n=%lld)", (long long)k, (long long)n);
  if (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT | NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gemm: unknown flags 0x%x", flags);
  if (m == 0) return NVFP4_OK;
  if (!a || !sfa || !b || !sfb || !alpha || !d) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gemm: null pointer");
  if (!aligned(a, 32) || !aligned(b, 32) || !aligned(d, 32) || !aligned(sfa, 16) || !aligned(sfb, 16) || !aligned(alpha, 4))
    return fail(NVFP4_ERR_MISALIGNED, "nvfp4_gemm: a, b, d need 32-B and sfa, sfb 16-B alignment");
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  const Plan pl = select_plan(m, n, k, dev.sm_count);
  // Kernel operand A fills the 128-row MMA slot; with swap it is the weight B.
  const uint8_t *opa = pl.swap ? b : a, *opb = pl.swap ? a : b;
  const uint8_t *sfopa = pl.swap ? sfb : sfa, *sfopb = pl.swap ? sfa : sfb;
  const int64_t rows_a = pl.swap ? n : m, rows_b = pl.swap ? m : n;
  CUtensorMap ta, tb;
  st = encode_tmap_2d_u8(&ta, opa, k / 2, rows_a, k / 2, 128, 128, true);
  if (st != NVFP4_OK) return st;
  st = encode_tmap_2d_u8(&tb, opb, k / 2, rows_b, k / 2, 128, pl.bn, true);
  if (st != NVFP4_OK) return st;

  GemmArgs args{};
  args.sfa = sfopa;
  args.sfb = sfopb;
  args.alpha = alpha;
  args.d = static_cast<__nv_bfloat16 *>(d);
  args.ldd = n;
  args.m = static_cast<int>(rows_a);
  args.n = static_cast<int>(rows_b);
  args.k = static_cast<int>(k);
  args.swap = pl.swap;
  // b (the weight) may be read before the PDL wait (header contract); only worth it under PDL
  args.weight_operand = (flags & NVFP4_FLAG_PDL) ? (pl.swap ? 1 : 2) : 0;
  args.m_tiles = pl.m_tiles;
  args.n_tiles = pl.n_tiles;
  args.k_tiles = pl.k_tiles;
  args.splits = pl.splits;
  args.sf_chunks = static_cast<int>(round_up(k / 16, 4) / 4);
  args.status = dev.status;
  args.wait_limit = wait_limit(flags);
  args.debug_skip_first_load = (flags & NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD) && (flags & NVFP4_FLAG_DEBUG_TIMEOUT);

  cudaStream_t s = (cudaStream_t)stream;
  switch (pl.bn) {
    // swap-AB CTAs own one tile each (single accumulator); large-M CTAs walk tiles persistently
    case 32: return run<32, 8, false>(pl, ta, tb, args, dev, flags, s);
    case 64: return run<64, 7, false>(pl, ta, tb, args, dev, flags, s);
    case 128:
      return pl.swap ? run<128, 6, false>(pl, ta, tb, args, dev, flags, s) : run<128, 6, true>(pl, ta, tb, args, dev, flags, s);
    default:
      return pl.swap ? run<256, 4, false>(pl, ta, tb, args, dev, flags, s) : run<256, 4, true>(pl, ta, tb, args, dev, flags, s);
  }
}
