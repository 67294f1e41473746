// MXFP4 and NVFP4 grouped (MoE expert) GEMM entry points.
//
// vLLM PR 51158 ("Enable CUTLASS MXFP4 W4A4 MoE on SM12x", "Changes"): a grouped GEMM over
// experts with e2m1 data and ue8m0 scales per 32 that share the block-scaled 128x4 layout;
// vLLM fork compare view "add pdl", ops.h passes expert row offsets as arguments.
// Here one persistent kernel walks the (expert, m-tile, n-tile) work list that each CTA derives
// in shared memory from the device row offsets; an expert's m-tiles are adjacent in that list
// so concurrently running CTAs share the expert's weight tile through L2.  The NVFP4 variant
// (vLLM fork compare view "add pdl", torch_bindings.cpp, cutlass_fp4_group_mm) takes e4m3 scales
// per 16 and one fp32 alpha per expert (each expert's weight has its own global scale).
#include "gemm.cuh"
#include "host.h"

using namespace nvfp4;

namespace {
constexpr int kGroupedBN = 128;
using GroupedCfg = GemmCfg<kGroupedBN, 6, true>;       // MXFP4: 34 KB stages
// NVFP4: 36 KB stages; expert tables for up to 512 experts leave room for a 6-deep ring
using GroupedCfgNv = GemmCfg<kGroupedBN, 6, false, true, 1, false, 512>;
// NVFP4 with K % 256 == 0: two K steps per 72 KB stage (one 3-D copy per operand), 3 stages
// (an expert tile's K run is short -- 3 steps at K = 768 -- so per-stage costs weigh)
using GroupedCfgNv2 = GemmCfg<kGroupedBN, 3, false, true, 1, false, 512, 2>;
// At most 256 experts (tables leave room for a 4-deep ring): 128 x 256 tiles.  Against 128 x 128
// tiles on two CTAs per SM, an activation tile is read half as often and an MMA does twice the
// work, which measured 3.5-5 % faster at the MoE shapes (MXFP4 gate+up 85.6 -> 82.2 us, down
// 65.0 -> 61.6 us; NVFP4 92.7 -> 88.1 and 68.2 -> 65.5 us); a 3-deep ring was slower than both.
using GroupedCfgWide = GemmCfg<256, 4, true, true, 1, false, 256>;     // MXFP4: 51 KB stages
using GroupedCfgNvWide = GemmCfg<256, 4, false, true, 1, false, 256>;  // NVFP4: 54 KB stages
static_assert(GroupedCfgNv::smem_bytes(true) <= 232448 && GroupedCfg::smem_bytes(true) <= 232448 &&
                  GroupedCfgNv2::smem_bytes(true) <= 232448 && GroupedCfgWide::smem_bytes(true) <= 232448 &&
                  GroupedCfgNvWide::smem_bytes(true) <= 232448,
              "smem");

// Shared by both grouped entry points: argument checks, tensor maps, launch.
template <class C>
nvfp4_status_t grouped_gemm(const char *name, const uint8_t *a, const uint8_t *sfa, const int64_t *row_offsets,
                            int num_experts, const uint8_t *b, const uint8_t *sfb, const float *alpha,
                            bool alpha_per_expert, void *d, int64_t t, int64_t n, int64_t k, uint32_t flags,
                            nvfp4_stream_t stream) {
  clear_error();
  if (t < 0 || n <= 0 || k <= 0 || t >= (1LL << 31) || k >= (1LL << 31))
    return fail(NVFP4_ERR_INVALID_ARG, "%s: t=%lld n=%lld k=%lld", name, (long long)t, (long long)n, (long long)k);
  if (num_experts < 1 || num_experts > C::MAX_EXPERTS)
    return fail(NVFP4_ERR_INVALID_ARG, "%s: num_experts=%d (1..%d)", name, num_experts, C::MAX_EXPERTS);
  if (n * static_cast<int64_t>(num_experts) >= (1LL << 31))
    return fail(NVFP4_ERR_INVALID_ARG, "%s: experts * n too large", name);
  if (k % 32 || n % 32)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: need k %% 32 == 0 and n %% 32 == 0", name);
  if (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT | NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD))
    return fail(NVFP4_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags);
  if (t == 0) return NVFP4_OK;
  if (!a || !sfa || !row_offsets || !b || !sfb || !d) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned(a, 32) || !aligned(b, 32) || !aligned(d, 32) || !aligned(sfa, 16) || !aligned(sfb, 16) ||
      !aligned(row_offsets, 8) || (alpha && !aligned(alpha, 4)))
    return fail(NVFP4_ERR_MISALIGNED, "%s: a, b, d need 32-B, sfa, sfb 16-B, row_offsets 8-B alignment", name);
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  CUtensorMap ta, tb;
  if constexpr (C::KS == 2) {  // stage views: a box is two 256-wide K steps of 128 rows
    st = encode_tmap_stages_u8(&ta, a, k / 2, t, 128, 2);
    if (st == NVFP4_OK) st = encode_tmap_stages_u8(&tb, b, k / 2, n * num_experts, C::BN, 2);
  } else {
    st = encode_tmap_2d_u8(&ta, a, k / 2, t, k / 2, 128, 128, true);
    if (st == NVFP4_OK) st = encode_tmap_2d_u8(&tb, b, k / 2, n * num_experts, k / 2, 128, C::BN, true);
  }
  if (st != NVFP4_OK) return st;

  GemmArgs args{};
  args.sfa = sfa;
  args.sfb = sfb;
  args.alpha = alpha;
  args.alpha_per_expert = alpha_per_expert ? 1 : 0;
  args.d = static_cast<__nv_bfloat16 *>(d);
  args.ldd = n;
  args.m = static_cast<int>(t);
  args.n = static_cast<int>(n);
  args.k = static_cast<int>(k);
  args.swap = 0;
  args.m_tiles = 0;
  args.n_tiles = static_cast<int>(ceil_div(n, C::BN));
  args.k_tiles = static_cast<int>(ceil_div(k, C::KSTAGE));
  args.splits = 1;
  args.sf_chunks = static_cast<int>(round_up(k / C::VEC, 4) / 4);
  args.row_offsets = row_offsets;
  args.experts = num_experts;
  args.sfb_expert_bytes = static_cast<int64_t>(nvfp4_sf_bytes(n, k, C::VEC));
  args.status = dev.status;
  args.wait_limit = wait_limit(flags);
  args.debug_skip_first_load = (flags & NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD) && (flags & NVFP4_FLAG_DEBUG_TIMEOUT);

  // Upper bound of the work list: sum_e ceil(M_e/128) <= ceil(t/128) + experts.
  const int64_t bound = (ceil_div(t, 128) + num_experts) * args.n_tiles;
  if (bound >= (1LL << 31)) return fail(NVFP4_ERR_INVALID_ARG, "%s: problem too large", name);
  args.max_tiles = static_cast<int>(bound);
  auto kern = bs_gemm_kernel<C, true>;
  st = allow_smem(reinterpret_cast<const void *>(kern), C::smem_bytes(true), dev.device);
  if (st != NVFP4_OK) return st;
  const int slots = C::MIN_BLOCKS * dev.sm_count;
  const int grid = static_cast<int>(bound < slots ? bound : slots);
  cudaError_t e = launch(kern, dim3(grid), dim3(C::THREADS), C::smem_bytes(true), (cudaStream_t)stream,
                         (flags & NVFP4_FLAG_PDL) != 0, 1, ta, tb, tb, args);
  return check_launch(e, name);
}
}  // namespace

extern "C" nvfp4_status_t mxfp4_grouped_gemm(const uint8_t *a, const uint8_t *sfa,
                                             const int64_t *row_offsets, int num_experts,
                                             const uint8_t *b, const uint8_t *sfb,
                                             const float *alpha, void *d, int64_t t, int64_t n,
                                             int64_t k, uint32_t flags, nvfp4_stream_t stream) {
  if (num_experts <= GroupedCfgWide::MAX_EXPERTS)
    return grouped_gemm<GroupedCfgWide>("mxfp4_grouped_gemm", a, sfa, row_offsets, num_experts, b, sfb, alpha, false,
                                       d, t, n, k, flags, stream);
  return grouped_gemm<GroupedCfg>("mxfp4_grouped_gemm", a, sfa, row_offsets, num_experts, b, sfb, alpha, false, d, t,
                                  n, k, flags, stream);
}

extern "C" nvfp4_status_t nvfp4_grouped_gemm(const uint8_t *a, const uint8_t *sfa, const int64_t *row_offsets,
                                             int num_experts, const uint8_t *b, const uint8_t *sfb,
                                             const float *alpha, void *d, int64_t t, int64_t n, int64_t k,
                                             uint32_t flags, nvfp4_stream_t stream) {
  if (num_experts <= GroupedCfgNvWide::MAX_EXPERTS)
    return grouped_gemm<GroupedCfgNvWide>("nvfp4_grouped_gemm", a, sfa, row_offsets, num_experts, b, sfb, alpha, true,
                                         d, t, n, k, flags, stream);
  if (k % 256 == 0)
    return grouped_gemm<GroupedCfgNv2>("nvfp4_grouped_gemm", a, sfa, row_offsets, num_experts, b, sfb, alpha, true,
                                       d, t, n, k, flags, stream);
  return grouped_gemm<GroupedCfgNv>("nvfp4_grouped_gemm", a, sfa, row_offsets, num_experts, b, sfb, alpha, true, d,
                                    t, n, k, flags, stream);
}
