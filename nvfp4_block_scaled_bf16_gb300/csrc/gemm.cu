// NVFP4 dense GEMM entry point and its M-based tile selector.
//
// Selector (the role of "SM103 Dispatch" in vLLM fork compare view "add pdl",
// nvfp4_scaled_mm_kernels.cu, which buckets M into [1,16], (16,256], (256,inf); and of the
// narrow output tiles FlashInfer PR 4865's "Reviewer Notes" credit for small-M speed):
//   M <= 256  (unless CTA-pair tiles fit, below) swap A and B: the weight's rows fill the
//             128-row MMA slot and the tokens the
//             N slot (N = 32, 64, 128 or 256, the smallest that holds M), so no MMA row is
//             wasted on padding; K is split over a thread-block cluster of up to 8 CTAs until the
//             grid covers the SMs (both CTA slots of each SM for N = 32), and the partial tiles
//             are reduced through distributed shared memory (decode shapes are weight-streaming,
//             so every SM must pull).
//             Measured against a stream-K split through the workspace, the cluster reduction
//             was 2 us faster at M <= 32 and 2x faster at M = 256, where one CTA would have to
//             read every 128 KB partial of a tile (and against partials pushed into the owning
//             CTA with st.async: 2 us faster per GEMM from cold L2).  When a CTA's K slice fits
//             its ring the operands land with few copies ("resident"), and at most 3 stages per
//             CTA are in flight: with cold HBM, requesting every stage at once made all of them
//             land together, leaving no load for the MMAs to overlap.
//   M >  256  256 x 256 tiles computed by CTA pairs (cta_group::2) when N is a multiple of 256
//             and either there are at least as many 128 x 256 tiles as SMs, or M > 128 and the
//             pair tiles occupy at least a quarter of the pairs; otherwise 128 x 128 tiles on
//             single CTAs.  A pair's ring stage holds two 256-wide K steps when K % 256 == 0.  Persistent over the SMs, double-buffered accumulators where tensor
//             memory allows (128 x 128).  When the tiles fill less than half the SMs and K is
//             long (>= 4 K stages per SM), the (tile, K stage) units are split stream-K over all
//             SMs and split tiles are added up through the workspace.  Splitting the last wave of
//             large shapes the same way was measured slower: every SM is already bound by its
//             own L2 -> shared-memory bandwidth, and the partials add traffic.
#include "gemm.cuh"
#include "host.h"

namespace nvfp4 {
namespace {

struct Plan {
  int swap, bn, splits, stages, ctas, m_tiles, n_tiles, k_tiles, dp_tiles, sk_tiles;
  int pair;  // 1: 256 x 256 tiles computed by CTA pairs (cta_group::2); m_tiles counts 256 rows
  int resident, nst_max, lookahead;  // see GemmArgs
  int ks;    // 256-wide K steps per ring stage (2: pairs whose K is a multiple of 256)
  size_t ws_bytes;
};

constexpr size_t kWsAlign = 256;

// Most CTAs sharing one stream-K tile: the fix-up stages n 16 KB column chunks in the ring.
constexpr int kMaxContributors = 12;

int max_contributors(int64_t sk_tiles, int k_tiles, int ctas) {
  const int64_t units = sk_tiles * k_tiles;
  auto owner = [&](int64_t v) { return ((v + 1) * ctas + units - 1) / units - 1; };
  int64_t most = 1;
  for (int64_t t = 0; t < sk_tiles; ++t) {
    const int64_t c = owner((t + 1) * k_tiles - 1) - owner(t * k_tiles) + 1;
    most = c > most ? c : most;
  }
  return static_cast<int>(most);
}

// weight_streaming: a plan of the swap-AB (weight-streaming) kind for every m <= 256, as the
// fused quantisation needs (its CTAs quantise the token rows they read).
Plan select_plan(int64_t m, int64_t n, int64_t k, int sm_count, bool weight_streaming = false) {
  Plan pl{};
  pl.ks = 1;
  pl.k_tiles = static_cast<int>(ceil_div(k, 256));
  pl.splits = 1;
  // 256 x 256 tiles on CTA pairs pay from 129 tokens on when they occupy at least a quarter of
  // the pairs (measured, cold PDL chains: 256 x 14336 x 4096 23.0 -> 16.0 us, 1024 x 4096 x 7168
  // 31.0 -> 23.8 us; with fewer tiles, e.g. 256 x 4096 x 7168, swap-AB split-K stays faster)
  const bool pair_tiles = n % 256 == 0 && m > 128 && ceil_div(m, 256) * (n / 256) >= sm_count / 4;
  // Whole 128 x 128 tiles beat the swap-AB split-K plans where K is short, since the split's
  // cluster reduction then costs more than the extra SMs streaming the weight gain (measured,
  // PDL chains of cold weights, us per GEMM):
  //  - K <= 2048 from 17 tokens on: 32 / 64 / 128 / 256 x 7168 x 2048 8.2 / 8.9 / 9.9 / 12.4 ->
  //    7.8 / 7.8 / 8.2 / 8.8, 128 / 256 x 4096 x 2048 9.6 / 12.4 -> 8.3 / 8.3, 128 x 14336 x 2048
  //    13.0 -> 9.0;
  //  - K <= 4096 from 129 tokens on (two token tiles): 256 x 7168 x 4096 15.0 -> 12.0, 256 x 4096
  //    x 4096 13.6 -> 11.6.  With one token tile (128 x 4096 x 4096: 10.9 -> 11.5) or at K = 7168
  //    with 64 tiles (256 x 4096 x 7168: 14.3 -> 15.7) they lose.
  // Kept to the measured N range, and never split stream-K (which measured slower here).
  const bool whole_tiles = !weight_streaming && n >= 4096 && n <= 16384 &&
                           ((m > 16 && k <= 2048) || (m > 128 && k <= 4096));
  if (m <= 256 && (weight_streaming || (!pair_tiles && !whole_tiles))) {
    pl.swap = 1;
    pl.bn = m <= 32 ? 32 : m <= 64 ? 64 : m <= 128 ? 128 : 256;
    pl.m_tiles = static_cast<int>(ceil_div(n, 128));  // weight rows
    pl.n_tiles = static_cast<int>(ceil_div(m, pl.bn));
    const int tiles = pl.m_tiles * pl.n_tiles;
    // CTA slots to fill: 32-wide tiles run two CTAs per SM, so they split K until both slots of
    // every SM are taken, at most 7 ways (at N=4096, K=7168: 7 splits of 4 stages, which fit the
    // ring at once, against 4 splits of 7 stages: 4.5 % faster in a cold PDL chain of decode
    // GEMMs, 10-14 % at larger N; clusters of 8 launch measurably slower than clusters of 7)
    const int slots = pl.bn == 32 ? 2 * sm_count : sm_count;
    int s = slots / (tiles > 0 ? tiles : 1);
    s = s < 1 ? 1 : (s > 8 ? 8 : s);
    if (pl.bn == 32 && s > 7) s = 7;
    if (s > pl.k_tiles) s = pl.k_tiles;
    pl.splits = s;
    pl.dp_tiles = tiles;
    pl.ctas = tiles * s;
  } else {
    pl.swap = 0;
    pl.bn = (pair_tiles || (n % 256 == 0 && ceil_div(m, 128) * (n / 256) >= sm_count)) ? 256 : 128;
    // 256-wide tiles go to CTA pairs: a single CTA's 128 x 256 tile moves 54 KB through shared
    // memory per K stage (TMA writes, MMA reads, scale reads) and is bound by that bandwidth; a
    // pair stages half of B per CTA.
    pl.pair = pl.bn == 256 ? 1 : 0;
    // a pair lands two K steps of each operand with one 3-D copy when K allows the stage view
    if (pl.pair && k % 256 == 0) {
      pl.ks = 2;
      pl.k_tiles = static_cast<int>(ceil_div(k, 512));
    }
    pl.m_tiles = static_cast<int>(ceil_div(m, pl.pair ? 256 : 128));
    pl.n_tiles = static_cast<int>(ceil_div(n, pl.bn));
    const int tiles = pl.m_tiles * pl.n_tiles;
    const int64_t units = static_cast<int64_t>(tiles) * pl.k_tiles;
    if (pl.pair) {
      const int pairs = sm_count / 2;
      pl.dp_tiles = tiles;
      pl.ctas = 2 * (tiles < pairs ? tiles : pairs);
    } else if (!whole_tiles && 2 * tiles <= sm_count && units >= 4LL * sm_count) {
      // few tiles with a long K: whole tiles would leave most SMs idle
      pl.sk_tiles = tiles;
      pl.ctas = sm_count;
    } else {
      pl.dp_tiles = tiles;
      pl.ctas = tiles < sm_count ? tiles : sm_count;
    }
  }
  if (pl.sk_tiles > 0 && max_contributors(pl.sk_tiles, pl.k_tiles, pl.ctas) > kMaxContributors) {
    const int tiles = pl.dp_tiles + pl.sk_tiles;  // too fine a split: whole tiles instead
    pl.dp_tiles = tiles;
    pl.sk_tiles = 0;
    pl.ctas = tiles < sm_count ? tiles : sm_count;
  }
  // (stream-K plans use 128-wide tiles and at most sm_count / 2 split tiles)
  if (pl.sk_tiles > 0) pl.ws_bytes = stream_k_workspace_bytes(pl.sk_tiles, pl.ctas, pl.bn);
  // Rings as deep as shared memory allows: a swap-AB CTA then has its whole K run in flight
  // from the start (the decode GEMM is bound by load latency, not by shared memory).  The
  // narrowest tiles instead keep a 4-stage ring so that two CTAs fit an SM: under PDL the next
  // GEMM's CTAs then start beside this one's and pull their weights (ring + L2 prefetch) while
  // this one finishes.
  switch (pl.bn) {
    case 32: pl.stages = 4; break;
    case 64: pl.stages = 7; break;
    case 128: pl.stages = 6; break;
    default: pl.stages = pl.pair ? (pl.ks == 2 ? 3 : 5) : 4; break;
  }
  // A swap-AB CTA holds one tile; when its whole K slice fits the ring (and K is a whole number of
  // 256-wide stages), the activation and both scale slices land with one copy each.
  pl.nst_max = static_cast<int>(ceil_div(pl.k_tiles, pl.splits));
  pl.resident = pl.swap && k % 256 == 0 && pl.nst_max <= pl.stages && pl.bn <= 128;
  // Weight-streaming (swap-AB) CTAs keep only a few stages in flight: when every CTA requests
  // its whole slice at once, cold HBM completes all of a CTA's stages at about the same time and
  // the MMAs cannot overlap the loads; paced requests land in order.
  pl.lookahead = pl.swap && pl.bn > 32 ? 3 : 0;
  return pl;
}

int plan_sm_count() {
  int sms = 152;
  DeviceInfo dev;
  int cur = -1;
  if (cudaGetDevice(&cur) == cudaSuccess && current_device(&dev) == NVFP4_OK) sms = dev.sm_count;
  clear_error();
  return sms;
}

// Calls f with the kernel configuration of a plan (a GemmCfg value).
template <class F>
nvfp4_status_t with_config(const Plan &pl, F &&f) {
  // swap-AB CTAs hold one tile (single accumulator); large-M CTAs walk tiles persistently and
  // overlap the epilogue with the next tile where tensor memory allows
  switch (pl.bn) {
    case 32: return f(GemmCfg<32, 4, false, false, 2>{});
    case 64: return f(GemmCfg<64, 7, false, false>{});
    case 128: return pl.swap ? f(GemmCfg<128, 6, false, false>{}) : f(GemmCfg<128, 6, false, true>{});
    default:
      if (pl.swap) return f(GemmCfg<256, 4, false, false>{});
      return pl.ks == 2 ? f(GemmCfg<256, 3, false, true, 1, true, 1024, 2>{}) : f(GemmCfg<256, 5, false, true, 1, true>{});
  }
}

// Raises the kernel's dynamic shared-memory limit (once per kernel and device).
template <class C, bool FUSED = false>
nvfp4_status_t prepare(const DeviceInfo &dev) {
  return allow_smem(reinterpret_cast<const void *>(bs_gemm_kernel<C, false, FUSED>), C::smem_bytes(false), dev.device);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status_t nvfp4_gemm_plan(int64_t m, int64_t n, int64_t k, nvfp4_gemm_plan_t *plan) {
  clear_error();
  if (!plan || m < 0 || n <= 0 || k <= 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gemm_plan: bad arguments");
  const Plan pl = select_plan(m, n, k, plan_sm_count());
  plan->swap_ab = pl.swap;
  plan->tile_m = pl.pair ? 256 : 128;
  plan->tile_n = pl.bn;
  plan->splits = pl.splits;
  plan->stages = pl.stages;
  plan->ctas = pl.ctas;
  plan->dp_tiles = pl.dp_tiles;
  plan->sk_tiles = pl.sk_tiles;
  return NVFP4_OK;
}

extern "C" nvfp4_status_t nvfp4_gemm_workspace_size(int64_t m, int64_t n, int64_t k, size_t *bytes) {
  clear_error();
  if (!bytes || m < 0 || n <= 0 || k <= 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gemm_workspace_size: bad arguments");
  *bytes = m == 0 ? 0 : select_plan(m, n, k, plan_sm_count()).ws_bytes;
  return NVFP4_OK;
}

namespace nvfp4 {
namespace {

// Activation to quantise inside the kernel (nvfp4_quantize_gemm); a == nullptr: none.
struct FusedA {
  const __nv_bfloat16 *x;
  int64_t ldx;
  const float *gs;
};

nvfp4_status_t run_gemm(const char *name, const uint8_t *a, const uint8_t *sfa, const uint8_t *b, const uint8_t *sfb,
                        const float *alpha, void *d, int64_t m, int64_t n, int64_t k, void *workspace,
                        size_t workspace_bytes, uint32_t flags, nvfp4_stream_t stream, const FusedA &fq) {
  const bool fused = fq.x != nullptr;
  if (m < 0 || n <= 0 || k <= 0 || m >= (1LL << 31) || n >= (1LL << 31) || k >= (1LL << 31))
    return fail(NVFP4_ERR_INVALID_ARG, "%s: m=%lld n=%lld k=%lld", name, (long long)m, (long long)n, (long long)k);
  if (k % 32 || n % 32)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: need k %% 32 == 0 and n %% 32 == 0 (k=%lld n=%lld)", name, (long long)k, (long long)n);
  if (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT | NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD | NVFP4_FLAG_SF_SM103))
    return fail(NVFP4_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags);
  if (m == 0) return NVFP4_OK;
  if ((!fused && (!a || !sfa)) || !b || !sfb || !alpha || !d) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", name);
  if ((!fused && (!aligned(a, 32) || !aligned(sfa, 16))) || !aligned(b, 32) || !aligned(d, 32) || !aligned(sfb, 16) ||
      !aligned(alpha, 4))
    return fail(NVFP4_ERR_MISALIGNED, "%s: a, b, d need 32-B and sfa, sfb 16-B alignment", name);
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  const Plan pl = select_plan(m, n, k, dev.sm_count, fused);
  // A swap-AB plan holds every token in one tile (tile_n >= m): the kernels read operand B's
  // scales with scale-factor ID 0, i.e. rows 0..BN-1 of each 128-row scale block, so a second
  // token tile at a row offset that is not a multiple of 128 would take the wrong scales.
  if (pl.swap && pl.n_tiles != 1)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: internal plan error (swap-AB with %d token tiles)", name, pl.n_tiles);
  if (fused && !pl.swap)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "%s: the quantisation is fused into the weight-streaming plans (m <= 256, got %lld); quantise with "
                "nvfp4_quantize and call nvfp4_gemm", name, (long long)m);
  st = with_config(pl, [&](auto cfg) {
    using C = decltype(cfg);
    if constexpr (C::SWAP_ONLY) {
      if (fused) return prepare<C, true>(dev);
    }
    return prepare<C>(dev);
  });
  if (st != NVFP4_OK) return st;
  if (pl.ws_bytes > 0) {
    if (!workspace || workspace_bytes < pl.ws_bytes)
      return fail(NVFP4_ERR_INVALID_ARG, "%s: this shape needs a workspace of %zu bytes (got %zu%s)", name,
                  pl.ws_bytes, workspace_bytes, workspace ? "" : ", NULL");
    if (!aligned(workspace, kWsAlign)) return fail(NVFP4_ERR_MISALIGNED, "%s: workspace needs 256-B alignment", name);
  }
  // Kernel operand A fills the 128-row MMA slot; with swap it is the weight B.
  const uint8_t *opa = pl.swap ? b : a, *opb = pl.swap ? a : b;
  const uint8_t *sfopa = pl.swap ? sfb : sfa, *sfopb = pl.swap ? sfa : sfb;
  const int64_t rows_a = pl.swap ? n : m, rows_b = pl.swap ? m : n;
  CUtensorMap ta, tb, tb3;
  if (pl.ks == 2) {
    // stage views: a box is two 256-wide K steps (two 128-byte rows) of 128 rows
    st = encode_tmap_stages_u8(&ta, opa, k / 2, rows_a, 128, 2);
    if (st == NVFP4_OK) st = encode_tmap_stages_u8(&tb, opb, k / 2, rows_b, pl.bn / 2, 2);
    tb3 = tb;  // unused
  } else {
    st = encode_tmap_2d_u8(&ta, opa, k / 2, rows_a, k / 2, 128, 128, true);
    if (st == NVFP4_OK && fused) tb = ta;  // operand B is produced in the kernel: its maps are unused
    else if (st == NVFP4_OK)
      st = encode_tmap_2d_u8(&tb, opb, k / 2, rows_b, k / 2, 128, pl.pair ? pl.bn / 2 : pl.bn, true);
    if (st == NVFP4_OK && pl.resident && !fused) st = encode_tmap_stages_u8(&tb3, opb, k / 2, rows_b, pl.bn, pl.nst_max);
    else tb3 = tb;  // unused
  }
  if (st != NVFP4_OK) return st;

  GemmArgs args{};
  args.sfa = sfopa;
  args.sfb = fused ? sfopa : sfopb;  // (unused when fused)
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
  args.dp_tiles = pl.dp_tiles;
  args.sk_tiles = pl.sk_tiles;
  args.resident = pl.resident;
  args.nst_max = pl.nst_max;
  args.lookahead = pl.lookahead;
  args.sf_sm103 = (flags & NVFP4_FLAG_SF_SM103) ? 1 : 0;
  args.xq = fq.x;
  args.ldx = fq.ldx;
  args.gs_q = fq.gs;
  if (pl.sk_tiles > 0) {
    args.ws_cnt = static_cast<unsigned int *>(workspace);
    args.ws = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                        round_up(static_cast<int64_t>(pl.sk_tiles) * 4, kWsAlign));
  }

  cudaStream_t s = (cudaStream_t)stream;
  return with_config(pl, [&](auto cfg) {
    using C = decltype(cfg);
    const bool pdl = (flags & NVFP4_FLAG_PDL) != 0;
    const int cx = pl.pair ? 2 : pl.splits;
    if constexpr (C::SWAP_ONLY) {
      if (fused)
        return check_launch(launch(bs_gemm_kernel<C, false, true>, dim3(pl.ctas), dim3(C::THREADS),
                                   C::smem_bytes(false), s, pdl, cx, ta, tb, tb3, args), name);
    }
    const cudaError_t e = launch(bs_gemm_kernel<C, false>, dim3(pl.ctas), dim3(C::THREADS), C::smem_bytes(false), s,
                                 pdl, cx, ta, tb, tb3, args);
    return check_launch(e, name);
  });
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status_t nvfp4_gemm(const uint8_t *a, const uint8_t *sfa, const uint8_t *b,
                                     const uint8_t *sfb, const float *alpha, void *d, int64_t m,
                                     int64_t n, int64_t k, void *workspace, size_t workspace_bytes,
                                     uint32_t flags, nvfp4_stream_t stream) {
  clear_error();
  return run_gemm("nvfp4_gemm", a, sfa, b, sfb, alpha, d, m, n, k, workspace, workspace_bytes, flags, stream,
                  FusedA{nullptr, 0, nullptr});
}

extern "C" nvfp4_status_t nvfp4_quantize_gemm(const void *x, int64_t ldx, const float *gs_x, const uint8_t *b,
                                              const uint8_t *sfb, const float *alpha, void *d, int64_t m,
                                              int64_t n, int64_t k, void *workspace, size_t workspace_bytes,
                                              uint32_t flags, nvfp4_stream_t stream) {
  clear_error();
  if (m > 0 && (!x || !gs_x)) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_gemm: null pointer");
  if (m > 0 && ldx < k)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_gemm: ldx=%lld < k=%lld", (long long)ldx, (long long)k);
  if (m > 0 && (!aligned(x, 16) || ldx % 8 || !aligned(gs_x, 4)))
    return fail(NVFP4_ERR_MISALIGNED, "nvfp4_quantize_gemm: x needs 16-B alignment and ldx %% 8 == 0");
  return run_gemm("nvfp4_quantize_gemm", nullptr, nullptr, b, sfb, alpha, d, m, n, k, workspace, workspace_bytes,
                  flags, stream, FusedA{static_cast<const __nv_bfloat16 *>(x), ldx, gs_x});
}
