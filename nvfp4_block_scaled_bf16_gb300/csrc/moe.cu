// The MoE steps around the grouped GEMMs, NVFP4 flavour: expert sort of the routed tokens,
// row gather, per-expert NVFP4 quantisation (plain, fused with the row gather, or fused with
// SiLU-and-mul), weighted combine.  Named on vLLM fork compare view "add pdl" (ops.h, torch_bindings.cpp:
// scaled_fp4_experts_quant, silu_and_mul_scaled_fp4_experts_quant with input_offset_by_experts /
// output_scale_offset_by_experts) and vLLM PR 51158 "Changes" (experts quantise, grouped GEMM);
// the pages give names and arguments only, the definitions used are stated per entry point in
// nvfp4.h.  All of these are CUDA-core kernels: the gather and combine are bound by memory
// bandwidth, the sort by latency, and the per-expert quantisers by instruction issue.
#include <cuda_bf16.h>

#include "host.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kMaxExpertsMoe = 1024;
// 128-row scale blocks whose owning expert the per-position quantiser tabulates in shared
// memory (8 KB; 512K scale rows); beyond that it searches the scale-row prefix per position.
constexpr int kExpertBlockTable = 4096;

// ------------------------------------------------------------------ expert sort
// A stable counting sort in two kernels over G CTAs, CTA g owning tokens [g*tpc, (g+1)*tpc):
//   1. moe_count_kernel: CTA g counts its (token, slot) pairs per expert -> hist[g][e];
//   2. moe_place_kernel: CTA g derives, for every expert e, its first row
//        row_offsets[e] + sum_{g' < g} hist[g'][e]   (row_offsets = prefix of the expert totals)
//      then its 8 warps (tokens split in order between them) count again per warp, take their own
//      first rows, and walk their tokens in order with lanes = slots; lanes holding the same expert
//      (a repeated id) are ranked by slot with __match_any_sync.  Rows of an expert therefore keep
//      (token, slot) order.
// Ids outside [0, E) are dropped (pos = -1) and set bit 3 of the status word.
constexpr int kPlaceWarps = 8;

__global__ void __launch_bounds__(256) moe_count_kernel(const int32_t *__restrict__ ids, int T, int topk, int E,
                                                        int tpc, int32_t *__restrict__ hist, unsigned int *status) {
  extern __shared__ int32_t c[];  // [E]
  pdl_trigger();
  pdl_wait();
  for (int e = threadIdx.x; e < E; e += blockDim.x) c[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * tpc, t1 = min(T, t0 + tpc);
  for (int i = t0 * topk + threadIdx.x; i < t1 * topk; i += blockDim.x) {
    const int v = ids[i];
    if (v >= 0 && v < E) atomicAdd(&c[v], 1);
    else atomicOr(status, 8u);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = c[e];
}

__global__ void __launch_bounds__(kPlaceWarps * 32) moe_place_kernel(const int32_t *__restrict__ ids, int T, int topk,
                                                                     int E, int tpc, const int32_t *__restrict__ hist,
                                                                     int64_t *__restrict__ row_offsets,
                                                                     int32_t *__restrict__ src,
                                                                     int32_t *__restrict__ pos) {
  extern __shared__ int32_t sm[];
  int32_t *base = sm;            // [E]: this CTA's first row per expert
  int32_t *cnt = sm + E;         // [kPlaceWarps][E]: per-warp counts, then per-warp first rows
  __shared__ int32_t scan[kMaxExpertsMoe];
  pdl_trigger();
  pdl_wait();
  const int G = gridDim.x, g = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    scan[e] = 0;
    base[e] = 0;
  }
  for (int i = threadIdx.x; i < kPlaceWarps * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  // Expert totals and the part of each expert that earlier CTAs own.  P threads share an expert's
  // column of the count table (strided over the CTAs), each with 8 loads in flight, and add
  // their integer partials into shared memory: a CTA's walk of the table is ~G/(8P) load
  // latencies instead of G.
  const int P = E < static_cast<int>(blockDim.x) ? static_cast<int>(blockDim.x) / E : 1;
  for (int i = threadIdx.x; i < E * P; i += blockDim.x) {
    const int e = i % E, p = i / E;
    int before = 0, total = 0;
    int h = p;
    for (; h + 7 * P < G; h += 8 * P) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = hist[static_cast<int64_t>(h + u * P) * E + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        total += v[u];
        before += h + u * P < g ? v[u] : 0;
      }
    }
    for (; h < G; h += P) {
      const int v = hist[static_cast<int64_t>(h) * E + e];
      total += v;
      before += h < g ? v : 0;
    }
    atomicAdd(&scan[e], total);
    atomicAdd(&base[e], before);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix of the totals: a warp scan, 32 experts at a time
    int carry = 0;
    for (int b0 = 0; b0 < E; b0 += 32) {
      const int e = b0 + lane;
      const int v = e < E ? scan[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) {
        scan[e] = carry + incl - v;
        if (g == 0) row_offsets[e] = carry + incl - v;
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (g == 0 && lane == 0) row_offsets[E] = carry;
  }
  __syncthreads();
  const int t0 = g * tpc, t1 = min(T, t0 + tpc);
  const int tpw = (t1 - t0 + kPlaceWarps - 1) / kPlaceWarps;
  const int w0 = min(t1, t0 + warp * tpw), w1 = min(t1, w0 + tpw);
  for (int i = w0 * topk + lane; i < w1 * topk; i += 32) {
    const int v = ids[i];
    if (v >= 0 && v < E) atomicAdd(&cnt[warp * E + v], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {  // per-warp first rows inside the CTA's share
    int run = scan[e] + base[e];
    for (int w = 0; w < kPlaceWarps; ++w) {
      const int v = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  for (int t = w0; t < w1; ++t) {
    const bool active = lane < topk;
    const int v = active ? ids[t * topk + lane] : -1;
    const bool ok = active && v >= 0 && v < E;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, ok ? v : -1 - lane);  // invalid lanes alone
    const int rank = __popc(peers & ((1u << lane) - 1));
    int first = 0;
    if (ok && rank == 0) {  // the lowest lane of each group advances the counter for the group
      first = cnt[warp * E + v];
      cnt[warp * E + v] = first + __popc(peers);
    }
    first = __shfl_sync(0xFFFFFFFFu, first, __ffs(peers) - 1);
    if (active) {
      if (ok) {
        const int row = first + rank;
        src[row] = t;
        pos[t * topk + lane] = row;
      } else {
        pos[t * topk + lane] = -1;
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ row gather
// out[r, :] = x[src[r], :] for r < rows; 16-byte pieces, grid-stride.  A source row outside
// [0, T) sets bit 3 of the status word and its output row is left untouched.
// I: the position type (32-bit when rows * pieces plus one grid stride < 2^31: a cheaper
// division per position).
template <typename I>
__global__ void __launch_bounds__(256) moe_gather_kernel(const uint4 *__restrict__ x, int64_t ldx16, int64_t T,
                                                         const int32_t *__restrict__ src, int64_t rows,
                                                         int64_t pieces_, uint4 *__restrict__ out,
                                                         unsigned int *status) {
  pdl_trigger();
  pdl_wait();
  const I pieces = static_cast<I>(pieces_);
  const I total = static_cast<I>(rows * pieces_);
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  for (I i = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const I r_ = i / pieces;
    const int64_t r = r_, c = i - r_ * pieces;
    const int64_t s = src[r];
    if (s < 0 || s >= T) {
      if (c == 0) atomicOr(status, 8u);
      continue;
    }
    out[r * pieces + c] = __ldg(x + s * ldx16 + c);
  }
}

// ------------------------------------------------------------------ weighted combine
// out[t, :] = bf16(sum_j w[t, j] * y[pos[t, j], :]), fp32 products and sums in slot order, no
// fused multiply-add; a slot with pos < 0 (an entry the sort dropped) contributes nothing.
// One thread per 8 output elements (16-byte loads of y, 16-byte store).
// I: the position type (as in the gather).
template <typename I>
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint4 *__restrict__ y, int64_t rows,
                                                          const int32_t *__restrict__ pos,
                                                          const float *__restrict__ w, int64_t T, int topk,
                                                          int64_t pieces_, uint4 *__restrict__ out,
                                                          unsigned int *status) {
  pdl_trigger();
  pdl_wait();
  const I pieces = static_cast<I>(pieces_);
  const I total = static_cast<I>(T * pieces_);
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  for (I i = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const I t_ = i / pieces;
    const int64_t t = t_, c = i - t_ * pieces;
    float acc[8];
    bool first = true;
    for (int j = 0; j < topk; ++j) {
      const int64_t p = pos[t * topk + j];
      if (p < 0) continue;
      if (p >= rows) {
        if (c == 0) atomicOr(status, 8u);
        continue;
      }
      const float wj = w[t * topk + j];
      const uint4 v = __ldg(y + p * pieces + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(u[q] << 16), hi = __uint_as_float(u[q] & 0xFFFF0000u);
        const float plo = __fmul_rn(wj, lo), phi = __fmul_rn(wj, hi);
        acc[2 * q] = first ? plo : __fadd_rn(acc[2 * q], plo);
        acc[2 * q + 1] = first ? phi : __fadd_rn(acc[2 * q + 1], phi);
      }
      first = false;
    }
    uint4 o;
    uint32_t *op = &o.x;
#pragma unroll
    for (int q = 0; q < 4; ++q) op[q] = first ? 0u : pack_bf16x2(acc[2 * q], acc[2 * q + 1]);
    out[t * pieces + c] = o;
  }
}

// ------------------------------------------------------------------ per-expert NVFP4 quantiser
// exp(t) in fp32 by Cody and Waite's range reduction and a degree-7 Taylor polynomial, every
// step rounded to nearest even and nothing fused (so it is reproducible off the GPU):
//   n = rint(t * log2 e); r = (t - n*LN2_HI) - n*LN2_LO; p = Horner(1/k!, k = 7..0); exp = p*2^n
// with LN2_HI = 0.693145751953125 (16 significant bits, so n*LN2_HI is exact), t > 88 -> inf,
// t < -87 -> 0.  Within 1.2 fp32 ulps of exp on [-87, 88].  silu(g) = g * (1 / (1 + exp(-g))).
// Both run on two values at once with Blackwell's packed fp32 instructions (mul/add/sub
// .rn.f32x2 round each lane to nearest even exactly as the scalar forms, so each lane's result
// is that of the scalar steps); the range tests are per-lane selects after the polynomial.
// rint: adding 1.5 * 2^23 rounds to an integer (nearest even) for |x| < 2^22 and leaves it in
// the low mantissa bits; subtracting it again gives rint(x) exactly.  Larger |x| only occur for
// t outside [-87, 88], whose results the selects replace.  This keeps the float<->int
// conversions, a low-rate pipe, off the path (SiLU form 45.0 -> 43.3 us, bit-identical).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t exp_cw2(float t0, float t1) {
  const uint64_t t = pk2(t0, t1);
  const uint64_t m = mul2(t, pk2(1.44269502162933349609375f, 1.44269502162933349609375f));
  const uint64_t sh = add2(m, pk2(12582912.0f, 12582912.0f));  // 1.5 * 2^23
  const uint64_t n = sub2(sh, pk2(12582912.0f, 12582912.0f));   // rint(m), exact
  float sh0, sh1;
  upk2(sh, sh0, sh1);
  const int i0 = __float_as_int(sh0) - 0x4B400000, i1 = __float_as_int(sh1) - 0x4B400000;  // rint(m) as int
  const uint64_t r = sub2(sub2(t, mul2(n, pk2(0.693145751953125f, 0.693145751953125f))),
                          mul2(n, pk2(1.428606765330187045037746429443359375e-06f, 1.428606765330187045037746429443359375e-06f)));
  const float c[7] = {1.388888922519981861114501953125e-03f, 8.333333767950534820556640625e-03f,
                      4.16666679084300994873046875e-02f, 0.16666667163372039794921875f, 0.5f, 1.0f, 1.0f};
  uint64_t p = pk2(1.98412701138295233249664306640625e-04f, 1.98412701138295233249664306640625e-04f);
#pragma unroll
  for (int q = 0; q < 7; ++q) p = add2(mul2(r, p), pk2(c[q], c[q]));
  float e0, e1;
  upk2(mul2(p, pk2(__int_as_float((i0 + 127) << 23), __int_as_float((i1 + 127) << 23))), e0, e1);
  e0 = t0 > 88.0f ? __int_as_float(0x7F800000) : (t0 < -87.0f ? 0.0f : e0);
  e1 = t1 > 88.0f ? __int_as_float(0x7F800000) : (t1 < -87.0f ? 0.0f : e1);
  return pk2(e0, e1);
}
// (g0, g1), (u0, u1) -> the fp32 values of h = bf16(silu(g) * u) for both
__device__ __forceinline__ void silu_mul_bf16x2(float &g0, float &g1, float u0, float u1) {
  float d0, d1;
  upk2(add2(pk2(1.0f, 1.0f), exp_cw2(-g0, -g1)), d0, d1);
  const uint64_t sig = pk2(__fdiv_rn(1.0f, d0), __fdiv_rn(1.0f, d1));
  float h0, h1;
  upk2(mul2(mul2(pk2(g0, g1), sig), pk2(u0, u1)), h0, h1);
  const uint32_t hb = pack_bf16x2(h0, h1);
  g0 = __uint_as_float(hb << 16);
  g1 = __uint_as_float(hb & 0xFFFF0000u);
}

__device__ __forceinline__ void bf16x8_to_f32_moe(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}


// One warp per scale row of the grouped padded scale matrix (expert e owns scale rows sfr[e] ..
// sfr[e+1]-1, sfr[e+1] - sfr[e] = round_up(M_e, 128)), lane = scale column within a 32-column
// pass; rows past an expert's last token and columns past K/16 get scale 0x00.  The expert of a
// row is looked up once per warp.  SILU: the 16 quantised values are
// h = bf16(silu(x[r, c]) * x[r, I + c]) for the block's columns c (x is [T, 2I]).
template <bool SILU>
__global__ void __launch_bounds__(256) expert_quant_kernel(const __nv_bfloat16 *__restrict__ x, int64_t t,
                                                           int kb, int64_t ldx, int64_t up_off,
                                                           const int64_t *__restrict__ row_offsets, int experts,
                                                           const float *__restrict__ gs_e, uint8_t *__restrict__ q,
                                                           uint8_t *__restrict__ sf, int64_t cap_rows, int cp) {
  __shared__ int64_t s_ro[kMaxExpertsMoe + 1];
  __shared__ int64_t s_sfr[kMaxExpertsMoe + 1];
  pdl_trigger();
  pdl_wait();
  for (int e = threadIdx.x; e <= experts; e += blockDim.x) s_ro[e] = row_offsets[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t acc = 0;
    s_sfr[0] = 0;
    for (int e = 0; e < experts; ++e) {
      int64_t cnt = s_ro[e + 1] - s_ro[e];
      cnt = cnt < 0 ? 0 : cnt;
      acc += (cnt + 127) / 128 * 128;
      s_sfr[e + 1] = acc;
    }
  }
  __syncthreads();
  const int64_t rows = s_sfr[experts] < cap_rows ? s_sfr[experts] : cap_rows;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t srow = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + warp; srow < rows; srow += wstride) {
    int lo = 0, hi = experts - 1;  // expert owning scale row srow: largest e with s_sfr[e] <= srow
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_sfr[mid] <= srow) lo = mid;
      else hi = mid - 1;
    }
    const int64_t local = srow - s_sfr[lo];
    const int64_t r = s_ro[lo] + local;
    const bool row_ok = local < s_ro[lo + 1] - s_ro[lo] && r >= 0 && r < t;
    const float gs = row_ok ? __ldg(gs_e + lo) : 0.0f;
    const __nv_bfloat16 *xrow = x + (row_ok ? r : 0) * ldx;
    uint8_t *qrow = q + (row_ok ? r : 0) * (static_cast<int64_t>(kb) * 8);
    uint8_t *sf_tile_row = sf + (srow >> 7) * (static_cast<int64_t>(cp) >> 2) * 512 + (srow & 31) * 16 + ((srow >> 5) & 3) * 4;
    // Passes of 32 blocks, P at a time: all P passes' loads are issued before any is converted,
    // so a warp keeps P KB in flight instead of one (65.5 -> 52.5 us at T=32768, K=2048).  The
    // SiLU form is bound by its arithmetic: it keeps one pass, and its registers, for occupancy.
    constexpr int P = SILU ? 1 : 4;
    for (int j00 = 0; j00 < cp; j00 += 32 * P) {  // every lane runs the same passes (shuffles below)
      uint4 xg[P][2], xu[P][2];
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        const int j = j00 + 32 * pp + lane;
        xg[pp][0] = xg[pp][1] = xu[pp][0] = xu[pp][1] = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok && j < kb) {
          const uint4 *src = reinterpret_cast<const uint4 *>(xrow + j * 16);
          xg[pp][0] = __ldg(src);
          xg[pp][1] = __ldg(src + 1);
          if (SILU) {
            const uint4 *up = reinterpret_cast<const uint4 *>(xrow + up_off + j * 16);
            xu[pp][0] = __ldg(up);
            xu[pp][1] = __ldg(up + 1);
          }
        }
      }
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        const int j0 = j00 + 32 * pp;
        if (j0 >= cp) break;  // uniform over the warp
        const int j = j0 + lane;
        uint32_t code = 0;
        if (row_ok && j < kb) {
          float f[16];
          bf16x8_to_f32_moe(xg[pp][0], f);
          bf16x8_to_f32_moe(xg[pp][1], f + 8);
          if (SILU) {
            float u[16];
            bf16x8_to_f32_moe(xu[pp][0], u);
            bf16x8_to_f32_moe(xu[pp][1], u + 8);
#pragma unroll
            for (int i = 0; i < 8; ++i) silu_mul_bf16x2(f[2 * i], f[2 * i + 1], u[2 * i], u[2 * i + 1]);
          }
          *reinterpret_cast<uint2 *>(qrow + j * 8) = nvfp4_block16(f, gs, code);
        }
        // 4 lanes (scale columns 4c .. 4c+3 of the row) -> one 32-bit word of the 128x4 layout
        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, code, 1);
        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, code, 2);
        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, code, 3);
        if ((j & 3) == 0 && j < cp)
          *reinterpret_cast<uint32_t *>(sf_tile_row + (j >> 2) * 512) = code | (b1 << 8) | (b2 << 16) | (b3 << 24);
      }
    }
  }
}

// The same quantisation with one thread per (scale row, scale column) position of the grouped
// padded scale matrix: consecutive threads take consecutive 16-element blocks, so a warp's loads
// are contiguous even where a row has few blocks (48 at K = 768), no lane idles on a partial
// pass, and each thread looks up the expert of its scale row in shared memory (a warp's lanes
// read the same entries).  The scale-row prefix is a warp scan.  32-bit positions, rows and
// offsets: the host launches it only when rows * columns < 2^31 (so t < 2^31 too).
// Measured at 128 experts, 32768 rows: SiLU form 67.5 -> 49.2 us, plain form (K=2048) 45.4 ->
// 38.9 us against the warp-per-row kernel, bit-identical.  The kernel is bound by instruction
// issue, not by memory: a position's expert comes from a table of 128-row scale blocks (one
// lookup instead of a binary search over the prefix) and its (row, column) advances by the grid
// stride (no division per position), plain 38.9 -> 32.8 us, SiLU 49.1 -> 47.1 us.  The table is
// filled with one search per entry, in parallel: filling it expert by expert cost more than the
// searches it saves.
template <bool SILU, bool GATHER>
__global__ void __launch_bounds__(256) expert_quant_pos_kernel(const __nv_bfloat16 *__restrict__ x, int64_t t,
                                                               int kb, int64_t ldx, int64_t up_off,
                                                               const int64_t *__restrict__ row_offsets,
                                                               int experts, const float *__restrict__ gs_e,
                                                               uint8_t *__restrict__ q, uint8_t *__restrict__ sf,
                                                               int64_t cap_rows, int cp,
                                                               const int32_t *__restrict__ src, int64_t tokens,
                                                               unsigned int *status) {
  __shared__ int s_ro[kMaxExpertsMoe + 1];
  __shared__ int s_sfr[kMaxExpertsMoe + 1];
  __shared__ uint16_t s_blk[kExpertBlockTable];
  pdl_trigger();
  pdl_wait();
  for (int e = threadIdx.x; e <= experts; e += blockDim.x) s_ro[e] = static_cast<int>(row_offsets[e]);
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < experts; base += 32) {
      const int e = base + lane;
      int v = 0;
      if (e < experts) {
        const int cnt = s_ro[e + 1] - s_ro[e];
        v = (cnt > 0 ? cnt + 127 : 0) / 128 * 128;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
      }
      if (e < experts) s_sfr[e + 1] = carry + v;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) s_sfr[0] = 0;
  }
  __syncthreads();
  // Every expert owns whole 128-row blocks of scale rows, so when there are at most
  // kExpertBlockTable blocks a table gives each block's expert in one lookup.
  const int nblk = s_sfr[experts] >> 7;
  const bool table = nblk >= 0 && nblk <= kExpertBlockTable;
  if (table) {
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
      const int row0 = b << 7;
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
  const int rows = static_cast<int>(s_sfr[experts] < cap_rows ? s_sfr[experts] : cap_rows);
  // a multiple of 512 (every warp runs the same trip count) and below 2^31, so the unsigned
  // position plus one grid stride cannot wrap
  const unsigned int total = rows > 0 ? static_cast<unsigned int>(rows) * cp : 0u;
  const unsigned int stride = gridDim.x * blockDim.x;
  unsigned int idx = blockIdx.x * blockDim.x + threadIdx.x;
  // (scale row, scale column) of idx, stepped by the grid stride without a division per step
  int srow = static_cast<int>(idx / cp), j = static_cast<int>(idx % cp);
  const int ds = static_cast<int>(stride / cp), dj = static_cast<int>(stride % cp);
  for (; idx < total; idx += stride, srow += ds, j += dj) {
    if (j >= cp) {
      j -= cp;
      ++srow;
    }
    int lo;  // expert owning scale row srow: largest e with s_sfr[e] <= srow
    if (table) {
      lo = s_blk[srow >> 7];  // srow < rows <= 128 * nblk; every entry holds an expert in range
    } else {
      lo = 0;
      int hi = experts - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_sfr[mid] <= srow) lo = mid;
        else hi = mid - 1;
      }
    }
    const int64_t local = srow - s_sfr[lo];
    const int64_t r = s_ro[lo] + local;
    bool row_ok = local < s_ro[lo + 1] - s_ro[lo] && r >= 0 && r < t;
    // GATHER: row r of the quantised matrix is row src[r] of x (moe_gather_rows fused in); a
    // source outside [0, tokens) quantises zeros and sets bit 3 of the status word
    int64_t xr = r;
    bool zero_row = false;  // GATHER: a row of the result whose source is out of range
    if (GATHER && row_ok) {
      xr = src[r];
      if (xr < 0 || xr >= tokens) {
        if (j == 0) atomicOr(status, 8u);
        zero_row = true;
      }
    }
    uint32_t code = 0;
    if (row_ok && j < kb) {
      const float gs = __ldg(gs_e + lo);
      const uint4 *xs = reinterpret_cast<const uint4 *>(x + xr * ldx + j * 16);
      uint4 g0 = make_uint4(0u, 0u, 0u, 0u), g1 = g0;
      if (!zero_row) {
        g0 = __ldg(xs);
        g1 = __ldg(xs + 1);
      }
      uint4 u0 = make_uint4(0u, 0u, 0u, 0u), u1 = u0;
      if (SILU) {
        const uint4 *up = reinterpret_cast<const uint4 *>(x + xr * ldx + up_off + j * 16);
        u0 = __ldg(up);
        u1 = __ldg(up + 1);
      }
      float f[16];
      bf16x8_to_f32_moe(g0, f);
      bf16x8_to_f32_moe(g1, f + 8);
      if (SILU) {
        float u[16];
        bf16x8_to_f32_moe(u0, u);
        bf16x8_to_f32_moe(u1, u + 8);
#pragma unroll
        for (int i = 0; i < 8; ++i) silu_mul_bf16x2(f[2 * i], f[2 * i + 1], u[2 * i], u[2 * i + 1]);
      }
      *reinterpret_cast<uint2 *>(q + r * (static_cast<int64_t>(kb) * 8) + j * 8) = nvfp4_block16(f, gs, code);
    }
    // 4 lanes (scale columns 4c .. 4c+3 of the row) -> one 32-bit word of the 128x4 layout
    const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, code, 1);
    const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, code, 2);
    const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, code, 3);
    if ((j & 3) == 0)
      *reinterpret_cast<uint32_t *>(sf + static_cast<int64_t>(srow >> 7) * (cp >> 2) * 512 + (srow & 31) * 16 +
                                    ((srow >> 5) & 3) * 4 + (j >> 2) * 512) = code | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
}

// CTAs of the two sort kernels: about 32 tokens each, at most 1024 (the workspace holds one
// count per CTA and expert).
int moe_sort_ctas(int64_t tokens) {
  const int64_t g = ceil_div(tokens > 0 ? tokens : 1, 32);
  return static_cast<int>(g < 1024 ? g : 1024);
}

int moe_grid(int64_t threads, int sm_count, int per_sm = 8) {
  const int64_t blocks = ceil_div(threads, 256);
  const int64_t cap = static_cast<int64_t>(sm_count) * per_sm;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}
// blocks per SM the gather and combine launch at most
constexpr int kMoveBlocksPerSm = 8;

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t moe_sort_workspace_size(int64_t num_tokens, int num_experts) {
  if (num_tokens < 0 || num_experts < 1) return 0;
  return static_cast<size_t>(moe_sort_ctas(num_tokens)) * num_experts * 4;
}

extern "C" nvfp4_status_t moe_sort_by_expert(const int32_t *topk_ids, int64_t num_tokens, int topk, int num_experts,
                                             int64_t *row_offsets, int32_t *src_rows, int32_t *pos, int32_t *workspace,
                                             size_t workspace_bytes, uint32_t flags, nvfp4_stream_t stream) {
  clear_error();
  if (num_tokens < 0 || topk < 1 || topk > 32 || num_experts < 1 || num_experts > kMaxExpertsMoe ||
      num_tokens * topk > (1LL << 31) - 512)  // the kernels' 32-bit slot loops step past the end by < 512
    return fail(NVFP4_ERR_INVALID_ARG, "moe_sort_by_expert: tokens=%lld topk=%d experts=%d (topk 1..32, experts 1..%d, "
                "tokens * topk <= 2^31 - 512)",
                (long long)num_tokens, topk, num_experts, kMaxExpertsMoe);
  if (flags & ~(uint32_t)NVFP4_FLAG_PDL) return fail(NVFP4_ERR_INVALID_ARG, "moe_sort_by_expert: unknown flags 0x%x", flags);
  const size_t need = moe_sort_workspace_size(num_tokens, num_experts);
  if (workspace_bytes < need)
    return fail(NVFP4_ERR_INVALID_ARG, "moe_sort_by_expert: needs a workspace of %zu bytes (got %zu)", need, workspace_bytes);
  if (!row_offsets || !workspace || (num_tokens > 0 && (!topk_ids || !src_rows || !pos)))
    return fail(NVFP4_ERR_INVALID_ARG, "moe_sort_by_expert: null pointer");
  if (!aligned(row_offsets, 8) || !aligned(topk_ids, 4) || !aligned(src_rows, 4) || !aligned(pos, 4) ||
      !aligned(workspace, 4))
    return fail(NVFP4_ERR_MISALIGNED, "moe_sort_by_expert: row_offsets need 8-B, the int32 arrays 4-B alignment");
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int G = moe_sort_ctas(num_tokens);
  const int tpc = static_cast<int>(ceil_div(num_tokens > 0 ? num_tokens : 1, G));
  const int smem_count = num_experts * 4, smem_place = (1 + kPlaceWarps) * num_experts * 4;
  st = allow_smem(reinterpret_cast<const void *>(moe_place_kernel), smem_place, dev.device);
  if (st != NVFP4_OK) return st;
  const bool pdl = (flags & NVFP4_FLAG_PDL) != 0;
  cudaError_t e = launch(moe_count_kernel, dim3(G), dim3(256), smem_count, (cudaStream_t)stream, pdl, 1, topk_ids,
                         static_cast<int>(num_tokens), topk, num_experts, tpc, workspace, dev.status);
  if (e == cudaSuccess)
    e = launch(moe_place_kernel, dim3(G), dim3(kPlaceWarps * 32), smem_place, (cudaStream_t)stream, pdl, 1, topk_ids,
               static_cast<int>(num_tokens), topk, num_experts, tpc, workspace, row_offsets, src_rows, pos);
  return check_launch(e, "moe_sort_by_expert");
}

extern "C" nvfp4_status_t moe_gather_rows(const void *x, int64_t num_tokens, int64_t h, int64_t ldx,
                                          const int32_t *src_rows, int64_t rows, void *out, uint32_t flags,
                                          nvfp4_stream_t stream) {
  clear_error();
  if (num_tokens < 0 || rows < 0 || h <= 0 || h % 8 || ldx < h || ldx % 8)
    return fail(NVFP4_ERR_INVALID_ARG, "moe_gather_rows: tokens=%lld rows=%lld h=%lld ldx=%lld (h, ldx multiples of 8)",
                (long long)num_tokens, (long long)rows, (long long)h, (long long)ldx);
  if (flags & ~(uint32_t)NVFP4_FLAG_PDL) return fail(NVFP4_ERR_INVALID_ARG, "moe_gather_rows: unknown flags 0x%x", flags);
  if (rows == 0) return NVFP4_OK;
  if (!x || !src_rows || !out) return fail(NVFP4_ERR_INVALID_ARG, "moe_gather_rows: null pointer");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(src_rows, 4))
    return fail(NVFP4_ERR_MISALIGNED, "moe_gather_rows: x and out need 16-B, src_rows 4-B alignment");
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t pieces = h / 8;
  const int grid = moe_grid(rows * pieces, dev.sm_count, kMoveBlocksPerSm);
  auto kern = fits_i32_loop(rows * pieces, grid * 256LL) ? moe_gather_kernel<int> : moe_gather_kernel<int64_t>;
  cudaError_t e = launch(kern, dim3(grid), dim3(256), 0,
                         (cudaStream_t)stream, (flags & NVFP4_FLAG_PDL) != 0, 1, static_cast<const uint4 *>(x),
                         ldx / 8, num_tokens, src_rows, rows, pieces, static_cast<uint4 *>(out), dev.status);
  return check_launch(e, "moe_gather_rows");
}

extern "C" nvfp4_status_t moe_combine(const void *y, int64_t rows, const int32_t *pos, const float *weights,
                                      int64_t num_tokens, int topk, int64_t h, void *out, uint32_t flags,
                                      nvfp4_stream_t stream) {
  clear_error();
  if (num_tokens < 0 || rows < 0 || topk < 1 || h <= 0 || h % 8)
    return fail(NVFP4_ERR_INVALID_ARG, "moe_combine: tokens=%lld rows=%lld topk=%d h=%lld (h a multiple of 8)",
                (long long)num_tokens, (long long)rows, topk, (long long)h);
  if (flags & ~(uint32_t)NVFP4_FLAG_PDL) return fail(NVFP4_ERR_INVALID_ARG, "moe_combine: unknown flags 0x%x", flags);
  if (num_tokens == 0) return NVFP4_OK;
  if (!y || !pos || !weights || !out) return fail(NVFP4_ERR_INVALID_ARG, "moe_combine: null pointer");
  if (!aligned(y, 16) || !aligned(out, 16) || !aligned(pos, 4) || !aligned(weights, 4))
    return fail(NVFP4_ERR_MISALIGNED, "moe_combine: y and out need 16-B, pos and weights 4-B alignment");
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t pieces = h / 8;
  const int grid = moe_grid(num_tokens * pieces, dev.sm_count, kMoveBlocksPerSm);
  auto kern = fits_i32_loop(num_tokens * pieces, grid * 256LL) ? moe_combine_kernel<int> : moe_combine_kernel<int64_t>;
  cudaError_t e = launch(kern, dim3(grid), dim3(256), 0,
                         (cudaStream_t)stream, (flags & NVFP4_FLAG_PDL) != 0, 1, static_cast<const uint4 *>(y), rows,
                         pos, weights, num_tokens, topk, pieces, static_cast<uint4 *>(out), dev.status);
  return check_launch(e, "moe_combine");
}

namespace {
// Which per-expert quantiser runs (positions: one thread per scale position; else one warp per
// scale row).
constexpr bool kPosQuant = true;


// src_rows != nullptr: row r of the input is row src_rows[r] of x [tokens, k] (gather fused in).
nvfp4_status_t expert_quant(const char *name, bool silu, const void *x, int64_t t, int64_t k, int64_t ldx,
                            const int64_t *row_offsets, int num_experts, const float *gs, uint8_t *q, uint8_t *sf,
                            size_t sf_bytes, uint32_t flags, nvfp4_stream_t stream,
                            const int32_t *src_rows = nullptr, int64_t tokens = 0) {
  clear_error();
  if (t < 0 || k <= 0 || k >= (1LL << 31)) return fail(NVFP4_ERR_INVALID_ARG, "%s: t=%lld k=%lld", name, (long long)t, (long long)k);
  if (k % 16) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: k=%lld is not a multiple of 16", name, (long long)k);
  const int64_t width = silu ? 2 * k : k;
  if (ldx < width || ldx % 8)
    return fail(NVFP4_ERR_MISALIGNED, "%s: ldx=%lld (need ldx >= %lld, ldx %% 8 == 0)", name, (long long)ldx, (long long)width);
  if (num_experts < 1 || num_experts > kMaxExpertsMoe)
    return fail(NVFP4_ERR_INVALID_ARG, "%s: num_experts=%d (1..%d)", name, num_experts, kMaxExpertsMoe);
  if (flags & ~(uint32_t)(NVFP4_FLAG_PDL | NVFP4_FLAG_DEBUG_TIMEOUT))
    return fail(NVFP4_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags);
  const int64_t cp = round_up(k / 16, 4);
  const size_t need = static_cast<size_t>((round_up(t, 128) + 128LL * num_experts) * cp);
  if (sf_bytes < need) return fail(NVFP4_ERR_INVALID_ARG, "%s: sf_bytes=%zu < %zu", name, sf_bytes, need);
  if (t == 0) return NVFP4_OK;
  if (!x || !row_offsets || !gs || !q || !sf) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", name);
  if (src_rows && !aligned(src_rows, 4)) return fail(NVFP4_ERR_MISALIGNED, "%s: src_rows needs 4-B alignment", name);
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(sf, 16) || !aligned(row_offsets, 8) || !aligned(gs, 4))
    return fail(NVFP4_ERR_MISALIGNED, "%s: x 16-B, q 8-B, sf 16-B, row_offsets 8-B, gs 4-B alignment", name);
  DeviceInfo dev;
  nvfp4_status_t st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t cap_rows = static_cast<int64_t>(sf_bytes) / cp / 128 * 128;
  const int64_t scale_rows = round_up(t, 128) + 128LL * num_experts;  // bound of sum_e round_up(M_e, 128)
  if (src_rows && scale_rows * cp >= (1LL << 31))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: (rows + 128 experts) * k/16 >= 2^31 positions", name);
  if (kPosQuant && scale_rows * cp < (1LL << 31)) {
    auto kern = src_rows ? expert_quant_pos_kernel<false, true>
                         : (silu ? expert_quant_pos_kernel<true, false> : expert_quant_pos_kernel<false, false>);
    // Exactly the resident blocks per SM: every block pays the prologue (offsets, prefix, expert
    // table) once and walks its share of positions, which measured faster than 16 or twice the
    // resident blocks per SM (plain 32.8 -> 30.7 us, gathered 41.0 -> 39.7, SiLU 47.1 -> 45.1 at
    // 128 experts, 32768 rows).
    const int64_t blocks = ceil_div(scale_rows * cp, 256);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * resident_blocks(reinterpret_cast<const void *>(kern), 256);
    cudaError_t e = launch(kern, dim3(static_cast<int>(blocks < cap ? blocks : cap)), dim3(256), 0,
                           (cudaStream_t)stream, (flags & NVFP4_FLAG_PDL) != 0, 1, static_cast<const __nv_bfloat16 *>(x),
                           t, static_cast<int>(k / 16), ldx, silu ? k : static_cast<int64_t>(0), row_offsets, num_experts,
                           gs, q, sf, cap_rows, static_cast<int>(cp), src_rows, tokens, dev.status);
    return check_launch(e, name);
  }
  auto kern = silu ? expert_quant_kernel<true> : expert_quant_kernel<false>;
  cudaError_t e = launch(kern, dim3(moe_grid(scale_rows * 32, dev.sm_count)), dim3(256), 0, (cudaStream_t)stream,
                         (flags & NVFP4_FLAG_PDL) != 0, 1, static_cast<const __nv_bfloat16 *>(x), t,
                         static_cast<int>(k / 16), ldx, silu ? k : static_cast<int64_t>(0), row_offsets, num_experts,
                         gs, q, sf, cap_rows, static_cast<int>(cp));
  return check_launch(e, name);
}
}  // namespace

extern "C" nvfp4_status_t nvfp4_quantize_experts(const void *x, int64_t t, int64_t k, int64_t ldx,
                                                 const int64_t *row_offsets, int num_experts, const float *gs,
                                                 uint8_t *q, uint8_t *sf, size_t sf_bytes, uint32_t flags,
                                                 nvfp4_stream_t stream) {
  return expert_quant("nvfp4_quantize_experts", false, x, t, k, ldx, row_offsets, num_experts, gs, q, sf, sf_bytes,
                      flags, stream);
}

extern "C" nvfp4_status_t nvfp4_gather_quantize_experts(const void *x, int64_t num_tokens, int64_t k, int64_t ldx,
                                                        const int32_t *src_rows, int64_t rows,
                                                        const int64_t *row_offsets, int num_experts, const float *gs,
                                                        uint8_t *q, uint8_t *sf, size_t sf_bytes, uint32_t flags,
                                                        nvfp4_stream_t stream) {
  clear_error();
  if (num_tokens < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gather_quantize_experts: num_tokens=%lld", (long long)num_tokens);
  if (rows > 0 && !src_rows) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_gather_quantize_experts: null pointer");
  return expert_quant("nvfp4_gather_quantize_experts", false, x, rows, k, ldx, row_offsets, num_experts, gs, q, sf,
                      sf_bytes, flags, stream, src_rows, num_tokens);
}

extern "C" nvfp4_status_t nvfp4_silu_mul_quantize_experts(const void *x, int64_t t, int64_t inter, int64_t ldx,
                                                          const int64_t *row_offsets, int num_experts,
                                                          const float *gs, uint8_t *q, uint8_t *sf, size_t sf_bytes,
                                                          uint32_t flags, nvfp4_stream_t stream) {
  return expert_quant("nvfp4_silu_mul_quantize_experts", true, x, t, inter, ldx, row_offsets, num_experts, gs, q, sf,
                      sf_bytes, flags, stream);
}
