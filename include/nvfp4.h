/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 / MXFP4 block-scaled GEMM library.
 *
 * Operations (each entry point cites the passage that defines it):
 *   nvfp4_quantize      bf16 -> NVFP4 (packed e2m1 + e4m3 scale per 16, 128x4 swizzled scales)
 *   nvfp4_gemm          D[M,N] = alpha * deq(A) deq(B)^T, bf16 out, fp32 accumulation
 *                       (+ nvfp4_gemm_plan, nvfp4_gemm_workspace_size, nvfp4_gemm_noalloc)
 *   nvfp4_quantize_gemm nvfp4_quantize of the activation fused into nvfp4_gemm (M <= 256)
 *   mxfp4_quantize      bf16 -> MXFP4 (packed e2m1 + ue8m0 scale per 32), optionally grouped by expert
 *   mxfp4_grouped_gemm  per-expert D_e = alpha * deq(A_e) deq(B_e)^T for MoE experts
 *   sf_swizzle          row-major scale matrix <-> 128x4 swizzled layout
 *   nvfp4_sf_convert_layout  128x4 ("SM100") <-> SM103 scale layout
 *   MoE steps           moe_sort_by_expert, moe_gather_rows, nvfp4_quantize_experts,
 *                       nvfp4_gather_quantize_experts (the two fused),
 *                       nvfp4_silu_mul_quantize_experts, nvfp4_grouped_gemm, moe_combine
 *   sizes and status    nvfp4_sf_bytes, mxfp4_grouped_sf_bytes, moe_sort_workspace_size,
 *                       nvfp4_check_status, nvfp4_last_error
 *
 * Sources ("page, section"):
 *   [vLLM-SM103]  vLLM fork compare view "add pdl" (sm103 branch)
 *   [FI-4865]     FlashInfer PR 4865 "perf(gemm): optimize SM103 CuTe DSL mm_fp4 kernel"
 *   [FI-4466]     FlashInfer PR 4466 "sm100 cute_dsl w4a16 gemm" (follow-up PR 4620 text)
 *   [vLLM-51158]  vLLM PR 51158 "Enable CUTLASS MXFP4 W4A4 MoE on SM12x"
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library never
 *     allocates device memory (nvfp4_gemm_noalloc's scratch is a static array of the library)
 *     and keeps no pointer after the call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Arguments are validated on the host before anything is enqueued.  On error nothing
 *     is launched, the status is returned and nvfp4_last_error() describes it.
 *   - Sizes of zero rows are legal and enqueue nothing.
 *   - The current device must be compute capability 10.3 (sm_103).
 *   - Packed FP4: element 2t of a row is the low nibble of byte t, element 2t+1 the high one.
 *   - 128x4 scale layout: a scale matrix of R rows and C scale columns is stored as
 *     round_up(R,128) * round_up(C,4) bytes; scale (r, j) sits at byte
 *       ((r/128) * (round_up(C,4)/4) + j/4) * 512 + (r%32)*16 + ((r/32)%4)*4 + j%4
 *     ([vLLM-SM103] nvfp4_quant_kernels.cu "Scale factor layout conversion: SM100 <-> SM103",
 *     SM100 offset; nvfp4_utils.cuh tile base).  Padding bytes must hold 0x00 (the
 *     quantisers write them so).
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *nvfp4_stream_t;

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum value */
  NVFP4_ERR_MISALIGNED = 2,         /* pointer or stride alignment rule broken */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 3,  /* divisibility rule broken (K % 32, N % 32, ...) */
  NVFP4_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103 */
  NVFP4_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed (message has the name) */
  NVFP4_ERR_TIMEOUT = 6             /* a kernel gave up a bounded wait (nvfp4_check_status) */
} nvfp4_status_t;

/* Launch flags (bitwise OR). */
enum {
  /* Launch with programmatic dependent launch (cudaLaunchAttributeProgrammaticStreamSerialization):
   * the kernel may start while the previous kernel on the stream is still running.  Every
   * kernel of this library waits (griddepcontrol.wait) before it reads an input that a
   * predecessor may produce or writes any output, and signals its own dependents
   * (griddepcontrol.launch_dependents) once its input reads are issued.  Exception, stated
   * per entry point: nvfp4_gemm and mxfp4_grouped_gemm may read the weight operand B and its
   * scales before the wait, so B must not be written by the kernels it overlaps.
   * [vLLM-SM103] summary.md "What is PDL?", nvfp4_quant_kernels.cu "Host entry: SM103
   * activation quantization" (use_pdl). */
  NVFP4_FLAG_PDL = 1u << 0,
  /* Scale buffers in the SM103 layout instead of the 128x4 ("SM100") one: nvfp4_quantize writes
   * its scales, nvfp4_gemm / nvfp4_gemm_noalloc read both sfa and sfb, in that layout.  Same
   * 512-byte tiles in the same order; inside a tile, row m = m4b + 4*m4a + 16*m8 and scale
   * column k sit at m8*16 + m4a*128 + m4b*4 + k.  [vLLM-SM103] nvfp4_quant_kernels.cu "Scale
   * factor layout conversion: SM100 <-> SM103", nvfp4_utils.cuh (SM103 swizzled SF offset).
   * Not accepted by the MXFP4 entry points. */
  NVFP4_FLAG_SF_SM103 = 1u << 2,
  /* Short (about 20 ms) limit on every pipeline wait instead of the default (about 10 s);
   * for tests of the timeout path. */
  NVFP4_FLAG_DEBUG_TIMEOUT = 1u << 8,
  /* Test hook of the time-out path (GEMMs only, honoured only together with
   * NVFP4_FLAG_DEBUG_TIMEOUT): the loader posts the byte count of the first K stage of each CTA
   * but issues none of its copies, so the wait for that stage runs out.  The kernel then records
   * the time-out (nvfp4_check_status returns NVFP4_ERR_TIMEOUT), drains its bounded waits, frees
   * its tensor memory and exits; the output is undefined.  Nothing is read or written out of
   * bounds. */
  NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD = 1u << 9
};

/* Message for the last error on the calling thread ("" when the last call succeeded). */
const char *nvfp4_last_error(void);

/* Bytes of a swizzled scale buffer for `rows` rows of `k` elements with one scale per
 * `sf_vec` (16 for NVFP4, 32 for MXFP4): round_up(rows,128) * round_up(k/sf_vec, 4).
 * Returns 0 for invalid arguments.  Host only. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t k, int sf_vec);

/* Bytes of the grouped MXFP4 scale buffer that mxfp4_quantize writes for `total_rows` rows
 * split over `num_experts` experts: an upper bound of sum_e round_up(M_e,128) rows, namely
 * (round_up(total_rows,128) + 128*num_experts) * round_up(k/32,4).  Host only. */
size_t mxfp4_grouped_sf_bytes(int64_t total_rows, int num_experts, int64_t k);

/* NVFP4 activation quantisation.
 * Source: [vLLM-SM103] nvfp4_quant_kernels.cu "SM103 (B300) activation quantization kernel"
 * (one fp32 global scale, a scale per 16 elements of a row, packed e2m1 out, swizzled scales,
 * padded scale rows/columns quantised from zero input) and test_nvfp4_quant.py (global scale
 * = 448*6/amax).  Per 16-element block, in fp32 with round-to-nearest-even on every step:
 *   s = (gs*amax)/6; sc = e4m3_satfinite(s); inv = sd ? gs/sd : 0 (sd = value of sc);
 *   q_i = e2m1_satfinite(x_i * inv) (the sign of a zero result is kept).
 *   x        bf16 [m, k], row stride `ldx` elements (ldx >= k, ldx % 8 == 0), 16-B aligned
 *   gs       device fp32 scalar (global scale), 4-B aligned
 *   q        uint8 [m, k/2] row-major, 8-B aligned
 *   sf       uint8 [nvfp4_sf_bytes(m, k, 16)], 16-B aligned; every byte is written
 *   k % 16 == 0.  Reads x/gs and writes q/sf only after the PDL wait. */
nvfp4_status_t nvfp4_quantize(const void *x, int64_t m, int64_t k, int64_t ldx, const float *gs,
                              uint8_t *q, uint8_t *sf, uint32_t flags, nvfp4_stream_t stream);

/* MXFP4 quantisation ("e2m1 data with e8m0 scale per 32", [vLLM-51158] "Changes",
 * mxfp4_experts_quant.cu).  Per 32-element block: s = amax/6 (fp32); scale = smallest power
 * of two >= s (ue8m0 code clamped to [0,254], 0 for an all-zero block);
 * q_i = e2m1_satfinite(x_i * 2^(127-code)).
 *   x            bf16 [t, k], row stride ldx (ldx >= k, ldx % 8 == 0), 16-B aligned
 *   row_offsets  NULL for one dense scale block of round_up(t,128) rows; otherwise a DEVICE
 *                int64 [num_experts+1] array, non-decreasing, row_offsets[0] == 0,
 *                row_offsets[num_experts] == t: rows of expert e are row_offsets[e] ..
 *                row_offsets[e+1]-1 and their scales form their own zero-padded 128-row
 *                block starting at scale row sum_{j<e} round_up(M_j,128).
 *   q            uint8 [t, k/2]; sf uint8 [sf_bytes] (16-B aligned), sf_bytes >=
 *                nvfp4_sf_bytes(t,k,32) (dense) or mxfp4_grouped_sf_bytes(t,E,k) (grouped).
 *   k % 32 == 0, 1 <= num_experts <= 1024 when row_offsets != NULL.
 *   Offsets that break the rules above are a caller error; the kernel never writes outside
 *   q[0..t) rows or sf[0..sf_bytes). */
nvfp4_status_t mxfp4_quantize(const void *x, int64_t t, int64_t k, int64_t ldx,
                              const int64_t *row_offsets, int num_experts, uint8_t *q, uint8_t *sf,
                              size_t sf_bytes, uint32_t flags, nvfp4_stream_t stream);

/* The tile configuration nvfp4_gemm picks for a shape (M-based selector, [vLLM-SM103]
 * nvfp4_scaled_mm_kernels.cu "SM103 Dispatch"; narrow tiles for small M, [FI-4865]
 * "Reviewer Notes").  Up to 256 tokens the weight fills the MMA's 128-row slot and K is split
 * inside clusters, except where 256 x 256 CTA-pair tiles fill a quarter of the pairs, or where K
 * is short (4096 <= N <= 16384 and K <= 2048 from 17 tokens, K <= 4096 from 129): there whole
 * 128 x 128 tiles run.
 * Host only. */
typedef struct {
  int swap_ab;   /* 1: the weight B fills the 128-row MMA slot and tokens the N slot */
  int tile_m;    /* rows of the MMA tile (128) */
  int tile_n;    /* MMA N */
  int splits;    /* K splits reduced inside a thread-block cluster (1 = none) */
  int stages;    /* shared-memory pipeline depth */
  int ctas;      /* CTAs launched */
  int dp_tiles;  /* output tiles each computed whole by one CTA */
  int sk_tiles;  /* output tiles after those whose K stages are split stream-K over all CTAs */
} nvfp4_gemm_plan_t;
nvfp4_status_t nvfp4_gemm_plan(int64_t m, int64_t n, int64_t k, nvfp4_gemm_plan_t *plan);

/* Bytes of device workspace nvfp4_gemm needs for this shape on the current device (0 when the
 * plan splits no tile).  Host only.  The split-K reduction is the library's own design (the
 * pages' kernels pick split-K for small M but do not describe how partials are added): the
 * workspace holds one arrival counter per split tile followed by two fp32 partial-tile slots
 * of 128 x tile_n per CTA. */
nvfp4_status_t nvfp4_gemm_workspace_size(int64_t m, int64_t n, int64_t k, size_t *bytes);

/* NVFP4 block-scaled GEMM with bf16 output.
 * Source: [vLLM-SM103] nvfp4_scaled_mm_kernels.cu "SM103 Entry Point" (A [M,K/2] packed e2m1
 * row-major, B [N,K/2] packed e2m1 K-major, scale_a/scale_b e4m3 in the 128x4 layout padded to
 * [round_up(rows,128), round_up(K/16,4)], alpha fp32 [1], k % 32 == 0, n % 32 == 0);
 * [FI-4865] "2. Alpha epilogue bug" (alpha multiplies the fp32 accumulator, then ONE
 * conversion to bf16) and "3. Restore 256-bit stores" (D compact N-major, 32-B aligned).
 *   D[m,n] = bf16( alpha * sum_k e2m1(A[m,k]) e4m3(sfa[m,k/16]) e2m1(B[n,k]) e4m3(sfb[n,k/16]) )
 *   a      uint8 [m, k/2], 32-B aligned         sfa  nvfp4_sf_bytes(m,k,16) bytes, 16-B aligned
 *   b      uint8 [n, k/2], 32-B aligned         sfb  nvfp4_sf_bytes(n,k,16) bytes, 16-B aligned
 *   alpha  device fp32 scalar, 4-B aligned       d    bf16 [m, n] row-major, 32-B aligned
 *   workspace    device buffer of at least nvfp4_gemm_workspace_size(m,n,k) bytes, 256-B
 *                aligned (may be NULL when that size is 0).  It must be zero-filled before its
 *                first use; every call that completes leaves it zero again, so one zeroing
 *                serves any number of calls.  Calls that can run at the same time (other
 *                streams) need separate workspaces: the kernel's counters and partial tiles
 *                would race.  After a call that reported NVFP4_ERR_TIMEOUT, zero it again.
 *   n % 32 == 0, k % 32 == 0, m, n, k < 2^31.
 * The output does not depend on timing: split tiles are added in a fixed order.
 * With NVFP4_FLAG_PDL, b and sfb may be read before the wait for the preceding kernel; the
 * workspace is touched only after that wait. */
nvfp4_status_t nvfp4_gemm(const uint8_t *a, const uint8_t *sfa, const uint8_t *b, const uint8_t *sfb,
                          const float *alpha, void *d, int64_t m, int64_t n, int64_t k,
                          void *workspace, size_t workspace_bytes, uint32_t flags,
                          nvfp4_stream_t stream);

/* nvfp4_quantize fused into nvfp4_gemm: D = nvfp4_gemm(nvfp4_quantize(x, gs_x), b), with the
 * activation quantised inside the GEMM kernel, so its codes and scales never go through global
 * memory and one launch replaces two.  Not an operation of the pages; it is the "quantise in
 * the GEMM's prologue" extension of [vLLM-SM103] "add pdl" (the PDL edge between the two).
 * The result is bit-identical to the two calls: every 16-element block is quantised with the
 * same arithmetic as nvfp4_quantize and the MMAs consume it in the same order.
 *   x      bf16 [m, k] row-major, row stride ldx >= k elements, 16-B aligned, ldx % 8 == 0
 *   gs_x   device fp32 scalar: x's global scale, as nvfp4_quantize's
 *   b, sfb, alpha, d, workspace, flags, stream: as nvfp4_gemm (NVFP4_FLAG_SF_SM103: sfb is in
 *          the SM103 layout); these plans split K inside clusters and need no workspace.
 *   1 <= m <= 256 (the weight-streaming plans, where each CTA quantises the token rows it
 *   needs; this call takes one for every such m, also where nvfp4_gemm_plan reports another
 *   kind for nvfp4_gemm); larger m: NVFP4_ERR_UNSUPPORTED_SHAPE, nothing launched (quantise
 *   separately).
 *   Every CTA that shares a token tile quantises it again (once per 128 weight rows), so the
 *   fused call is faster than the PDL-chained pair only for a few tokens (measured on GB300,
 *   N=4096, K=7168, cold weights: M=1 3 % faster, M=4 even, M >= 16 slower).
 * With NVFP4_FLAG_PDL, b and sfb may be read before the wait for the preceding kernel; x after it.
 */
nvfp4_status_t nvfp4_quantize_gemm(const void *x, int64_t ldx, const float *gs_x, const uint8_t *b,
                                   const uint8_t *sfb, const float *alpha, void *d, int64_t m, int64_t n,
                                   int64_t k, void *workspace, size_t workspace_bytes, uint32_t flags,
                                   nvfp4_stream_t stream);

/* nvfp4_gemm without a workspace argument: when the plan splits tiles stream-K, the partial
 * tiles and arrival counters go to a static 20 MiB device array inside the library instead of a
 * caller buffer.  The pages have no counterpart of this entry point: it exists for callers that
 * cannot allocate or hold device memory for a workspace at call time, such as a plugin inside an
 * inference engine whose device memory is planned once up front, or code on a latency path where
 * a cudaMalloc would synchronise the device.
 *   Arguments, layouts, alignment and errors are those of nvfp4_gemm.  The call never allocates.
 *   Shapes whose workspace (nvfp4_gemm_workspace_size) exceeds the array (20 MiB + 4 KiB) are
 *   refused with NVFP4_ERR_UNSUPPORTED_SHAPE; every plan the selector makes on a GPU of up to
 *   160 SMs fits (the largest: 80 split tiles on 160 CTAs, 20 MiB + 512 bytes).
 *   The array is shared by every call on the device: calls that may overlap (other streams,
 *   other threads) race on it and must not use this entry point concurrently.
 *   The array's address is looked up (cudaGetSymbolAddress) on the first call on each device,
 *   and again on the first call after the device got a new context (a device reset); a caller
 *   that records work for later replay should make one call before it starts recording.
 *   The arrival counters must read zero when the kernel starts: before each launch of a split
 *   plan this entry point enqueues a one-CTA kernel on `stream` that clears them (so a call
 *   after one that timed out starts clean); the partial-tile slots need no initialisation.
 *   That kernel takes the call's NVFP4_FLAG_PDL too: it waits for the preceding kernel before
 *   clearing, while the GEMM starts beside it and streams its weight as nvfp4_gemm would. */
nvfp4_status_t nvfp4_gemm_noalloc(const uint8_t *a, const uint8_t *sfa, const uint8_t *b, const uint8_t *sfb,
                                  const float *alpha, void *d, int64_t m, int64_t n, int64_t k,
                                  uint32_t flags, nvfp4_stream_t stream);

/* MXFP4 grouped (MoE) GEMM: for every expert e, D[rows of e, :] = alpha * deq(A_e) deq(B_e)^T.
 * The kernel checks row_offsets on the device (row_offsets[0] == 0, row_offsets[E] == t,
 * non-decreasing); if they are malformed it does no work and nvfp4_check_status reports
 * NVFP4_ERR_INVALID_ARG.
 * Source: [vLLM-51158] "Changes" (CUTLASS MXFP4 grouped GEMM over experts; SM10x/SM12x share
 * the block-scaled scale layout) and [vLLM-SM103] ops.h (expert offsets as arguments).
 *   a            uint8 [t, k/2] (rows sorted by expert), 32-B aligned
 *   sfa          grouped ue8m0 scales as mxfp4_quantize(row_offsets) writes them, 16-B aligned
 *   row_offsets  DEVICE int64 [num_experts+1] (same rules as mxfp4_quantize)
 *   b            uint8 [num_experts, n, k/2], 32-B aligned
 *   sfb          uint8 [num_experts, nvfp4_sf_bytes(n,k,32)] (each expert's block swizzled)
 *   alpha        device fp32 scalar or NULL for 1.0
 *   d            bf16 [t, n] row-major, 32-B aligned
 *   n % 32 == 0, k % 32 == 0, 1 <= num_experts <= 1024.
 * With NVFP4_FLAG_PDL, b and sfb may be read before the wait for the preceding kernel. */
nvfp4_status_t mxfp4_grouped_gemm(const uint8_t *a, const uint8_t *sfa, const int64_t *row_offsets,
                                  int num_experts, const uint8_t *b, const uint8_t *sfb,
                                  const float *alpha, void *d, int64_t t, int64_t n, int64_t k,
                                  uint32_t flags, nvfp4_stream_t stream);

/* ---------------------------------------------------------------- MoE steps (NVFP4)
 * The steps around the grouped GEMMs of an NVFP4 mixture-of-experts layer:
 *   moe_sort_by_expert -> moe_gather_rows -> nvfp4_quantize_experts -> nvfp4_grouped_gemm (gate+up)
 *   -> nvfp4_silu_mul_quantize_experts -> nvfp4_grouped_gemm (down) -> moe_combine.
 * [vLLM-SM103] ops.h / torch_bindings.cpp name scaled_fp4_experts_quant,
 * silu_and_mul_scaled_fp4_experts_quant (arguments input_offset_by_experts,
 * output_scale_offset_by_experts) and cutlass_fp4_group_mm; [vLLM-51158] "Changes" describes the
 * experts-quantise + grouped-GEMM structure.  The pages give names and arguments only; the
 * definitions below are this library's reading of them. */

/* Bytes of device workspace moe_sort_by_expert needs (one int32 count per CTA and expert).  Host only. */
size_t moe_sort_workspace_size(int64_t num_tokens, int num_experts);

/* Stable sort of routed (token, slot) pairs by expert.
 *   topk_ids     DEVICE int32 [num_tokens, topk], expert of each slot (0 <= id < num_experts;
 *                other values are dropped (pos = -1) and make nvfp4_check_status report
 *                NVFP4_ERR_INVALID_ARG)
 *   row_offsets  DEVICE int64 [num_experts + 1] out: rows of expert e are row_offsets[e] ..
 *                row_offsets[e+1]-1 of the permuted order (the grouped kernels' row_offsets)
 *   src_rows     DEVICE int32 [num_tokens * topk] out: token of each permuted row
 *   pos          DEVICE int32 [num_tokens, topk] out: permuted row of each (token, slot)
 *   workspace    DEVICE, 4-B aligned, workspace_bytes >= moe_sort_workspace_size(); no
 *                initialisation needed (every byte used is written first)
 * Inside an expert, rows keep (token, slot) row-major order.  1 <= topk <= 32,
 * 1 <= num_experts <= 1024, num_tokens * topk <= 2^31 - 512.  Two kernels over ceil(num_tokens/32) CTAs (at most 1024). */
nvfp4_status_t moe_sort_by_expert(const int32_t *topk_ids, int64_t num_tokens, int topk, int num_experts,
                                  int64_t *row_offsets, int32_t *src_rows, int32_t *pos, int32_t *workspace,
                                  size_t workspace_bytes, uint32_t flags, nvfp4_stream_t stream);

/* Row gather (permutation into expert order): out[r, :] = x[src_rows[r], :] for r < rows.
 *   x        bf16 [num_tokens, h], row stride ldx (ldx >= h, ldx % 8 == 0), 16-B aligned
 *   out      bf16 [rows, h] contiguous, 16-B aligned; h % 8 == 0
 * A src_rows entry outside [0, num_tokens) is skipped (that row is not written) and makes
 * nvfp4_check_status report NVFP4_ERR_INVALID_ARG. */
nvfp4_status_t moe_gather_rows(const void *x, int64_t num_tokens, int64_t h, int64_t ldx, const int32_t *src_rows,
                               int64_t rows, void *out, uint32_t flags, nvfp4_stream_t stream);

/* Per-expert NVFP4 quantisation (scaled_fp4_experts_quant): rows of expert e (row_offsets as
 * moe_sort_by_expert writes them) are quantised as nvfp4_quantize does with global scale gs[e];
 * expert e's scales form their own zero-padded 128-row block starting at scale row
 * sum_{j<e} round_up(M_j, 128) of a round_up(k/16, 4)-column 128x4-swizzled matrix.
 *   x      bf16 [t, k], row stride ldx, 16-B aligned;  gs  DEVICE fp32 [num_experts]
 *   q      uint8 [t, k/2], 8-B aligned
 *   sf     uint8 [sf_bytes], 16-B aligned, sf_bytes >= (round_up(t,128) + 128*num_experts) *
 *          round_up(k/16, 4)  (the same bound as mxfp4_grouped_sf_bytes with k/16 columns)
 *   k % 16 == 0, 1 <= num_experts <= 1024. */
nvfp4_status_t nvfp4_quantize_experts(const void *x, int64_t t, int64_t k, int64_t ldx, const int64_t *row_offsets,
                                      int num_experts, const float *gs, uint8_t *q, uint8_t *sf, size_t sf_bytes,
                                      uint32_t flags, nvfp4_stream_t stream);

/* moe_gather_rows fused into nvfp4_quantize_experts: row r of the quantised matrix is row
 * src_rows[r] of x, so the gathered bf16 copy is never written.  For src_rows entries in
 * [0, num_tokens) the result (q, sf) is bit-identical to moe_gather_rows(x, src_rows) followed
 * by nvfp4_quantize_experts on its output.  A row whose entry is outside [0, num_tokens) is
 * quantised from zeros and makes nvfp4_check_status report NVFP4_ERR_INVALID_ARG.  The sources
 * define no such call: it joins two of the steps above ([vLLM-SM103] ops.h quantises the
 * already permuted activation with scaled_fp4_experts_quant).
 *   x         bf16 [num_tokens, k], row stride ldx >= k (ldx % 8 == 0), 16-B aligned
 *   src_rows  DEVICE int32 [rows] (as moe_sort_by_expert writes it), 4-B aligned
 *   row_offsets, num_experts, gs, q ([rows, k/2]), sf, sf_bytes: as nvfp4_quantize_experts
 *   with t = rows.  (rows + 128*num_experts) * round_up(k/16,4) < 2^31, else
 *   NVFP4_ERR_UNSUPPORTED_SHAPE (quantise the gathered rows with nvfp4_quantize_experts). */
nvfp4_status_t nvfp4_gather_quantize_experts(const void *x, int64_t num_tokens, int64_t k, int64_t ldx,
                                             const int32_t *src_rows, int64_t rows, const int64_t *row_offsets,
                                             int num_experts, const float *gs, uint8_t *q, uint8_t *sf,
                                             size_t sf_bytes, uint32_t flags, nvfp4_stream_t stream);

/* SiLU-and-mul fused with the per-expert NVFP4 quantisation (silu_and_mul_scaled_fp4_experts_quant).
 * x is bf16 [t, 2*inter] = [gate | up]; the quantised matrix is h [t, inter] with
 *   h = bf16(silu(gate) * up),  silu(g) = g * (1 / (1 + exp(-g)))  in fp32,
 * exp computed by Cody-Waite range reduction and a degree-7 Taylor polynomial, every fp32 step
 * rounded to nearest even (so the result equals "silu_and_mul to bf16, then quantise" done the
 * same way), then h is quantised as nvfp4_quantize_experts does (q [t, inter/2], sf as there
 * with k = inter).  ldx >= 2*inter, inter % 16 == 0. */
nvfp4_status_t nvfp4_silu_mul_quantize_experts(const void *x, int64_t t, int64_t inter, int64_t ldx,
                                               const int64_t *row_offsets, int num_experts, const float *gs,
                                               uint8_t *q, uint8_t *sf, size_t sf_bytes, uint32_t flags,
                                               nvfp4_stream_t stream);

/* NVFP4 grouped (MoE) GEMM (cutlass_fp4_group_mm): D[rows of e, :] = alpha[e] * deq(A_e) deq(B_e)^T.
 *   a      uint8 [t, k/2] rows sorted by expert;  sfa  as nvfp4_quantize_experts writes it
 *   b      uint8 [num_experts, n, k/2];  sfb  uint8 [num_experts, nvfp4_sf_bytes(n, k, 16)]
 *   alpha  DEVICE fp32 [num_experts] (one per expert: 1/(gsA_e * gsB_e)) or NULL for 1.0
 *   d      bf16 [t, n], 32-B aligned;  n % 32 == 0, k % 32 == 0;  1 <= num_experts <= 512 (the
 *          expert tables share the CTA's shared memory with the operand ring: 128 x 256 tiles on a
 *          4-deep ring up to 256 experts, 128 x 128 tiles beyond).
 * Same kernel, other checks and PDL behaviour as mxfp4_grouped_gemm. */
nvfp4_status_t nvfp4_grouped_gemm(const uint8_t *a, const uint8_t *sfa, const int64_t *row_offsets, int num_experts,
                                  const uint8_t *b, const uint8_t *sfb, const float *alpha, void *d, int64_t t,
                                  int64_t n, int64_t k, uint32_t flags, nvfp4_stream_t stream);

/* Weighted combine of the experts' outputs:
 *   out[t, :] = bf16( sum_{j < topk} weights[t, j] * y[pos[t, j], :] )
 * in fp32, slots in order, each product and sum rounded (no fused multiply-add); slots with
 * pos < 0 are skipped (a token with none gets zeros); pos >= rows is skipped too and makes
 * nvfp4_check_status report NVFP4_ERR_INVALID_ARG.
 *   y        bf16 [rows, h] (expert order), 16-B aligned;  pos  DEVICE int32 [num_tokens, topk]
 *   weights  DEVICE fp32 [num_tokens, topk];  out  bf16 [num_tokens, h], 16-B aligned;  h % 8 == 0 */
nvfp4_status_t moe_combine(const void *y, int64_t rows, const int32_t *pos, const float *weights,
                           int64_t num_tokens, int topk, int64_t h, void *out, uint32_t flags,
                           nvfp4_stream_t stream);

/* Scale layout conversion between a row-major scale matrix [rows, cols] (bytes) and the
 * 128x4 swizzled layout of nvfp4_sf_bytes size (swizzle writes the zero padding).
 * Source: [vLLM-SM103] nvfp4_utils.py swizzle_blockscale (pad to (128,4), then block
 * interleave) and the in-tile offset quoted at the top of this header.
 *   to_swizzled = 1: src [rows, cols] row-major -> dst swizzled
 *   to_swizzled = 0: src swizzled -> dst [rows, cols] row-major
 * Buffers must not overlap.  No alignment requirement. */
nvfp4_status_t sf_swizzle(const uint8_t *src, uint8_t *dst, int64_t rows, int64_t cols,
                          int to_swizzled, nvfp4_stream_t stream);

/* Converts a swizzled NVFP4 scale buffer between the 128x4 ("SM100") layout and the SM103
 * layout (see NVFP4_FLAG_SF_SM103): every byte of every 512-byte tile moves to its place in the
 * other layout, padding bytes included.
 * Source: [vLLM-SM103] nvfp4_quant_kernels.cu "Scale factor layout conversion: SM100 <-> SM103"
 * (convert_sf_layout_sm100_to_sm103 / _sm103_to_sm100).
 *   src, dst   uint8 [round_up(rows,128) * round_up(cols,4)], 16-B aligned, must not overlap
 *   rows, cols the scale matrix (cols = K/16 scale columns)
 *   to_sm103   1: SM100 -> SM103, 0: SM103 -> SM100
 * Reads src only after the PDL wait (NVFP4_FLAG_PDL semantics are implied: the kernel always
 * waits, so it is safe after any producer). */
nvfp4_status_t nvfp4_sf_convert_layout(const uint8_t *src, uint8_t *dst, int64_t rows, int64_t cols,
                                       int to_sm103, nvfp4_stream_t stream);

/* Synchronises `stream`, then reads and clears the device status word that kernels set when a
 * bounded pipeline wait gave up, a grouped GEMM found malformed row offsets or a MoE step found
 * an index out of range.  Returns NVFP4_ERR_INVALID_ARG for malformed offsets or indices, NVFP4_ERR_TIMEOUT if a
 * kernel timed out since the last check, NVFP4_ERR_CUDA if the synchronisation failed,
 * NVFP4_OK otherwise.
 * The word is one per device, shared by every stream and thread: the call reports what any of
 * this library's kernels on the current device recorded since the previous check, and a bit
 * that a kernel on another, still-running stream sets between the read and the clear is lost.
 * For an exact account, call it when no other stream of the device has this library's work in
 * flight. */
nvfp4_status_t nvfp4_check_status(nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
