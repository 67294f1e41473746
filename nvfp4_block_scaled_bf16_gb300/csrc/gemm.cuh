// Warp-specialised block-scaled FP4 GEMM for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (vLLM fork compare view "add pdl", nvfp4_scaled_mm_kernels.cu, "SM103 Entry
// Point"; FlashInfer PR 4865, "2. Alpha epilogue bug" and "3. Restore 256-bit stores"):
//   C[i, j] = sum_k deq(A)[i, k] * deq(B)[j, k]   (fp32 accumulation in tensor memory)
//   D       = bf16(alpha * C)                     (alpha on the fp32 value, one conversion)
// A and B are K-major packed e2m1 (two per byte); their scales (ue4m3 per 16 for NVFP4, ue8m0
// per 32 for MXFP4) are in the 128x4 swizzled layout.  The block-scaled MMA reads the scales of
// the 128 rows of a 512-byte tile from 4 tensor-memory columns of each 32-lane quadrant: lane
// 32q+i, column j holds the 4 bytes at tile offset 16*i + 4*j, the same in every quadrant.
//
// CTA = 10 warps (11 in CTA pairs):
//   warp 0      TMA producer (one thread issues every copy): A/B tiles (128-byte swizzle) and
//               scale chunks (bulk copies) into a STAGES-deep shared-memory ring, one mbarrier
//               pair per stage.  A single-tile CTA whose K slice fits the ring ("resident")
//               lands B and both scale slices with one copy each and A stage by stage, the
//               first copies going out before the rest of the CTA is set up; weight-streaming
//               CTAs keep at most `lookahead` stages in flight so cold HBM returns them in order;
//   warp 1      allocates tensor memory; one lane issues the MMAs (K = 64 each; 4 per 256-wide
//               K step), waiting once per K step for its scale slot, commits each scale slot
//               back to the scale writers and each stage back to the producer, and after the
//               last stage of a tile the accumulator to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quadrant, alpha * acc in fp32, one RNE
//               conversion to bf16; dense CTAs that walk whole tiles stage each 32-column chunk
//               in shared memory and write it with one tensor store, the others store 256-bit
//               vectors per row (in the fused-quantisation kernels they first quantise the
//               bf16 activation into the operand-B stages);
//   warps 6..9  scale writers: each waits until the stage's operands (and scales) have landed,
//               reads the scale tiles from shared memory and writes them into its own quadrant
//               of a tensor-memory scale slot with tcgen05.st (one slot per 256-wide K step,
//               SF_SLOTS in a ring; a resident CTA fills one slot per stage with a single
//               hand-off to the MMA lane).  Their arrival is the MMA lane's only wait per K step.
//               Copying the scales with tcgen05.cp from the MMA lane instead was measured to
//               cap a 128x256x256 step at ~840 cycles against 520 of MMA: the copy unit takes
//               ~55 cycles per 512-byte tile and such a step needs 12 of them;
//   warp 10     (pairs only) copies the scales into a ring of their own, ahead of the operands.
// NACC accumulator buffers let the epilogue of tile t overlap the mainloop of tile t+1.
//
// CTA pairs (PAIR, 256 x 256 tiles for large M): a cluster of two CTAs runs cta_group::2 MMAs
// (M = 256, issued by the first CTA; a 256x256x64 MMA occupies the pipe for the same ~128 cycles
// as a 128x256x64 one on a single CTA).  Each CTA stages its 128 rows of A and its 128 rows of B;
// the scales of its A rows and of all 256 B rows go through a separate ring that warp 10 fills
// ahead of the operands.  When K allows, a stage holds two 256-wide K steps, landed with one 3-D
// copy per operand (the copy engine's cost per instruction bounded the one-step stage).  The
// hand-offs across the pair: the second CTA's scale writers and epilogue arrive on the first
// CTA's barriers (the writers only after their own CTA's operands landed, so the first CTA's
// MMA lane needs no other signal from its peer), and the first CTA's commits arrive on both
// CTAs' barriers (multicast).  Arrivals use the default CTA-scope release: a cluster-scope
// release measured 1000-1500 cycles per arrive; every arrival follows the completion of what it
// announces (tcgen05.wait::st / ::ld, a completed barrier).
//
// Work decomposition: each CTA walks a list of segments (tile, K-stage range).
//   - whole tiles: CTA c takes tiles c, c+G, c+2G, ... below dp_tiles (G = grid size; for
//     pairs, cluster c of G/2);
//   - stream-K: the (tile, K stage) units of the sk_tiles tiles after them are cut into G
//     contiguous runs of equal length, one per CTA.  A run that covers only part of a tile
//     stores its fp32 partial tile in a workspace slot; the last CTA to finish the tile (an
//     atomic counter per tile) adds the partials in contributor order -- a fixed order, so the
//     result does not depend on timing -- and writes the bf16 output;
//   - cluster split-K (splits > 1): the CTAs of a (splits, 1, 1) cluster each take a K slice of
//     one tile and add their partials through distributed shared memory, also in a fixed order.
//
// Every mbarrier wait is bounded (WaitCtl).  When one gives up, the CTA records the time-out
// in the device status word, every role leaves its loop, outstanding copies and MMAs are
// drained with bounded waits, and tensor memory is freed before the CTA exits.
#pragma once

#include "ptx.cuh"

namespace nvfp4 {

// Wait sites recorded in the status word when a bounded wait gives up (bit 8 + site).
enum : int {
  kSiteLoadEmpty = 0,   // loader: free ring slot
  kSiteMmaAcc = 1,      // MMA: accumulator drained by the epilogue
  kSiteMmaFull = 2,     // MMA: stage landed
  kSiteMmaScale = 3,    // MMA: scale slot written
  kSiteScaleSlot = 4,   // scale writers: scale slot free
  kSiteScaleFull = 5,   // scale writers: stage landed
  kSiteEpilogue = 6     // epilogue: accumulator complete
};

template <int BN_, int STAGES_, bool MX_, bool MULTI_TILE_ = true, int MIN_BLOCKS_ = 1, bool PAIR_ = false,
          int MAX_EXPERTS_ = 1024, int KS_ = 1>
struct GemmCfg {
  static constexpr int BN = BN_;          // MMA N: rows of operand B per tile
  static constexpr int STAGES = STAGES_;  // shared-memory pipeline depth
  static constexpr bool MX = MX_;         // true: MXFP4 (ue8m0 / 32); false: NVFP4 (ue4m3 / 16)
  // MULTI_TILE: CTAs walk several tiles (whole tiles or stream-K; never swap-AB).  Otherwise the
  // configuration serves swap-AB plans only: one tile per CTA, K split over a cluster.
  static constexpr bool MULTI_TILE = MULTI_TILE_;
  static constexpr bool SWAP_ONLY = !MULTI_TILE_;
  // CTAs per SM the registers are budgeted for (2: consecutive GEMMs of a PDL chain can share
  // the SMs, the next one streaming its weights while this one finishes)
  static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
  // PAIR: a cluster of two CTAs computes one 256 x BN tile with cta_group::2 MMAs issued by the
  // first CTA.  Each CTA stages 128 rows of A and BN/2 rows of B (the MMA reads the other half
  // of B from the peer's shared memory) plus the scales of its A rows and of all BN B rows, and
  // holds its 128 rows of the accumulator.  Per K stage an SM then moves 38 KB through shared
  // memory instead of 54 KB, and shared-memory bandwidth is what bounds the single-CTA tile.
  static constexpr bool PAIR = PAIR_;
  static constexpr int CG = PAIR ? 2 : 1;
  static constexpr int BM = 128;          // MMA M: rows of operand A per tile (per CTA)
  // KS: 256-wide K steps per ring stage.  KS = 2 (CTA pairs) lands two K steps of each operand
  // with one 3-D copy (box of 2 x 128-byte rows): the copy engine's cost per instruction, not
  // its bytes, bounded the pair's stage rate, and this halves the instructions per MMA.
  static constexpr int KS = KS_;
  static constexpr int KSTAGE = 256 * KS;  // K elements per stage
  static constexpr int MMAS = KSTAGE / 64;  // MMAs (K = 64) per full stage
  static constexpr int A_TILE = BM * 128;  // bytes of one 256-wide K step of A (one swizzled tile)
  static constexpr int VEC = MX ? 32 : 16;
  static constexpr int CHUNKS = KSTAGE / VEC / 4;  // 512-byte scale chunks per 128 rows per stage
  static constexpr int SFB_BLOCKS = (BN + 127) / 128;
  static constexpr int A_BYTES = BM * 128 * KS;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // rows of operand B a CTA stages
  static constexpr int B_TILE = B_ROWS * 128;
  static constexpr int B_BYTES = B_TILE * KS;
  static constexpr int SFA_BYTES = CHUNKS * 512;
  static constexpr int SFB_BYTES = SFB_BLOCKS * CHUNKS * 512;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // Tensor-memory scale slots hold one 256-wide K step each (SUB slots per ring stage), so that
  // the scale writers can run ahead of the MMAs by several K steps even when a stage holds two.
  static constexpr int SUB = KS;                     // scale slots per ring stage
  static constexpr int SUB_CHUNKS = CHUNKS / SUB;    // 512-byte chunks per 128 rows per slot
  static constexpr int SFA_COLS = SUB_CHUNKS * 4;
  static constexpr int SFB_COLS = SFB_BLOCKS * SUB_CHUNKS * 4;
  static constexpr int SF_SLOT = SFA_COLS + SFB_COLS;  // columns of one scale slot
  // a second accumulator only helps CTAs that walk several tiles (epilogue of tile t overlaps
  // the mainloop of t+1)
  // (two CTAs per SM share the tensor memory: one accumulator each)
  static constexpr int NACC = (MULTI_TILE_ && MIN_BLOCKS_ == 1 && 2 * BN + 2 * SF_SLOT <= 512) ? 2 : 1;
  static constexpr int SF_COL0 = NACC * BN;
  // Tensor-memory scale slots: one per ring stage for single-tile (swap-AB) CTAs, so a CTA
  // whose K slice fits the ring writes every stage's scales once, with no slot reuse.
  // (at most one group per ring stage: the writers learn that a group is free from the ring
  // barrier of the stage that last read it, which is unambiguous only then)
  static constexpr int SF_SLOTS_FIT = (SF_COL0 + 4 * SF_SLOT <= 512) ? 4 : 2;
  static constexpr int SF_SLOTS = !MULTI_TILE_ ? STAGES : (SF_SLOTS_FIT < STAGES * SUB ? SF_SLOTS_FIT : STAGES * SUB);
  // The slots of one stage form a group with one written / free barrier pair, so that the MMA
  // lane waits and commits once per stage whatever the number of K steps in it.
  static constexpr int SF_GROUPS = SF_SLOTS / SUB;
  static constexpr int TMEM_USED = SF_COL0 + SF_SLOTS * SF_SLOT;
  static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
  static constexpr int RED_BYTES = BM * BN * 4;  // partial tile: cluster split-K buffer, stream-K slot
  static constexpr int MAX_EXPERTS = MAX_EXPERTS_;  // grouped: expert tables in shared memory
  static constexpr int TABLE_BYTES = 3 * (MAX_EXPERTS + 1) * 4;
  static constexpr int CTRL_BYTES = 512;
  // A pair adds warp 10, which copies the scales into a ring of their own (SF_STAGES deep) ahead
  // of the operands, so that writing them to tensor memory is off the operand ring's critical
  // path and the producer issues two copies per stage instead of five.
  static constexpr int SF_STAGES = PAIR ? (KS == 2 ? 2 : 5) : STAGES;
  static constexpr int THREADS = PAIR ? 352 : 320;
  // The ring keeps each operand in a region of its own (stage i of A at A_REGION + i * A_BYTES,
  // and so on), so the stages of one operand are contiguous and a CTA whose whole K slice fits
  // the ring can land an operand's slice with a single copy.
  static constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES) + SF_STAGES * (SFA_BYTES + SFB_BYTES);
  static constexpr int B_REGION = STAGES * A_BYTES;
  static constexpr int SFA_REGION = B_REGION + STAGES * B_BYTES;
  static constexpr int SFB_REGION = SFA_REGION + SF_STAGES * SFA_BYTES;
  // dynamic shared memory: alignment slack, stage ring, barriers, expert tables (grouped only)
  // PUSH_RED (32-wide swap-AB tiles, two CTAs per SM; used from 16 tokens on): the cluster
  // split-K reduction pushes each rank's slice of the partial into that rank's receive buffer
  // with bulk copies completing on the receiver's own barrier, instead of publishing every
  // partial with a cluster-scope release and reading it remotely.  The buffer holds one slice per
  // other rank: with U = BN*32 units of 16 bytes and S <= 8 ranks, (S-1) * ceil(U/S) <= U - U/8
  // + 7 units; it follows the control block.
  static constexpr bool PUSH_RED = !MULTI_TILE_ && BN_ == 32;
  static constexpr int RCV_BYTES = PUSH_RED ? (BN_ * 32 - BN_ * 32 / 8 + 8) * 16 : 0;
  static constexpr int smem_bytes(bool grouped) {
    return 1024 + RING_BYTES + CTRL_BYTES + RCV_BYTES + (grouped ? TABLE_BYTES : 0);
  }
  static constexpr uint32_t IDESC = idesc_block_scaled(PAIR ? 2 * BM : BM, BN, MX, 0);
  // arrivals on the scale-slot-written and accumulator-drained barriers (both CTAs of a pair
  // arrive on the first CTA's)
  static constexpr int SLOT_ARRIVALS = PAIR ? 8 : 4;
  static constexpr int ACC_ARRIVALS = PAIR ? 8 : 4;
  static_assert(TMEM_USED <= 512 && SF_SLOTS <= 8 && SF_SLOTS % SUB == 0, "tensor memory budget, scale-slot barriers");
  static_assert(SF_GROUPS <= STAGES, "a scale group's reuse is read off the ring barriers: at most one per stage");
  static_assert(STAGES <= 7 && SF_STAGES <= 8 && (2 * STAGES + 46) * 8 + 8 * 4 <= CTRL_BYTES,
                "barriers and flags fit the control block");
  static_assert(smem_bytes(false) <= 232448, "shared memory per CTA");
  static_assert(MIN_BLOCKS == 1 || (MIN_BLOCKS * (smem_bytes(false) + 1024) <= 233472 && MIN_BLOCKS * TMEM_COLS <= 512),
                "shared and tensor memory for MIN_BLOCKS CTAs per SM");
  static_assert(RED_BYTES <= RING_BYTES, "split-K buffer must fit in the stage ring");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "MMA N (N = 16 tiles gave wrong results)");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "128-byte swizzle tiles need 1024-byte alignment");
  static_assert(!PAIR || (MULTI_TILE && BN == 256 && !MX), "CTA pairs: NVFP4 256-wide whole tiles only");
  static_assert(KS == 1 || (KS == 2 && MULTI_TILE && !MX), "two K steps per stage: NVFP4 multi-tile CTAs only");
};

struct GemmArgs {
  const uint8_t *sfa;       // scales of operand A (swizzled, 128-row blocks)
  const uint8_t *sfb;       // scales of operand B
  const float *alpha;       // device scalar, or nullptr for 1
  __nv_bfloat16 *d;         // output
  int64_t ldd;              // output row stride (elements)
  int m, n, k;              // operand A rows, operand B rows (per expert when grouped), K
  int swap;                 // 1: D[j][i] = C[i][j] (operand A is the weight)
  int weight_operand;       // launched with PDL: 1 = A, 2 = B is the weight (loaded before the wait)
  int m_tiles, n_tiles, k_tiles, splits;
  int sf_chunks;            // 512-byte scale chunks per 128-row block = round_up(K/VEC, 4) / 4
  const int64_t *row_offsets;  // grouped: [experts + 1] rows of operand A per expert
  int experts;
  int64_t sfb_expert_bytes;    // grouped: bytes of one expert's B scales
  unsigned int *status;
  long long wait_limit;
  int debug_skip_first_load;  // test hook of the time-out path (see NVFP4_FLAG_DEBUG_SKIP_FIRST_LOAD)
  int max_tiles;              // grouped: host bound of the work list, (ceil(t/128) + experts) * n_tiles
  int dp_tiles;               // tiles [0, dp_tiles) are computed whole
  int sk_tiles;               // tiles [dp_tiles, dp_tiles + sk_tiles) are split stream-K
  float *ws;                  // stream-K: 2 partial-tile slots (BM x BN fp32) per CTA
  unsigned int *ws_cnt;       // stream-K: one arrival counter per split tile, zero between calls
  int resident;               // 1: each CTA's K slice (at most nst_max stages) fits the ring and
                              // K % 256 == 0: operand B and both scale slices land with one copy
                              // each, operand A stage by stage (single-tile, non-grouped CTAs)
  int nst_max;                // resident: K stages of the longest slice = z extent of tmB3's box
  int lookahead;              // > 0: at most this many K stages in flight per CTA (stage i + L is
                              // issued once stage i has landed); 0: as many as the ring holds
  int sf_sm103;               // 1: both scale buffers are in the SM103 layout
  int alpha_per_expert;       // grouped: alpha points to one fp32 per expert
  // Fused quantisation (swap-AB plans only; xq == nullptr: off): operand B is the bf16
  // activation xq [n, k] (row stride ldx elements) under global scale *gs_q, quantised to NVFP4
  // inside the kernel instead of loaded; sfb is then unused.
  const __nv_bfloat16 *xq;
  int64_t ldx;
  const float *gs_q;
};

// The 16 scale bytes of 512-byte scale tile `tile` that lane i of a scale writer puts in its
// tensor-memory lane: rows i, i+32, i+64, i+96 (4 consecutive bytes each, one per scale column).
// In the 128x4 layout those are bytes 16i .. 16i+15; in the SM103 layout the word of row m sits
// at ((m/16)%8)*16 + ((m/4)%4)*128 + (m%4)*4, which for m = i + 32q is base(i) + 32q.
__device__ __forceinline__ uint4 ld_sf_lane(uint32_t tile, int lane, int sm103) {
  if (!sm103) return lds128(tile + 16 * lane);
  const uint32_t base = tile + ((lane >> 4) * 16 + ((lane >> 2) & 3) * 128 + (lane & 3) * 4);
  uint4 v;
  asm volatile("ld.shared.b32 %0, [%4];\n ld.shared.b32 %1, [%4+32];\n ld.shared.b32 %2, [%4+64];\n ld.shared.b32 %3, [%4+96];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(base));
  return v;
}

struct TileInfo {
  int a_y, b_y;                // TMA row coordinates of the A and B tiles
  const uint8_t *sfa_blk;      // first chunk of A's 128-row scale block
  const uint8_t *sfb_blk;      // first chunk of B's first 128-row scale block
  int sfb_blocks;              // B scale blocks present (<= SFB_BLOCKS)
  int rows, cols;              // valid rows of A / of B in this tile
  int64_t out_i0, out_j0;      // output coordinates of C[0][0] of the tile (before swap)
  int expert;                  // grouped: the tile's expert
};

// One piece of a CTA's work: K stages [kt0, kt1) of tile `tile`.  n CTAs share the tile (n == 1:
// this CTA computes it whole); this CTA is contributor j, counted from the one that holds K stage
// 0, and c0 is the index of that first contributor (stream-K).
struct Seg {
  int tile, kt0, kt1, j, n, c0;
};

// Segment iterator.  Every role of the CTA walks the same sequence.
struct Work {
  int tile, tile_end, tile_step;  // whole tiles, or the one tile of a cluster split
  int kt_lo, kt_hi, split, splits;
  int64_t u, u_end, units;        // stream-K: this CTA's units [u, u_end) of `units`

  // CTA whose run holds stream-K unit v: run c is [c*units/G, (c+1)*units/G)
  __device__ __forceinline__ int owner(int64_t v) const {
    return static_cast<int>(((v + 1) * gridDim.x + units - 1) / units - 1);
  }
  __device__ __forceinline__ bool next(const GemmArgs &p, Seg &s) {
    if (tile < tile_end) {
      s = Seg{tile, kt_lo, kt_hi, split, splits, 0};
      tile += tile_step;
      return true;
    }
    if (u < u_end) {
      const int kt_n = p.k_tiles;
      const int t = static_cast<int>(u / kt_n);
      const int64_t first = static_cast<int64_t>(t) * kt_n;
      const int kt0 = static_cast<int>(u - first);
      const int kt1 = static_cast<int>(min(static_cast<int64_t>(kt_n), kt0 + (u_end - u)));
      const int c0 = owner(first);
      s = Seg{p.dp_tiles + t, kt0, kt1, static_cast<int>(blockIdx.x) - c0, owner(first + kt_n - 1) - c0 + 1, c0};
      u += kt1 - kt0;
      return true;
    }
    return false;
  }
};

// PAIR: the two CTAs of a cluster walk the same tiles (cluster c takes tiles c, c+G/2, ...).
template <bool GROUPED, bool PAIR = false>
__device__ __forceinline__ Work make_work(const GemmArgs &p, int grouped_tiles) {
  Work w{};
  w.kt_lo = 0;
  w.kt_hi = p.k_tiles;
  w.split = 0;
  w.splits = 1;
  w.u = w.u_end = 0;
  w.units = 1;
  w.tile = PAIR ? blockIdx.x >> 1 : blockIdx.x;
  w.tile_step = PAIR ? gridDim.x >> 1 : gridDim.x;
  if (GROUPED) {
    w.tile_end = grouped_tiles;
  } else if (p.splits > 1) {
    w.tile = blockIdx.x / p.splits;
    w.tile_end = w.tile + 1;
    w.tile_step = 1;
    w.split = blockIdx.x % p.splits;
    w.splits = p.splits;
    w.kt_lo = w.split * p.k_tiles / p.splits;  // splits <= 8, k_tiles < 2^23: no overflow
    w.kt_hi = (w.split + 1) * p.k_tiles / p.splits;
  } else {
    w.tile_end = p.dp_tiles;
    if (p.sk_tiles > 0) {
      w.units = static_cast<int64_t>(p.sk_tiles) * p.k_tiles;
      w.u = blockIdx.x * w.units / gridDim.x;
      w.u_end = (blockIdx.x + 1) * w.units / gridDim.x;
    }
  }
  return w;
}

template <class C, bool GROUPED>
struct Tables {
  int *ro;   // [experts+1] row offsets (grouped only)
  int *sfr;  // [experts+1] scale-row offsets (multiples of 128)
  int *tp;   // [experts+1] tile prefix
};

// rank: this CTA's place in its pair (PAIR only).
template <class C, bool GROUPED>
__device__ __forceinline__ TileInfo tile_info(const GemmArgs &p, const Tables<C, GROUPED> &tb, int tile, int rank = 0) {
  TileInfo t;
  int64_t sfb_base_block;
  if constexpr (C::PAIR) {
    // 256 x BN tiles (m_tiles counts 256-row tiles); CTA `rank` holds rows 128*rank .. +127 of
    // the tile and rows B_ROWS*rank .. +B_ROWS-1 of its B block.  A CTA wholly past the last
    // row stages zero-filled A and the tile's first scale block, and stores nothing.
    const int mb = tile % p.m_tiles, nb = tile / p.m_tiles;
    t.a_y = mb * 2 * C::BM + C::BM * rank;
    t.b_y = nb * C::BN + C::B_ROWS * rank;
    t.rows = max(0, min(C::BM, p.m - t.a_y));
    const int sfa_block = t.rows > 0 ? 2 * mb + rank : 2 * mb;
    t.sfa_blk = p.sfa + static_cast<int64_t>(sfa_block) * p.sf_chunks * 512;
    sfb_base_block = (nb * C::BN) / 128;
    t.sfb_blk = p.sfb + sfb_base_block * p.sf_chunks * 512;
    t.cols = min(C::BN, p.n - nb * C::BN);
    t.out_i0 = t.a_y;
    t.out_j0 = nb * C::BN;
    t.expert = 0;
  } else if constexpr (GROUPED) {
    int lo = 0, hi = p.experts - 1;  // largest e with tp[e] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tb.tp[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    t.expert = e;
    const int rows_e = tb.ro[e + 1] - tb.ro[e];
    const int mt_e = (rows_e + 127) / 128;
    const int local = tile - tb.tp[e];
    const int mt = local % mt_e, nt = local / mt_e;
    t.a_y = tb.ro[e] + mt * 128;
    t.b_y = e * p.n + nt * C::BN;
    t.sfa_blk = p.sfa + (static_cast<int64_t>(tb.sfr[e] / 128 + mt) * p.sf_chunks) * 512;
    sfb_base_block = (nt * C::BN) / 128;
    t.sfb_blk = p.sfb + e * p.sfb_expert_bytes + sfb_base_block * p.sf_chunks * 512;
    t.rows = min(128, rows_e - mt * 128);
    t.cols = min(C::BN, p.n - nt * C::BN);
    t.out_i0 = t.a_y;
    t.out_j0 = nt * C::BN;
  } else {
    const int mb = tile % p.m_tiles, nb = tile / p.m_tiles;
    t.a_y = mb * 128;
    t.b_y = nb * C::BN;
    t.sfa_blk = p.sfa + static_cast<int64_t>(mb) * p.sf_chunks * 512;
    sfb_base_block = t.b_y / 128;
    t.sfb_blk = p.sfb + sfb_base_block * p.sf_chunks * 512;
    t.rows = min(128, p.m - t.a_y);
    t.cols = min(C::BN, p.n - t.b_y);
    t.out_i0 = t.a_y;
    t.out_j0 = t.b_y;
    t.expert = 0;
  }
  t.sfb_blocks = min(C::SFB_BLOCKS, (t.cols + 127) / 128);
  return t;
}

// Chunks / MMAs in K stage kt: the last stage may be short (K % KSTAGE != 0).
template <class C>
__device__ __forceinline__ int stage_chunks(const GemmArgs &p, int kt) {
  return min(C::CHUNKS, p.sf_chunks - kt * C::CHUNKS);
}
template <class C = GemmCfg<32, 4, false>>
__device__ __forceinline__ int stage_mmas(const GemmArgs &p, int kt) {
  return min(C::MMAS, (p.k - kt * C::KSTAGE + 63) / 64);
}

// Operand tile of K stage kt: KS = 1 a 2-D box at byte column kt * 128; KS = 2 a 3-D box of two
// 256-wide K steps from the stage view (z = K step), landing as two consecutive tiles.
// A CTA pair's copies complete on the first CTA's barrier (`bar` is then a shared::cluster
// address), so that one barrier there tells the MMA lane that both CTAs' operands have landed.
template <class C>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap *map, uint32_t bar, int kt, int row) {
  if constexpr (C::PAIR) {
    if constexpr (C::KS == 1) tma_load_2d_pair(dst, map, bar, kt * 128, row);
    else tma_load_3d_pair(dst, map, bar, 0, row, kt * C::KS);
  } else {
    if constexpr (C::KS == 1) tma_load_2d(dst, map, bar, kt * 128, row);
    else tma_load_3d(dst, map, bar, 0, row, kt * C::KS);
  }
}

// Copies of K stage kt into ring slot stg (only the requested operand halves), all issued by the
// calling thread: a copy instruction costs the issuing thread ~100 cycles whatever its size,
// and spreading them over divergent lanes of one warp was measured slower still.
template <class C, bool FUSED = false>
__device__ __forceinline__ void issue_stage(const GemmArgs &p, const TileInfo &t, int kt, int stg, uint8_t *smem,
                                            uint64_t *full, const CUtensorMap *tmA, const CUtensorMap *tmB,
                                            bool do_a, bool do_b) {
  const int nch = stage_chunks<C>(p, kt);
  const uint32_t bar = C::PAIR ? map_to_rank(smem_u32(&full[stg]), 0) : smem_u32(&full[stg]);
  if (do_a) {
    load_operand<C>(smem_u32(smem + stg * C::A_BYTES), tmA, bar, kt, t.a_y);
    if constexpr (!C::PAIR)  // (a pair's scales go through their own ring)
      bulk_load(smem_u32(smem + C::SFA_REGION + stg * C::SFA_BYTES),
                t.sfa_blk + static_cast<int64_t>(kt) * C::CHUNKS * 512, nch * 512, bar);
  }
  if (do_b && !FUSED) {
    load_operand<C>(smem_u32(smem + C::B_REGION + stg * C::B_BYTES), tmB, bar, kt, t.b_y);
    if constexpr (!C::PAIR)
      for (int b = 0; b < t.sfb_blocks; ++b)
        bulk_load(smem_u32(smem + C::SFB_REGION + stg * C::SFB_BYTES + b * C::CHUNKS * 512),
                  t.sfb_blk + (static_cast<int64_t>(b) * p.sf_chunks + kt * C::CHUNKS) * 512, nch * 512, bar);
  }
}

// Bytes that land on full[] for K stage kt (operands, and scales unless they have their own ring).
template <class C, bool FUSED = false>
__device__ __forceinline__ uint32_t stage_tx(const GemmArgs &p, const TileInfo &t, int kt) {
  if constexpr (C::PAIR) return 2 * (C::A_BYTES + C::B_BYTES);  // both CTAs' operands, on the first CTA's barrier
  else if constexpr (FUSED) return C::A_BYTES + stage_chunks<C>(p, kt) * 512;  // B is quantised in-kernel
  else return C::A_BYTES + C::B_BYTES + stage_chunks<C>(p, kt) * 512 * (1 + t.sfb_blocks);
}

// Stream-K partial tiles.  A slot holds one CTA's fp32 partial of a 128 x BN tile in chunk-row
// order: float (c*128 + r)*32 + i is row r, column 32c + i, i.e. what epilogue thread r reads
// from tensor memory for chunk c, so the store is four full 32-byte sectors per thread and chunk.
template <class C>
__device__ __forceinline__ float *sk_slot(const GemmArgs &p, int cta, int j) {
  return p.ws + static_cast<int64_t>(2 * cta + (j == 0 ? 1 : 0)) * (C::BM * C::BN);
}

// Fix-up of a split tile by the last CTA to finish it, run by the four epilogue warps (thread
// tid = tile row) while the stage ring is idle:
//   out = bf16(alpha * (P_0 + P_1 + ... + P_{n-1})), partials added in contributor order.
// Columns are taken CW at a time: the n partials' chunks are copied into the ring with cp.async
// (every copy in flight at once, 16-byte pieces XOR-swizzled by row so the row-wise reads hit
// distinct banks), then each thread adds its row and writes 64 bytes of bf16 per chunk with
// 256-bit stores.  The plan keeps n * 16 KB within the ring.
template <class C>
__device__ __forceinline__ void sk_fixup(const GemmArgs &p, const TileInfo &t, const Seg &s, float alpha, int tid,
                                         uint8_t *smem) {
  constexpr int RING = C::RING_BYTES;
  constexpr int CHUNK_BYTES = 128 * 32 * 4;  // one 32-column chunk of a partial
  if (s.n * CHUNK_BYTES > RING) {  // never planned (the host caps contributors); uniform exit
    if (tid == 0) atomicOr(p.status, 4u);
    return;
  }
  int cw = C::BN;  // columns per pass, a power of two >= 32
  while (cw > 32 && s.n * cw * 512 > RING) cw >>= 1;
  const int chunks = cw / 32;
  const uint32_t buf = smem_u32(smem);
  const int row = tid;
  fence_proxy_async_smem();  // the ring was last written by TMA and read by the tensor cores
#pragma unroll 1
  for (int c0 = 0; c0 < C::BN / 32; c0 += chunks) {
#pragma unroll 1
    for (int jj = 0; jj < s.n; ++jj) {
      const float *src = sk_slot<C>(p, s.c0 + jj, jj) + static_cast<int64_t>(c0) * 128 * 32;
#pragma unroll 1
      for (int cc = 0; cc < chunks; ++cc) {
        const uint32_t dst = buf + static_cast<uint32_t>((jj * chunks + cc) * CHUNK_BYTES);
        const float *srcc = src + cc * 128 * 32;
#pragma unroll
        for (int e = tid; e < 1024; e += 128) {  // 1024 pieces of 16 bytes: row e/8, piece e%8
          const int r = e >> 3, q = e & 7;
          cp_async_16(dst + r * 128 + ((q ^ (r & 7)) << 4), srcc + e * 4);
        }
      }
    }
    cp_async_wait_all();
    named_barrier_sync(2, 128);
#pragma unroll 1
    for (int cc = 0; cc < chunks; ++cc) {
      const int c = c0 + cc;
      if (row >= t.rows || 32 * c >= t.cols) continue;
      float acc[32];
#pragma unroll 1
      for (int jj = 0; jj < s.n; ++jj) {
        const uint32_t base = buf + static_cast<uint32_t>((jj * chunks + cc) * CHUNK_BYTES + row * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = lds128(base + ((q ^ (row & 7)) << 4));
          const float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[4 * q + i] = jj == 0 ? f[i] : __fadd_rn(acc[4 * q + i], f[i]);
        }
      }
      __nv_bfloat16 *out = p.d + (t.out_i0 + row) * p.ldd + t.out_j0 + 32 * c;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = pack_bf16x2(__fmul_rn(alpha, acc[16 * h + 2 * i]), __fmul_rn(alpha, acc[16 * h + 2 * i + 1]));
        st_global_v8(out + 16 * h, v);
      }
    }
    named_barrier_sync(2, 128);  // the next pass overwrites the buffer
  }
}

// Fused quantisation (swap-AB plans): the four epilogue warps, idle until the accumulator is
// ready, quantise the activation rows of the CTA's K stages into the stages' operand-B tiles
// (e2m1 codes in the 128-byte swizzle the TMA would have produced) and B-scale chunks (e4m3,
// 128x4 or SM103 layout), block by block with the standalone quantiser's arithmetic
// (nvfp4_block16), so the MMAs see exactly the operand nvfp4_quantize would have written.  Rows
// without a token and K positions past k are zero, as the TMA's out-of-bounds fill.  Each
// thread keeps 4 blocks' loads in flight; then the writes are fenced for the tensor cores and
// one thread makes the second arrival on the stage's full barrier (resident slices: on every
// stage's barrier once all are written, because the scale writers take all stages' scales after
// stage 0 lands).  Every CTA of a token tile quantises that tile's slice again, once per weight
// tile, so this pays only for a few tokens.  Returns false when a wait gave up.
template <class C, bool GROUPED>
__device__ __forceinline__ void quantize_b_block(const GemmArgs &p, const TileInfo &t, uint8_t *smem, int stage, int kt,
                                                 int r, int b, const uint4 &lo, const uint4 &hi, float gs) {
  uint32_t code = 0;
  uint2 out = make_uint2(0u, 0u);
  if (kt * 256 + b * 16 < p.k) {
    float f[16];
    bf16x16_to_f32(lo, hi, f);
    out = nvfp4_block16(f, gs, code);
  }
  *reinterpret_cast<uint2 *>(smem + C::B_REGION + stage * C::B_BYTES + r * 128 + (((b >> 1) ^ (r & 7)) << 4) +
                             (b & 1) * 8) = out;
  const int m = r & 127;
  const int in_tile = p.sf_sm103 ? ((m >> 4) & 7) * 16 + ((m >> 2) & 3) * 128 + (m & 3) * 4 + (b & 3)
                                 : (m & 31) * 16 + (m >> 5) * 4 + (b & 3);
  smem[C::SFB_REGION + stage * C::SFB_BYTES + ((r >> 7) * C::CHUNKS + (b >> 2)) * 512 + in_tile] =
      static_cast<uint8_t>(code);
}

template <class C, bool GROUPED>
__device__ bool quantize_operand_b(const GemmArgs &p, const Tables<C, GROUPED> &tb, Work w, int crank, uint8_t *smem,
                                   uint64_t *full, uint64_t *empty, const WaitCtl &wc, int tid) {
  Seg sg;
  if (!w.next(p, sg)) return true;  // (swap-AB CTAs hold one segment)
  const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
  const float gs = __ldg(p.gs_q);
  const int rows = t.cols < C::BN ? t.cols : C::BN;  // tokens in this tile (operand B rows)
  // Rows without a token, and the scale rows nobody fills, are zero in every stage slot; they
  // are written once here (the slots are reused, the tile's token count is fixed).
  for (int i = tid; i < C::STAGES * C::SFB_BYTES / 16; i += 128)
    *reinterpret_cast<uint4 *>(smem + C::SFB_REGION + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
  const int pad16 = (C::BN - rows) * 8;  // 16-byte words of padding rows per stage slot
  for (int i = tid; i < C::STAGES * pad16; i += 128) {
    const int st = i / pad16, o = i - st * pad16;
    *reinterpret_cast<uint4 *>(smem + C::B_REGION + st * C::B_BYTES + rows * 128 + 16 * o) = make_uint4(0u, 0u, 0u, 0u);
  }
  const bool resident = p.resident != 0;
  const int nst = sg.kt1 - sg.kt0;
  // Blocks with data: (stage, token row, 16-element block); a resident slice takes all its
  // stages at once, the ring one stage at a time.  Each thread keeps QB blocks' loads in flight.
  constexpr int QB = 4;
  const int per_stage = rows * 16;
  int stage = 0;
  uint32_t phase = 0;
  for (int s0 = 0; s0 < nst;) {
    const int s1 = resident ? nst : s0 + 1;  // stages [s0, s1) of this pass
    if (!resident && !mbar_wait(smem_u32(&empty[stage]), phase ^ 1, wc, kSiteLoadEmpty)) return false;
    const int total = (s1 - s0) * per_stage;
    for (int base = tid; base < total; base += 128 * QB) {
      uint4 lo[QB], hi[QB];
#pragma unroll
      for (int u = 0; u < QB; ++u) {
        const int idx = base + 128 * u;
        lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < total) {
          const int ls = idx / per_stage, rem = idx - ls * per_stage;
          const int r = rem >> 4, b = rem & 15, k0 = (sg.kt0 + s0 + ls) * 256 + b * 16;
          if (k0 < p.k) {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.xq + (t.b_y + r) * p.ldx + k0);
            lo[u] = __ldg(src);
            hi[u] = __ldg(src + 1);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < QB; ++u) {
        const int idx = base + 128 * u;
        if (idx < total) {
          const int ls = idx / per_stage, rem = idx - ls * per_stage;
          quantize_b_block<C, GROUPED>(p, t, smem, resident ? s0 + ls : stage, sg.kt0 + s0 + ls, rem >> 4, rem & 15,
                                       lo[u], hi[u], gs);
        }
      }
    }
    fence_proxy_async_smem();  // generic writes -> visible to the tensor cores' reads
    named_barrier_sync(2, 128);
    if (tid == 0)
      for (int i = s0; i < s1; ++i) mbar_arrive(smem_u32(&full[resident ? i : stage]));
    s0 = s1;
    if (!resident && ++stage == C::STAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// Read form of the cluster split-K reduction: this rank sums the float4 units [u0, u1) of the
// column-major partials of all p.splits ranks (at red0 in each rank's shared memory).  A thread
// takes UPT units at a time and issues the distributed-shared-memory loads of every rank's
// partial for all of them before any sum, so that their latencies overlap.  It then adds each
// unit in rank order (a fixed order: deterministic output) and writes bf16(alpha * sum).
template <int UPT, int SMAX>
__device__ __forceinline__ void reduce_read(const GemmArgs &p, const TileInfo &t, uint32_t red0, int u0, int u1,
                                            float alpha, int tid, int nt) {
  for (int ub = u0 + tid; ub < u1; ub += UPT * nt) {
    float4 part[UPT][SMAX];
#pragma unroll
    for (int h = 0; h < UPT; ++h) {
      const int u = ub + h * nt;
      const uint32_t off = red0 + static_cast<uint32_t>((u < u1 ? u : ub) * 16);
#pragma unroll
      for (int s = 0; s < SMAX; ++s)
        if (s < p.splits) part[h][s] = ld_cluster_v4(map_to_rank(off, s));
    }
#pragma unroll
    for (int h = 0; h < UPT; ++h) {
      const int u = ub + h * nt;
      if (u >= u1) break;
      float4 v = part[h][0];
#pragma unroll
      for (int s = 1; s < SMAX; ++s)
        if (s < p.splits) {
          v.x += part[h][s].x;
          v.y += part[h][s].y;
          v.z += part[h][s].z;
          v.w += part[h][s].w;
        }
      const int c = (u * 4) / 128, r0 = (u * 4) % 128;
      if (r0 < t.rows) {
        const float o[4] = {v.x, v.y, v.z, v.w};
        if (p.swap) {
          uint2 pk;
          pk.x = pack_bf16x2(__fmul_rn(alpha, o[0]), __fmul_rn(alpha, o[1]));
          pk.y = pack_bf16x2(__fmul_rn(alpha, o[2]), __fmul_rn(alpha, o[3]));
          *reinterpret_cast<uint2 *>(p.d + (t.out_j0 + c) * p.ldd + t.out_i0 + r0) = pk;
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            p.d[(t.out_i0 + r0 + i) * p.ldd + t.out_j0 + c] = __float2bfloat16_rn(__fmul_rn(alpha, o[i]));
        }
      }
    }
  }
}

// Arrive on `bar` once the calling thread's tcgen05 operations so far are complete; for a CTA
// pair, on the barrier at that offset in both CTAs.
template <class C>
__device__ __forceinline__ void commit_to(uint32_t bar) {
  if constexpr (C::PAIR) tc_commit_pair_mc(bar, static_cast<uint16_t>(0x3));
  else tc_commit(bar);
}

// FUSED (swap-AB configurations only): operand B is quantised in the kernel (GemmArgs::xq); a
// separate instantiation, so the other kernels carry none of that code.
template <class C, bool GROUPED, bool FUSED = false>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB3, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ctrl = smem + C::RING_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(ctrl);
  uint64_t *empty = full + C::STAGES;
  uint64_t *accf = empty + C::STAGES;
  uint64_t *acce = accf + 2;
  uint64_t *sff = acce + 2;           // scale slot written (the scale writers arrive: 4, 8 in a pair)
  uint64_t *drain = sff + 16;
  uint64_t *sf_full = drain + 1;       // pair: scale ring slot landed
  uint64_t *sf_empty = sf_full + 8;    // pair: scale ring slot read by the 4 scale writers
  uint64_t *rbar = sf_empty + 16;     // push reduction: this rank's slices received
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(rbar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  volatile int *consumed = abort_flag + 1;  // K stages the MMA lane has taken (abort drain)
  volatile int *issued_count = consumed + 1;  // K stages the producer issued (abort drain)
  volatile int *sk_last = consumed + 2;       // stream-K: epilogue decision broadcast
  volatile float *alpha_s = reinterpret_cast<volatile float *>(sk_last + 1);  // alpha, read once
  volatile int *sf_issued = reinterpret_cast<volatile int *>(alpha_s + 1);   // pair: scale stages issued
  int *tables = reinterpret_cast<int *>(ctrl + C::CTRL_BYTES);
  Tables<C, GROUPED> tb{tables, tables + (C::MAX_EXPERTS + 1), tables + 2 * (C::MAX_EXPERTS + 1)};

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int crank = C::PAIR ? static_cast<int>(cluster_ctarank()) : 0;  // place in the CTA pair
  constexpr bool fused_q = FUSED;  // operand B quantised in-kernel
  // split-K reduction by pushes (32-wide tiles, at least 16 tokens: with fewer, a slice is a few
  // units and reading the partials remotely was measured faster); the same on every CTA
  const bool push_red = C::PUSH_RED && p.splits > 1 && p.n >= 16;
  static_assert(!FUSED || (C::SWAP_ONLY && !GROUPED), "fused quantisation serves the swap-AB plans");
  const WaitCtl wc{p.wait_limit, abort_flag, p.status};
  // The next kernel may launch now: it waits (griddepcontrol.wait) for this grid to complete
  // before it reads our output, and its CTAs can meanwhile take the SM space we leave free.
  if (threadIdx.x == 0) pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), fused_q ? 2 : 1);  // fused: the quantising warps arrive too
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&accf[a]), 1);
      mbar_init(smem_u32(&acce[a]), C::ACC_ARRIVALS);
    }
    for (int q = 0; q < C::SF_GROUPS; ++q) {
      mbar_init(smem_u32(&sff[q]), C::SLOT_ARRIVALS);
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(rbar), 1);
    if constexpr (C::PAIR) {
      for (int j = 0; j < C::SF_STAGES; ++j) {
        mbar_init(smem_u32(&sf_full[j]), 1);
        mbar_init(smem_u32(&sf_empty[j]), 4);
      }
    }
    *sf_issued = 0;
    *abort_flag = 0;
    *consumed = 0;
    *issued_count = 0;
    fence_barrier_init();
    if constexpr (!GROUPED) {
      if (p.resident) {
        // The CTA's one segment fits the ring: every copy goes out now, before the rest of the
        // CTA is set up.  Stage i of A has barrier full[i]; the slices of A's scales, of B and
        // of B's scales complete on full[0].  B's half waits for griddepcontrol.wait under PDL
        // (it is the activation) and is issued by the producer warp below.
        // (the segment and tile of make_work / tile_info, in 32-bit arithmetic: one tile per CTA)
        const int sp = p.splits, cta = static_cast<int>(blockIdx.x);
        const int tile = cta / sp, split = cta % sp;
        const int kt0 = split * p.k_tiles / sp, nst = (split + 1) * p.k_tiles / sp - kt0;
        const int mb = tile % p.m_tiles, b_y = (tile / p.m_tiles) * C::BN;
        const uint8_t *sfa_blk = p.sfa + (static_cast<int64_t>(mb) * p.sf_chunks + kt0 * C::CHUNKS) * 512;
        const uint8_t *sfb_blk = p.sfb + (static_cast<int64_t>(b_y / 128) * p.sf_chunks + kt0 * C::CHUNKS) * 512;
        mbar_arrive_expect_tx(smem_u32(&full[0]), fused_q ? C::A_BYTES + nst * C::SFA_BYTES
                                                          : C::A_BYTES + p.nst_max * C::B_BYTES + nst * (C::SFA_BYTES + C::SFB_BYTES));
        for (int i = 1; i < nst; ++i) mbar_arrive_expect_tx(smem_u32(&full[i]), C::A_BYTES);
        bulk_load(smem_u32(smem + C::SFA_REGION), sfa_blk, nst * C::SFA_BYTES, smem_u32(&full[0]));
        const int first = p.lookahead > 0 && p.lookahead < nst ? p.lookahead : nst;
        for (int i = 0; i < first; ++i)
          if (!(p.debug_skip_first_load && i == 0))
            tma_load_2d(smem_u32(smem + i * C::A_BYTES), &tmA, smem_u32(&full[i]), (kt0 + i) * 128, mb * 128);
        if (p.weight_operand != 1 && !fused_q) {
          tma_load_3d(smem_u32(smem + C::B_REGION), &tmB3, smem_u32(&full[0]), 0, b_y, kt0);
          bulk_load(smem_u32(smem + C::SFB_REGION), sfb_blk, nst * C::SFB_BYTES, smem_u32(&full[0]));
        }
        *issued_count = first;
      }
    }
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if constexpr (GROUPED) {
    // Row offsets are produced by earlier kernels: read them only after the PDL wait.
    pdl_wait();
    const int E = p.experts;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) tb.ro[e] = static_cast<int>(p.row_offsets[e]);
    __syncthreads();
    if (threadIdx.x == 0) {
      // The offsets are caller data: they must start at 0, end at the row count and never
      // decrease, otherwise tile addresses could leave the caller's buffers.  A malformed array
      // sets bit 1 of the status word and the kernel does no work.
      bool ok = tb.ro[0] == 0 && tb.ro[E] == p.m;
      int sfr = 0, tp = 0;
      for (int e = 0; e < E; ++e) {
        tb.sfr[e] = sfr;
        tb.tp[e] = tp;
        const int cnt = tb.ro[e + 1] - tb.ro[e];
        ok = ok && cnt >= 0;
        sfr += (max(cnt, 0) + 127) / 128 * 128;
        tp += (max(cnt, 0) + 127) / 128 * p.n_tiles;
      }
      if (!ok || tp > p.max_tiles) {
        if (blockIdx.x == 0) atomicOr(p.status, 2u);
        tp = 0;
      }
      tb.sfr[E] = sfr;
      tb.tp[E] = tp;
    }
  }

  // barriers initialised (and expert tables written, grouped); a pair's CTAs arrive on each
  // other's barriers, so both must have initialised theirs
  if constexpr (C::PAIR) cluster_sync();
  else __syncthreads();
  // push reduction: every rank's receive barrier is initialised before any slice is pushed (the
  // matching wait comes after the mainloop, when this arrive has long completed)
  if constexpr (C::PUSH_RED) {
    if (push_red) cluster_arrive_relaxed();
  }
  const Work work0 = make_work<GROUPED, C::PAIR>(p, GROUPED ? tb.tp[p.experts] : 0);
  // The loader (warp 0) starts right away; warp 1 allocates tensor memory meanwhile and a named
  // barrier among warps 1..9 (the tensor-memory users) publishes its address.
  uint32_t tmem = 0;
  if (warp != 0) {
    if (warp == 1) {
      tmem_alloc<C::CG>(smem_u32(tmem_holder), C::TMEM_COLS);
      tmem_relinquish<C::CG>();
    }
    tc_fence_before();
    named_barrier_sync(1, C::THREADS - 32);
    tc_fence_after();
    tmem = *tmem_holder;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One thread keeps the ring bookkeeping and issues every copy.
    if (lane == 0) {
      int issued = 0;
      if (!GROUPED && p.resident) {
        // Everything but B's half (the activation, under PDL) went out during set-up.
        Seg s0;
        if (Work(work0).next(p, s0)) {
          const TileInfo t = tile_info<C, GROUPED>(p, tb, s0.tile, crank);
          if (p.weight_operand == 1 && !fused_q) {
            pdl_wait();
            tma_load_3d(smem_u32(smem + C::B_REGION), &tmB3, smem_u32(&full[0]), 0, t.b_y, s0.kt0);
            bulk_load(smem_u32(smem + C::SFB_REGION), t.sfb_blk + static_cast<int64_t>(s0.kt0) * C::CHUNKS * 512,
                      (s0.kt1 - s0.kt0) * C::SFB_BYTES, smem_u32(&full[0]));
          }
          // the rest of A, paced: stage i goes out once stage i - lookahead has landed
          issued = *issued_count;
          for (int i = issued; i < s0.kt1 - s0.kt0; ++i) {
            if (!mbar_wait(smem_u32(&full[i - p.lookahead]), 0, wc, kSiteLoadEmpty)) goto producer_done;
            tma_load_2d(smem_u32(smem + i * C::A_BYTES), &tmA, smem_u32(&full[i]), (s0.kt0 + i) * 128, t.a_y);
            issued = i + 1;
          }
        }
      } else {
        int stage = 0;
        uint32_t phase = 0;
        const bool skip_first = p.debug_skip_first_load != 0;
        // Under PDL (p.weight_operand != 0) the weight half of the first ring of stages goes out
        // before griddepcontrol.wait, so it streams while the preceding kernel finishes; the
        // activation half follows in the loop below.
        int pre = 0;
        const bool pre_a = p.weight_operand == 1, pre_b = p.weight_operand == 2;
        Work w = work0;
        Seg s0;
        if (!GROUPED && (pre_a || pre_b) && Work(work0).next(p, s0)) {
          const TileInfo t = tile_info<C, GROUPED>(p, tb, s0.tile, crank);
          pre = min(p.lookahead > 0 ? p.lookahead : C::STAGES, min(C::STAGES, s0.kt1 - s0.kt0));
          for (int i = 0; i < pre; ++i) {  // the ring is empty at start: no wait for a free slot
            const int kt = s0.kt0 + i;
            if (crank == 0) mbar_arrive_expect_tx(smem_u32(&full[i]), stage_tx<C, FUSED>(p, t, kt));
            if (!(skip_first && i == 0)) issue_stage<C, FUSED>(p, t, kt, i, smem, full, &tmA, &tmB, pre_a, pre_b);
          }
          if (C::SWAP_ONLY && pre_a) {
            // The rest of this CTA's weight slice goes to L2 now, while the preceding kernel runs;
            // the ring then refills from L2 instead of from cold HBM.
            for (int kt = s0.kt0 + pre; kt < s0.kt1; ++kt) tma_prefetch_l2_2d(&tmA, kt * 128, t.a_y);
            if (s0.kt0 + pre < s0.kt1)
              bulk_prefetch_l2(t.sfa_blk + static_cast<int64_t>(s0.kt0 + pre) * C::CHUNKS * 512,
                               (s0.kt1 - s0.kt0 - pre) * C::CHUNKS * 512);
          }
        }
        pdl_wait();
        bool first = true;
        for (Seg sg; w.next(p, sg); first = false) {
          const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
          for (int kt = sg.kt0; kt < sg.kt1; ++kt) {
            const bool early_stage = first && kt - sg.kt0 < pre;
            if (p.lookahead > 0 && issued >= p.lookahead) {  // pacing: stage issued - L has landed
              const int j = issued - p.lookahead;
              if (!mbar_wait(smem_u32(&full[j % C::STAGES]), (j / C::STAGES) & 1, wc, kSiteLoadEmpty)) goto producer_done;
            }
            if (!early_stage) {
              if (!mbar_wait<C::PAIR>(smem_u32(&empty[stage]), phase ^ 1, wc, kSiteLoadEmpty)) goto producer_done;
              if (crank == 0) mbar_arrive_expect_tx(smem_u32(&full[stage]), stage_tx<C, FUSED>(p, t, kt));
            }
            const bool do_a = !(early_stage && pre_a), do_b = !(early_stage && pre_b);
            if (!(skip_first && issued == 0) && (do_a || do_b))
              issue_stage<C, FUSED>(p, t, kt, stage, smem, full, &tmA, &tmB, do_a, do_b);
            ++issued;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
    producer_done:
      *issued_count = issued;  // stages issued, for the abort drain
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One wait per stage: the scale writers arrive on sff only after they saw the stage land
    // (full), so sff covers both.  A full stage's four MMAs are issued unrolled with the
    // accumulate predicates fixed (a runtime loop costs about a third more issue time).
    if (lane == 0 && !GROUPED && p.resident) {
      // Resident slice: the scale writers fill every stage's scale slot once (one hand-off);
      // the MMAs of stage i then only wait for A's stage i to land.
      int taken = 0;
      Seg sg;
      Work w = work0;
      if (w.next(p, sg)) {
        const int nst = sg.kt1 - sg.kt0;
        if (!mbar_wait(smem_u32(&sff[0]), 0, wc, kSiteMmaScale)) goto mma_done_r;
        taken = 1;  // the scale writers saw full[0]
        tc_fence_after();
        for (int i = 0; i < nst; ++i) {
          if (i > 0) {
            if (!mbar_wait(smem_u32(&full[i]), 0, wc, kSiteMmaFull)) goto mma_done_r;
            taken = i + 1;
          }
          const uint32_t slot = tmem + C::SF_COL0 + i * C::SF_SLOT;
          const uint64_t adesc = sdesc_k_sw128(smem_u32(smem + i * C::A_BYTES));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(smem + C::B_REGION + i * C::B_BYTES));
          const uint32_t sb = slot + C::SFA_COLS;
          constexpr uint32_t SB = 4 * C::SFB_BLOCKS;
          // (resident CTAs are swap-AB, never pairs; the group template only keeps every
          // tcgen05 instruction of a pair kernel in the same CTA group)
          if constexpr (!C::MX) {
            mma_nvf4<C::CG>(tmem, adesc, bdesc, C::IDESC, slot, sb, i > 0 ? 1u : 0u);
            mma_nvf4<C::CG>(tmem, adesc + 2, bdesc + 2, C::IDESC, slot + 4, sb + SB, 1u);
            mma_nvf4<C::CG>(tmem, adesc + 4, bdesc + 4, C::IDESC, slot + 8, sb + 2 * SB, 1u);
            mma_nvf4<C::CG>(tmem, adesc + 6, bdesc + 6, C::IDESC, slot + 12, sb + 3 * SB, 1u);
          }
        }
        tc_commit<C::CG>(smem_u32(&accf[0]));
      }
    mma_done_r:
      *consumed = taken;
    } else if (lane == 0 && crank == 0) {
      int stage = 0;
      uint32_t phase = 0;  // of full[] (pairs wait on it; for the others sff implies it)
      int taken = 0;  // stages known landed (abort drain)
      int acc = 0;
      uint32_t acc_phase = 0;
      int g = 0;             // scale-slot group of the stage
      uint32_t g_phase = 0;
      // Per stage the lane waits once for the scale group (and, in a pair, once for the operands),
      // issues the stage's MMAs and commits twice; the descriptors of stage 0 are computed once
      // (the other stages sit at fixed offsets), so that the lane's own work between MMAs stays
      // below the tensor pipe's time for them.
      const uint64_t adesc0 = sdesc_k_sw128(smem_u32(smem));
      const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(smem + C::B_REGION));
      const uint32_t sf_base = tmem + C::SF_COL0;
      Work w = work0;
      for (Seg sg; w.next(p, sg);) {
        if (!mbar_wait<C::PAIR>(smem_u32(&acce[acc]), acc_phase ^ 1, wc, kSiteMmaAcc)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * C::BN;
        for (int kt = sg.kt0; kt < sg.kt1; ++kt) {
          if (!mbar_wait(smem_u32(&sff[g]), g_phase, wc, kSiteMmaScale)) goto mma_done;
          if constexpr (C::PAIR) {
            // a pair's scale writers do not wait for the operands: both CTAs' operand copies of
            // the stage complete on this CTA's barrier
            if (!mbar_wait(smem_u32(&full[stage]), phase, wc, kSiteMmaFull)) goto mma_done;
          }
          ++taken;
          tc_fence_after();
          const uint64_t adesc = adesc0 + static_cast<uint64_t>(stage * (C::A_BYTES >> 4));
          const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(stage * (C::B_BYTES >> 4));
          const uint32_t acc0 = kt > sg.kt0 ? 1u : 0u;
          // K step h of the stage reads its scales from slot g * SUB + h
#pragma unroll
          for (int h = 0; h < C::SUB; ++h) {
            const uint32_t slot = sf_base + (g * C::SUB + h) * C::SF_SLOT;
            if constexpr (C::MX) {
              // MXFP4: a 512-byte scale chunk covers 128 K elements = two MMAs (scale ids 0, 2)
              constexpr uint32_t I0 = C::IDESC, I2 = C::IDESC | (2u << 29) | (2u << 4);
              const uint32_t sb = slot + C::SFA_COLS;
              if (stage_mmas(p, kt) == 4) {
                mma_mxf4(d_tmem, adesc, bdesc, I0, slot, sb, acc0);
                mma_mxf4(d_tmem, adesc + 2, bdesc + 2, I2, slot, sb, 1u);
                mma_mxf4(d_tmem, adesc + 4, bdesc + 4, I0, slot + 4, sb + 4 * C::SFB_BLOCKS, 1u);
                mma_mxf4(d_tmem, adesc + 6, bdesc + 6, I2, slot + 4, sb + 4 * C::SFB_BLOCKS, 1u);
              } else {
                for (int j = 0; j < stage_mmas(p, kt); ++j) {
                  const int c = j >> 1;
                  mma_mxf4(d_tmem, adesc + 2 * j, bdesc + 2 * j, (j & 1) ? I2 : I0, slot + 4 * c,
                           sb + c * 4 * C::SFB_BLOCKS, j > 0 ? 1u : acc0);
                }
              }
            } else {
              const uint32_t sb = slot + C::SFA_COLS;
              constexpr uint32_t SB = 4 * C::SFB_BLOCKS;  // B scale columns per MMA
              // MMA j of K step h: 32 bytes into the step's 128-byte-row tile (descriptor units of
              // 16 bytes), the step's tile at +h * A_TILE / +h * B_TILE
              const uint64_t ad = adesc + h * (C::A_TILE >> 4), bd = bdesc + h * (C::B_TILE >> 4);
              const int nm = stage_mmas<C>(p, kt) - 4 * h;
              if (nm >= 4) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  mma_nvf4<C::CG>(d_tmem, ad + 2 * j, bd + 2 * j, C::IDESC, slot + 4 * j, sb + j * SB,
                                  (j > 0 || h > 0) ? 1u : acc0);
              } else {
                for (int j = 0; j < nm; ++j)
                  mma_nvf4<C::CG>(d_tmem, ad + 2 * j, bd + 2 * j, C::IDESC, slot + 4 * j, sb + j * SB,
                                  (j > 0 || h > 0) ? 1u : acc0);
              }
            }
          }
          // (one commit: the scale writers learn from the same barrier that the stage's scale
          // group is free again)
          commit_to<C>(smem_u32(&empty[stage]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (++g == C::SF_GROUPS) {
            g = 0;
            g_phase ^= 1;
          }
        }
        commit_to<C>(smem_u32(&accf[acc]));
        if (++acc == C::NACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    mma_done:
      *consumed = taken;
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ scale writers
    // Each warp fills its own 32-lane quadrant of the slot with the full scale data of the
    // stage (the MMA reads every quadrant): lane i takes bytes 16*i .. 16*i+15 of every
    // 512-byte scale tile, i.e. 4 consecutive columns per tile.
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    int g = 0;  // scale-slot group of the stage
    uint32_t g_phase = 0;
    Work w = work0;
    if (!GROUPED && p.resident) {
      // Resident slice: all scale slices landed with stage 0; fill every stage's slot, then
      // hand the slots to the MMA lane with a single arrival.
      Seg sg;
      if (w.next(p, sg)) {
        if (!mbar_wait(smem_u32(&full[0]), 0, wc, kSiteScaleFull)) goto scale_done;
        for (int i = 0; i < sg.kt1 - sg.kt0; ++i) {
          const uint32_t sfa_s = smem_u32(smem + C::SFA_REGION + i * C::SFA_BYTES);
          const uint32_t sfb_s = smem_u32(smem + C::SFB_REGION + i * C::SFB_BYTES);
          uint32_t ra[C::SFA_COLS], rb[C::SFB_COLS];
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c) {
            const uint4 v = ld_sf_lane(sfa_s + 512 * c, lane, p.sf_sm103);
            ra[4 * c] = v.x;
            ra[4 * c + 1] = v.y;
            ra[4 * c + 2] = v.z;
            ra[4 * c + 3] = v.w;
#pragma unroll
            for (int b = 0; b < C::SFB_BLOCKS; ++b) {
              const uint4 u = ld_sf_lane(sfb_s + (b * C::CHUNKS + c) * 512, lane, p.sf_sm103);
              const int o = c * 4 * C::SFB_BLOCKS + 4 * b;
              rb[o] = u.x;
              rb[o + 1] = u.y;
              rb[o + 2] = u.z;
              rb[o + 3] = u.w;
            }
          }
          const uint32_t slot = tmem + lane_base + C::SF_COL0 + i * C::SF_SLOT;
          tmem_st_32x32b<C::SFA_COLS>(slot, ra);
          tmem_st_32x32b<C::SFB_COLS>(slot + C::SFA_COLS, rb);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sff[0]));
      }
    } else {
      uint32_t sit = 0;  // ring stages (the scale ring of a pair is indexed by stage)
      for (Seg sg; w.next(p, sg);) {
        for (int kt = sg.kt0; kt < sg.kt1; ++kt, ++sit) {
          // The stage's scales land with its operands, or (pair) in the scale ring ahead of them.
          const int sf_slot = C::PAIR ? static_cast<int>(sit % C::SF_STAGES) : stage;
          if constexpr (C::PAIR) {
            if (!mbar_wait(smem_u32(&sf_full[sf_slot]), (sit / C::SF_STAGES) & 1, wc, kSiteScaleFull)) goto scale_done;
          } else {
            if (!mbar_wait(smem_u32(&full[stage]), phase, wc, kSiteScaleFull)) goto scale_done;
          }
          const uint32_t sfa_s = smem_u32(smem + C::SFA_REGION + sf_slot * C::SFA_BYTES);
          const uint32_t sfb_s = smem_u32(smem + C::SFB_REGION + sf_slot * C::SFB_BYTES);
          // The stage's group of tensor-memory slots, one per 256-wide K step (chunks h * SUB_CHUNKS ..),
          // was last read by the MMAs of stage sit - SF_GROUPS; their completion is the phase
          // (sit - SF_GROUPS) / STAGES of that stage's ring barrier empty[], which the MMA lane
          // commits to (both CTAs' of a pair).  The writers are never a full ring turn behind
          // the MMAs (those need this stage's scales first), so the parity is unambiguous.
          if (sit >= static_cast<uint32_t>(C::SF_GROUPS)) {
            const uint32_t done = sit - C::SF_GROUPS;
            if (!mbar_wait(smem_u32(&empty[done % C::STAGES]), (done / C::STAGES) & 1, wc, kSiteScaleSlot)) goto scale_done;
          }
#pragma unroll
          for (int h = 0; h < C::SUB; ++h) {
            uint32_t ra[C::SFA_COLS], rb[C::SFB_COLS];
#pragma unroll
            for (int cc = 0; cc < C::SUB_CHUNKS; ++cc) {
              const int c = h * C::SUB_CHUNKS + cc;
              const uint4 v = ld_sf_lane(sfa_s + 512 * c, lane, p.sf_sm103);
              ra[4 * cc] = v.x;
              ra[4 * cc + 1] = v.y;
              ra[4 * cc + 2] = v.z;
              ra[4 * cc + 3] = v.w;
#pragma unroll
              for (int b = 0; b < C::SFB_BLOCKS; ++b) {
                const uint4 w = ld_sf_lane(sfb_s + (b * C::CHUNKS + c) * 512, lane, p.sf_sm103);
                const int o = cc * 4 * C::SFB_BLOCKS + 4 * b;
                rb[o] = w.x;
                rb[o + 1] = w.y;
                rb[o + 2] = w.z;
                rb[o + 3] = w.w;
              }
            }
            const uint32_t slot = tmem + lane_base + C::SF_COL0 + (g * C::SUB + h) * C::SF_SLOT;
            tmem_st_32x32b<C::SFA_COLS>(slot, ra);
            tmem_st_32x32b<C::SFB_COLS>(slot + C::SFA_COLS, rb);
          }
          if constexpr (C::PAIR) {  // the stage's scales are in registers: the ring slot may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sf_empty[sf_slot]));
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (C::PAIR) mbar_arrive_remote(map_to_rank(smem_u32(&sff[g]), 0));
            else mbar_arrive(smem_u32(&sff[g]));
          }
          if (++g == C::SF_GROUPS) {
            g = 0;
            g_phase ^= 1;
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  scale_done:;
    if constexpr (!GROUPED && C::SWAP_ONLY && C::BN >= 64) {
      // A split tile's partial: the scale writers, idle once the stages are consumed, move the
      // upper half of the accumulator's columns into the reduction buffer beside the epilogue
      // warps (each warp reaches the same lane quadrant, warp % 4, as one epilogue warp).
      Work w2 = work0;
      Seg sg2;
      if (p.splits > 1 && w2.next(p, sg2)) {
        const TileInfo t = tile_info<C, GROUPED>(p, tb, sg2.tile, crank);
        if (mbar_wait(smem_u32(&accf[0]), 0, wc, kSiteEpilogue)) {
          tc_fence_after();
          const int row = (warp & 3) * 32 + lane;
          float *red = reinterpret_cast<float *>(smem);
#pragma unroll 1
          for (int c = C::BN / 64; c < C::BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem + lane_base + 32 * c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * c + i < t.cols) red[(32 * c + i) * 128 + row] = __uint_as_float(r[i]);
          }
        }
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ scale copies (pairs only)
    // One thread fills the scale ring: both scale slices of each K stage, as far ahead of the
    // scale writers as the ring allows.
    if (lane == 0) {
      pdl_wait();  // the activation's scales may come from the preceding kernel
      int it = 0;
      Work w = work0;
      for (Seg sg; w.next(p, sg);) {
        const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
        for (int kt = sg.kt0; kt < sg.kt1; ++kt, ++it) {
          const int j = it % C::SF_STAGES;
          if (!mbar_wait(smem_u32(&sf_empty[j]), ((it / C::SF_STAGES) & 1) ^ 1, wc, kSiteLoadEmpty)) goto sfcopy_done;
          const int nch = stage_chunks<C>(p, kt);
          const uint32_t bar = smem_u32(&sf_full[j]);
          mbar_arrive_expect_tx(bar, nch * 512 * (1 + t.sfb_blocks));
          bulk_load(smem_u32(smem + C::SFA_REGION + j * C::SFA_BYTES),
                    t.sfa_blk + static_cast<int64_t>(kt) * C::CHUNKS * 512, nch * 512, bar);
          for (int b = 0; b < t.sfb_blocks; ++b)
            bulk_load(smem_u32(smem + C::SFB_REGION + j * C::SFB_BYTES + b * C::CHUNKS * 512),
                      t.sfb_blk + (static_cast<int64_t>(b) * p.sf_chunks + kt * C::CHUNKS) * 512, nch * 512, bar);
          *sf_issued = it + 1;
        }
      }
    sfcopy_done:;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int quad = warp & 3;  // tcgen05.ld: warp w reaches lanes 32*(w%4) .. +31
    const int row = quad * 32 + lane;
    const int tid = threadIdx.x - 64;  // 0..127 over the four epilogue warps
    if constexpr (FUSED) {
      // (a wait that gave up set the abort flag; the epilogue below then does no work)
      quantize_operand_b<C, GROUPED>(p, tb, work0, crank, smem, full, empty, wc, tid);
    }
    // alpha is read by one thread and shared: a load left to each thread's first use was
    // scheduled there, putting a full memory latency (~1400 cycles) in front of the stores.
    if (tid == 0) *alpha_s = p.alpha ? *p.alpha : 1.0f;
    {
      // Touch the output lines of this CTA's first tile now: the first store to a cold page
      // otherwise waits for its address translation at the very end of the kernel.
      Work w = work0;
      Seg sg{};
      if (w.next(p, sg)) {
        const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
        if (row < t.rows) {
          if (p.swap) {
            prefetch_l2(p.d + t.out_j0 * p.ldd + t.out_i0 + row);
            prefetch_l2(p.d + (t.out_j0 + t.cols - 1) * p.ldd + t.out_i0 + row);
          } else {
            prefetch_l2(p.d + (t.out_i0 + row) * p.ldd + t.out_j0);
          }
        }
      }
    }
    named_barrier_sync(2, 128);
    const float alpha = *alpha_s;
    int acc = 0;
    uint32_t acc_phase = 0;
    Work w = work0;
    Seg pending{};  // a split tile this CTA must finish once its ring is idle
    bool has_pending = false;
    // After a failed wait the warps keep walking the segments without doing work (every later
    // wait returns at once), so all four always meet the same named barriers.
    for (Seg sg; w.next(p, sg);) {
      const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
      const bool sk_part = C::MULTI_TILE && !GROUPED && p.splits == 1 && sg.n > 1;
      const bool ok = mbar_wait<C::PAIR>(smem_u32(&accf[acc]), acc_phase, wc, kSiteEpilogue);
      tc_fence_after();
      const uint32_t t_base = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * C::BN;
      const float tile_alpha = (GROUPED && p.alpha_per_expert && p.alpha) ? __ldg(p.alpha + t.expert) : alpha;
      float *red = reinterpret_cast<float *>(smem);
      float *slot = sk_part ? sk_slot<C>(p, blockIdx.x, sg.j) : nullptr;
      // (a split swap-AB tile of 64 or more columns: the scale writers take the upper half)
      const int c_end = (!GROUPED && C::SWAP_ONLY && C::BN >= 64 && p.splits > 1) ? C::BN / 64 : C::BN / 32;
#pragma unroll 1
      for (int c = 0; ok && c < c_end; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + 32 * c, r);
        tmem_ld_wait();
        if (C::SWAP_ONLY && p.splits > 1) {
          // (the reduction reads the valid columns only)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i < t.cols) red[(32 * c + i) * 128 + row] = __uint_as_float(r[i]);
        } else if (sk_part) {
          float *dst = slot + (c * 128 + row) * 32;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = r[8 * q + i];
            st_global_v8(dst + 8 * q, v);
          }
        } else if (!C::SWAP_ONLY) {
          if (row < t.rows && 32 * c < t.cols) {
            __nv_bfloat16 *out = p.d + (t.out_i0 + row) * p.ldd + t.out_j0 + 32 * c;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t v[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                v[i] = pack_bf16x2(__fmul_rn(tile_alpha, __uint_as_float(r[16 * h + 2 * i])),
                                   __fmul_rn(tile_alpha, __uint_as_float(r[16 * h + 2 * i + 1])));
              st_global_v8(out + 16 * h, v);
            }
          }
        } else if (row < t.rows) {
          // operand A is the weight: TMEM lane = output column, TMEM column = output row
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int j = 32 * c + i;
            if (j < t.cols) {
              const float v = __fmul_rn(alpha, __uint_as_float(r[i]));
              p.d[(t.out_j0 + j) * p.ldd + t.out_i0 + row] = __float2bfloat16_rn(v);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (C::PAIR) mbar_arrive_remote(map_to_rank(smem_u32(&acce[acc]), 0));
        else mbar_arrive(smem_u32(&acce[acc]));
      }
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1;
      }
      if (sk_part) {
        // Publish the partial: the four warps' stores are ordered before one acquire-release
        // increment of the tile's counter; the CTA that brings it to n adds the partials and
        // sets it back to zero for the next call.
        named_barrier_sync(2, 128);
        if (tid == 0) {
          int last = -1;  // -1: a wait gave up, do nothing more
          if (!*abort_flag) {
            unsigned int *cnt = p.ws_cnt + (sg.tile - p.dp_tiles);
            last = atom_add_acq_rel_gpu(cnt, 1u) == static_cast<unsigned int>(sg.n - 1) ? 1 : 0;
            if (last) *reinterpret_cast<volatile unsigned int *>(cnt) = 0u;
          }
          *sk_last = last;
        }
        named_barrier_sync(2, 128);
        if (*sk_last == 1) {
          // The ring is idle once no segment follows (all stages consumed, none to load); a
          // split tile finished earlier waits for that point (at most one: only a CTA's first
          // segment can be a partial that is not its last).
          Work rest = w;
          Seg more;
          if (!rest.next(p, more)) {
            sk_fixup<C>(p, t, sg, alpha, tid, smem);
          } else {
            pending = sg;
            has_pending = true;
          }
        }
      }
    }
    if (has_pending) {  // uniform over the four warps
      named_barrier_sync(2, 128);
      if (tid == 0) *sk_last = *abort_flag ? -1 : 1;  // after a time-out copies may still land in the ring
      named_barrier_sync(2, 128);
      if (*sk_last == 1) sk_fixup<C>(p, tile_info<C, GROUPED>(p, tb, pending.tile, crank), pending, alpha, tid, smem);
    }
  }

  tc_fence_before();  // order this warp's tcgen05 work before the barrier (dealloc follows it)
  if (push_red) fence_proxy_async_smem();  // partials -> visible to the bulk copies
  __syncthreads();
  if (*abort_flag) {
    // Drain: wait (bounded) for copies still landing in shared memory and for outstanding
    // tcgen05 operations, so nothing writes shared or tensor memory after the CTA is gone.
    if (threadIdx.x == 0) {
      // (a pair's operand copies complete on the first CTA's barriers: the first CTA drains them
      // for both, and the second stays until then at the cluster barrier before exit)
      const int issued = crank == 0 ? *issued_count : 0;
      const int done = *consumed;
      for (int i = (done > issued - C::STAGES ? done : issued - C::STAGES); i < issued; ++i) {
        const uint32_t bar = smem_u32(&full[i % C::STAGES]);
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, (i / C::STAGES) & 1) && clock64() - t0 < p.wait_limit) {
        }
      }
      if constexpr (C::PAIR) {  // and the scale ring's copies
        const int sfi = *sf_issued;
        for (int i = sfi > C::SF_STAGES ? sfi - C::SF_STAGES : 0; i < sfi; ++i) {
          const uint32_t bar = smem_u32(&sf_full[i % C::SF_STAGES]);
          const long long t0 = clock64();
          while (!mbar_try_wait(bar, (i / C::SF_STAGES) & 1) && clock64() - t0 < p.wait_limit) {
          }
        }
      }
    }
    if (threadIdx.x == 32) {
      tc_commit<C::CG>(smem_u32(drain));
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(drain), 0) && clock64() - t0 < p.wait_limit) {
      }
    }
    __syncthreads();
  }

  if constexpr (!GROUPED && C::SWAP_ONLY) {
    if (p.splits > 1) {
      if (push_red) {
        // Split-K reduction by pushes: CTA `rank` reduces the contiguous 1/splits of the valid
        // units (float4 groups of the column-major partial) [u0, u1); every other rank copies
        // that slice of its partial into this CTA's receive buffer (slot s for source rank s
        // below this one, s - 1 above), the copies completing on this CTA's rbar; the sum runs
        // in rank order, as below.
        cluster_wait();
        const int rank = static_cast<int>(cluster_ctarank()), S = p.splits;
        Work w = work0;
        Seg sg{};
        w.next(p, sg);
        const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
        const float alpha = *alpha_s;
        const int units = min(t.cols, C::BN) * 32;
        const int slot = (units + S - 1) / S;  // units of the largest slice
        const int u0 = rank * units / S, u1 = (rank + 1) * units / S;
        const uint32_t red0 = smem_u32(smem), rcv0 = smem_u32(ctrl + C::CTRL_BYTES);
        if (threadIdx.x == 0) {
          mbar_arrive_expect_tx(smem_u32(rbar), static_cast<uint32_t>((S - 1) * (u1 - u0) * 16));
          for (int r = 0; r < S; ++r) {
            const int a0 = r * units / S, a1 = (r + 1) * units / S;
            if (r != rank && a1 > a0)
              bulk_copy_to_peer(map_to_rank(rcv0 + static_cast<uint32_t>((rank < r ? rank : rank - 1) * slot * 16), r),
                                red0 + a0 * 16,
                                static_cast<uint32_t>((a1 - a0) * 16), map_to_rank(smem_u32(rbar), r));
          }
        }
        if (mbar_wait(smem_u32(rbar), 0, wc, kSiteEpilogue)) {
          const float4 *own = reinterpret_cast<const float4 *>(smem);
          const float4 *rcv = reinterpret_cast<const float4 *>(ctrl + C::CTRL_BYTES);
          for (int u = u0 + static_cast<int>(threadIdx.x); u < u1; u += C::THREADS) {
            float4 v = rank == 0 ? own[u] : rcv[u - u0];  // (source 0 sits in slot 0)
            for (int s2 = 1; s2 < S; ++s2) {
              const float4 q = s2 == rank ? own[u] : rcv[(s2 < rank ? s2 : s2 - 1) * slot + (u - u0)];
              v.x += q.x;
              v.y += q.y;
              v.z += q.z;
              v.w += q.w;
            }
            const int c = (u * 4) / 128, r0 = (u * 4) % 128;
            if (r0 < t.rows) {
              uint2 pk;  // (swap-AB: the output row is the token, the 4 values are weight rows)
              pk.x = pack_bf16x2(__fmul_rn(alpha, v.x), __fmul_rn(alpha, v.y));
              pk.y = pack_bf16x2(__fmul_rn(alpha, v.z), __fmul_rn(alpha, v.w));
              *reinterpret_cast<uint2 *>(p.d + (t.out_j0 + c) * p.ldd + t.out_i0 + r0) = pk;
            }
          }
        }
        // the copies out of this CTA's partial have completed (every receiver saw its slices)
        // before any CTA leaves; the arrive publishes nothing
        cluster_sync_relaxed();
      } else {
      // Split-K reduction across the cluster.  The partial tile is stored column-major
      // (128 rows per column, a 4-row group per float4 unit); only the units of the tile's
      // valid columns are reduced, CTA `rank` taking a contiguous 1/splits of them.  Every
      // thread of the CTA takes part, several units at a time (reduce_read).
      cluster_sync();
      {
        const int rank = static_cast<int>(cluster_ctarank());
        Work w = work0;
        Seg sg{};
        w.next(p, sg);
        const TileInfo t = tile_info<C, GROUPED>(p, tb, sg.tile, crank);
        const float alpha = *alpha_s;
        const int units = min(t.cols, C::BN) * 32;  // float4 groups of the valid columns
        const int u0 = rank * units / p.splits, u1 = (rank + 1) * units / p.splits;
        const uint32_t red0 = smem_u32(smem);
        // Two ranks of a 128- or 256-wide tile: four units per thread in flight, else two.  (More
        // loads in flight per thread were measured slower with four ranks: the distributed
        // shared-memory reads congest.  The narrower tiles keep one form, whose code measured
        // faster there.)
        bool done = false;
        if constexpr (C::BN >= 128) {
          if (p.splits <= 2) {
            reduce_read<4, 2>(p, t, red0, u0, u1, alpha, static_cast<int>(threadIdx.x), C::THREADS);
            done = true;
          }
        }
        if (!done) reduce_read<2, 8>(p, t, red0, u0, u1, alpha, static_cast<int>(threadIdx.x), C::THREADS);
      }
      // no CTA leaves while another may still read its partial; those reads are complete here
      // (their sums are stored), so the arrive publishes nothing
      cluster_sync_relaxed();
      }
    }
  }

  // A pair's CTAs stay until both are done: the first CTA's MMAs read the second's shared memory
  // and write its tensor memory, and the second arrives on the first's barriers.
  if constexpr (C::PAIR) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<C::CG>(tmem, C::TMEM_COLS);
  }
}

}  // namespace nvfp4
