// rsm_params.h -- launch parameters and the shared-memory plan of the
// materialization kernel, shared by the host launcher and the kernel.
#pragma once
#include <cstdint>

#include "../../include/replayssm.h"  // the state formats

namespace rsm {

constexpr int kConsumerWarps = 8;  // 16-bit and fp32 state, and the tensor-core kernel
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kThreads = 32 + kConsumerThreads;
// One-byte state (both rounding modes): four consumer warps per CTA (each
// lane owns 64 codes, so the per-item work of a lane is spread over twice the
// elements), three CTAs per SM.
constexpr int kQ8ConsumerWarps = 4;
constexpr int kQ8Threads = 32 * (1 + kQ8ConsumerWarps);
constexpr int kQ8MaxRegs = 128;  // 15 warps per SM: four on three sub-partitions, 4 x 32 x 128 = 16384
constexpr int kMaxWindow = 64;
constexpr int kMaxStages = 16;
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s: never reached by a correct run

// Shared memory: [full mbarriers][empty mbarriers] | abort flag | per-warp
// decay weights | per-warp token-chunk buffers | item descriptors (one per
// pipeline slot) | the item arena.
constexpr uint32_t kAbortOff = 2 * 8 * kMaxStages;
constexpr uint32_t kWeightOff = 512;
constexpr uint32_t kWeightStride = kMaxWindow + 4;  // floats per consumer warp: w_0..w_63, P
constexpr uint32_t kWarpBufOff = 3072;  // per-consumer-warp fp32 token-chunk buffers start here
static_assert(kWeightOff + kConsumerWarps * kWeightStride * 4 <= kWarpBufOff, "smem head overflow");
constexpr int kTokChunk = 8;  // tokens converted to fp32 per consumer-warp pass
// Ring rows of prefixes this long or longer are fetched as 16-byte cp.async
// chunks spread over the loader's lanes; shorter ones as one bulk copy per row.
constexpr int kChunkedRingMinK = 32;

// How the consumer warps tile a [dim, dstate] state tile.  Each thread owns
// RPT consecutive rows x VEC consecutive columns (one vector per row).
// Inside a warp, LPR lanes cover one row (LPR*VEC columns), RPW rows side by
// side; the tile's column span is split into CT column tiles and its rows into
// SLABS slabs, one (column tile, slab) per warp.
struct ThreadLayout {
  int vec, tct, lpr, rpw, ct, slabs, slab_rows, rpt, cols;
};

__host__ __device__ constexpr ThreadLayout thread_layout(int dim, int dstate, int state_bytes,
                                                         int cw = kConsumerWarps) {
  // 16-byte vectors, except one-byte formats: 8 codes (8 bytes), with a whole
  // row inside one warp so that the row's amax is a warp reduction
  const int vec = state_bytes == 1 ? 8 : 16 / state_bytes;
  const int tct = dstate / vec;
  const int lpr = state_bytes == 1 ? tct : (tct < 8 ? tct : 8);
  const int rpw = 32 / lpr;
  const int ct = tct / lpr;
  const int slabs = cw / ct;
  const int slab_rows = dim / slabs;
  const int rpt = slab_rows >= rpw ? slab_rows / rpw : 1;
  return ThreadLayout{vec, tct, lpr, rpw, ct, slabs, slab_rows, rpt, lpr * vec};
}

// fp32 floats in one consumer warp's token-chunk buffer: c = w*x for its
// slab's rows and B for its column tile, kTokChunk tokens each.
__host__ __device__ constexpr uint32_t warp_buf_floats(int dim, int dstate, int state_bytes,
                                                       int cw = kConsumerWarps) {
  return static_cast<uint32_t>(kTokChunk * (thread_layout(dim, dstate, state_bytes, cw).slab_rows +
                                            thread_layout(dim, dstate, state_bytes, cw).cols));
}

__host__ __device__ constexpr uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

constexpr uint32_t kDescBytes = 48;  // sizeof(ItemDesc)

// Offset of the descriptor table: the fixed head plus the consumer warps' buffers.
__host__ __device__ constexpr uint32_t desc_base(int dim, int dstate, int state_bytes, int cw = kConsumerWarps) {
  return round_up(kWarpBufOff + cw * warp_buf_floats(dim, dstate, state_bytes, cw) * 4u, 128u);
}

// Offset of the item arena (after one descriptor per pipeline slot).
__host__ __device__ constexpr uint32_t arena_base(int dim, int dstate, int state_bytes, int cw = kConsumerWarps) {
  return round_up(desc_base(dim, dstate, state_bytes, cw) + kMaxStages * kDescBytes, 128u);
}

// The one-byte kernel's token buffer: each of its warps owns a 16-row slab,
// stored as (c, c) pairs (a pair feeds a packed fp32x2 FMA without a register
// move), and B for all 128 columns, kTokChunk tokens each.
constexpr uint32_t kQ8WarpBufFloats = kTokChunk * (2 * 16 + 128);
constexpr uint32_t kQ8DescBase = round_up(kWarpBufOff + kQ8ConsumerWarps * kQ8WarpBufFloats * 4u, 128u);
constexpr uint32_t kQ8ArenaBase = round_up(kQ8DescBase + kMaxStages * kDescBytes, 128u);

// Byte layout of one work item in the arena: the source tile at offset 0, its
// scales (one-byte formats), then the item's own k ring rows of x, of B (left
// out for an item that reuses the previous item's B) and its k dt values per
// head (`heads` > 1: an item of consecutive heads, whose tiles, scales and x
// rows are adjacent and counted in `dim`; head j's dt at off_dt + 4 j k).
// Every part starts on a 16-byte boundary (D*N*ES, D*IE and N*IE are
// multiples of 16); items start on 128-byte boundaries.
struct ItemLayout {
  uint32_t off_scale, off_x, off_B, off_dt, bytes;
};

__host__ __device__ constexpr ItemLayout item_layout(int dim, int dstate, int state_bytes, bool quant, int in_bytes,
                                                     int k, bool with_B = true, int heads = 1) {
  const uint32_t off_scale = static_cast<uint32_t>(dim * dstate * state_bytes);
  const uint32_t off_x = off_scale + (quant ? static_cast<uint32_t>(dim) * 4u : 0u);
  const uint32_t off_B = off_x + static_cast<uint32_t>(k * dim * in_bytes);
  const uint32_t off_dt = off_B + (with_B ? static_cast<uint32_t>(k * dstate * in_bytes) : 0u);
  return ItemLayout{off_scale, off_x, off_B, off_dt,
                    round_up(off_dt + 4u * static_cast<uint32_t>(k * heads), 128u)};
}

// Arena offset of the next item, given where the previous one ended (`head`):
// there if an item of the longest window would still end inside the arena,
// else at 0.  It depends on the sizes of the items alone, so the loader that
// places the items and the consumers that read them agree without exchanging
// offsets.
__host__ __device__ constexpr uint32_t arena_next(uint32_t head, uint32_t item_max, uint32_t arena_bytes) {
  return head + item_max <= arena_bytes ? head : 0u;
}

// Shared memory of the tensor-core (long-window) variant: the same head up to
// kWarpBufOff, then its mbarriers and the TMEM address word, the two MMA
// operands, the descriptor table and the arena.  Its consumer warps form two
// groups: a builder group (operands, MMA issue) and an epilogue group (TMEM ->
// state), joined by two TMEM accumulators so that consecutive items overlap.
constexpr int kTcMinWindow = 16;                  // tensor path for max_window >= this (16-bit state)
constexpr int kTcKMax = kMaxWindow;               // tokens one item's MMA covers at most
// CTA of the tensor-core kernel: the loader warp, kTcBuilderWarps builder
// warps and four epilogue warps (one per TMEM lane quarter); eight warps, so
// that two CTAs per SM leave 128 registers a thread.
constexpr int kTcBuilderWarps = 3;
constexpr int kTcEpilogueWarps = 4;
constexpr int kTcConsumerWarps = kTcBuilderWarps + kTcEpilogueWarps;
constexpr int kTcThreads = 32 * (1 + kTcConsumerWarps);
constexpr uint32_t kTcBarOff = kWarpBufOff;       // mbarriers, see below
constexpr uint32_t kTcMmaDone = kTcBarOff;        // [2] an accumulator's MMAs completed (1 arrival: commit)
constexpr uint32_t kTcTmemFree = kTcBarOff + 16;  // [2] the epilogue read an accumulator (kTcEpilogueWarps)
constexpr uint32_t kTcBuildBar = kTcBarOff + 32;  // the builder group's operands are written (kTcBuilderWarps)
constexpr uint32_t kTcExitBar = kTcBarOff + 40;   // every consumer warp is done with TMEM (kTcConsumerWarps)
constexpr uint32_t kTcTmemSlot = kTcBarOff + 48;  // TMEM base address written by tcgen05.alloc
// The two MMA operands, MN-major with the 128-byte swizzle: a token's row of
// the operand is a contiguous 64-element (128-byte) row of a swizzle atom
// (8 token rows, 1024 bytes, 1024-byte aligned), 16-byte chunk c of row r
// stored at chunk c ^ r.  C^T = (w x)^T (64 dim rows): one atom column, token
// groups of 8 rows 1024 bytes apart.  A = B^T (128 dstate columns): two atom
// columns 1024 bytes apart, token groups 2048 bytes apart.
// fp16 state: C = w x goes in as two bf16 operands, hi (c with its low 16
// bits cleared) and lo (the remainder, rounded to bf16), so that each term
// keeps 16 significant bits (2^-16 relative) instead of bf16's 8 (2^-9, coarser
// than fp16's own 2^-11).  Token group g of C^T is then followed by its lo
// rows (hi at 2048 g, lo at 2048 g + 1024).  Up to eight tokens, one MMA
// (K = 16) takes their hi and lo rows against the same eight rows of A, read
// twice (the A descriptor's K stride is 0); longer items read C^T as 128 rows
// (hi rows, then lo rows: atom columns 1024 bytes apart) into N = 128.
__host__ __device__ constexpr bool tc_split_c(int sf) { return sf == RSM_F16; }
constexpr uint32_t kTcBOff = 4096;  // C^T: 64 x kTcKMax bf16 (8 KiB), with lo rows 16 KiB
__host__ __device__ constexpr uint32_t tc_c_group(int sf) { return tc_split_c(sf) ? 2048u : 1024u; }
__host__ __device__ constexpr uint32_t tc_a_off(int sf) {  // A: 128 x kTcKMax bf16 (16 KiB)
  return kTcBOff + (tc_split_c(sf) ? 2u : 1u) * 64u * kTcKMax * 2u;
}
constexpr uint32_t kTcAGroup = 2048;  // bytes between token groups of A
static_assert(kTcBarOff + 128 <= kTcBOff && kTcBOff % 1024 == 0 && tc_a_off(RSM_BF16) % 1024 == 0 &&
                  tc_a_off(RSM_F16) % 1024 == 0,
              "operand alignment");
// One fp32 accumulator: 128 lanes x 64 columns, and for fp16 state 64 more
// (an item of more than eight tokens takes its hi and lo products separately:
// one MMA of N = 128 per 16 tokens, C^T's token groups read as 128 rows, hi
// then lo; the epilogue adds the two halves).
constexpr uint32_t kTcAccCols = 128;
constexpr uint32_t kTcLoCols = 64;                // the lo half of an accumulator
constexpr uint32_t kTcTmemCols = 2 * kTcAccCols;  // two accumulators
__host__ __device__ constexpr uint32_t tc_desc_base(int sf) { return round_up(tc_a_off(sf) + 128u * kTcKMax * 2u, 128u); }
__host__ __device__ constexpr uint32_t tc_arena_base(int sf) {
  return round_up(tc_desc_base(sf) + kMaxStages * kDescBytes, 128u);
}
constexpr int kTcMinK = 1;  // every prefix of one token or more goes through the MMA

// The one-byte tensor-core kernel (rsm_q8tc_kernel.cuh): items of two heads
// of one B group (HPI = 2), the replay sum_t w_t x_t B_t^T as MMAs of M = 128
// (two heads x 64 dim rows) x N = 128 (dstate) x K = 16 tokens.  CTA: the
// loader warp, two builder warps (one per head of the item) and four epilogue
// warps (one per TMEM lane quarter, a thread per tile row).  Two accumulators
// of 128 columns.
constexpr int kQtHeads = 2;
constexpr int kQtBuilderWarps = 2;
constexpr int kQtEpilogueWarps = 4;
constexpr int kQtConsumerWarps = kQtBuilderWarps + kQtEpilogueWarps;
constexpr int kQtThreads = 32 * (1 + kQtConsumerWarps);
constexpr int kQtMaxRegs = 128;  // 14 warps per SM at two CTAs: four on three sub-partitions, 4 x 32 x 128 = 16384
constexpr uint32_t kQtMmaDone = kWarpBufOff;       // [2] an accumulator's MMAs completed (1 arrival: commit)
constexpr uint32_t kQtTmemFree = kWarpBufOff + 16; // [2] the epilogue is done with an accumulator (kQtEpilogueWarps)
constexpr uint32_t kQtBuildBar = kWarpBufOff + 32; // the builders' operands are written (kQtBuilderWarps)
constexpr uint32_t kQtExitBar = kWarpBufOff + 40;  // every consumer warp is done with TMEM (kQtConsumerWarps)
constexpr uint32_t kQtTmemSlot = kWarpBufOff + 48; // TMEM base address written by tcgen05.alloc
constexpr uint32_t kQtAccCols = 128;               // one fp32 accumulator: 128 lanes x 128 columns
constexpr uint32_t kQtTmemCols = 2 * kQtAccCols;
constexpr uint32_t kQtOpOff = 4096;                // operands from here, 1024-byte aligned
constexpr uint32_t kQtGroup = 2048;                // bytes between token groups of 8 rows (two atom columns)
constexpr uint32_t kQtStageBytes = 32 * 128;       // one epilogue warp's store staging: 32 rows x 128 codes
static_assert(kQtMmaDone + 64 <= kQtOpOff && kWeightOff + kQtBuilderWarps * kWeightStride * 4 <= kWarpBufOff,
              "one-byte tensor-core smem head");
// tokens of one item's MMAs (the window rounded up to whole MMAs of 16)
__host__ __device__ constexpr uint32_t qt_kpad(int window) { return round_up(static_cast<uint32_t>(window), 16u); }
// bytes of one operand: 128 rows (MN) x kpad tokens of bf16, a multiple of 4096
__host__ __device__ constexpr uint32_t qt_op_bytes(int window) { return 128u * qt_kpad(window) * 2u; }
// [C hi | C lo | B] operands, then the epilogue warps' staging, the descriptors and the arena
__host__ __device__ constexpr uint32_t qt_stage_off(int window) { return kQtOpOff + 3u * qt_op_bytes(window); }
__host__ __device__ constexpr uint32_t qt_desc_base(int window) {
  return qt_stage_off(window) + kQtEpilogueWarps * kQtStageBytes;
}
__host__ __device__ constexpr uint32_t qt_arena_base(int window) {
  return round_up(qt_desc_base(window) + kMaxStages * kDescBytes, 128u);
}

struct Params {
  const int64_t* state_ptrs;
  const int64_t* state_strides;
  const int64_t* x_ptrs;
  const int64_t* x_strides;
  const int64_t* B_ptrs;
  const int64_t* B_strides;
  const int64_t* dt_ptrs;
  const int64_t* dt_strides;
  const int64_t* A_ptrs;
  const int64_t* scale_ptrs;
  const int64_t* scale_strides;
  const int32_t* src_slots;
  const int32_t* dst_slots;
  const int32_t* ring_start;
  const int32_t* prefix_len;
  const int32_t* active;
  const int64_t* rand_seed;
  uint32_t* status;
  int32_t L, Bt, H, hpg, W, R, pad, philox_rounds;
  int32_t num_slots;  // slots per pool; a slot >= num_slots is skipped (0: not checked)
  int32_t tc_min_k;  // tensor-core variant: prefixes this long or longer go to the MMA (0: no tensor path)
  // shared-memory plan: descriptor table at desc0, item arena of arena_bytes at
  // arena0, `stages` pipeline slots (mbarrier pairs and descriptors)
  uint32_t desc0, arena0, arena_bytes, stages;
};

}  // namespace rsm
