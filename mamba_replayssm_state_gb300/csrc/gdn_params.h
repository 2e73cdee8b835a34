// gdn_params.h -- constants, descriptor, arena item layout and launch
// parameters of the gated-delta-rule commit kernel, shared by the host
// launcher and the kernel.
#pragma once
#include <cuda.h>  // CUtensorMap (the tcgen05 backend's tensor map; no driver call is made here)

#include <cstdint>

#include "rsm_params.h"

namespace gdn {

using rsm::round_up;

constexpr int kDK = 128, kDV = 128;
constexpr int kSlabRows = 64;
constexpr int kSlabs = kDV / kSlabRows;
constexpr uint32_t kSlabBytes = kSlabRows * kDK * 4;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kMaxWindow = 64;
constexpr int kMaxSlots = 16;
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;
static_assert(kConsumerWarps * 8 == kSlabRows, "eight rows per consumer warp (two per lane)");

// shared memory: [full mbarriers][empty mbarriers] | abort flag | descriptors |
// per-consumer-warp token tables (exp(g), beta, 1/|k|, exp(-g) per token) | arena
constexpr uint32_t kAbortOff = 2 * 8 * kMaxSlots;
constexpr uint32_t kDescOff = 512;
constexpr uint32_t kDescBytes = 32;
constexpr uint32_t kTokOff = kDescOff + kMaxSlots * kDescBytes;      // 1024
constexpr uint32_t kTokBytes = kMaxWindow * 16;                      // one float4 per token
constexpr uint32_t kArenaOff = kTokOff + kConsumerWarps * kTokBytes;  // 9216

struct alignas(16) Desc {
  unsigned long long slab;   // global address of the slab (read and written in place)
  unsigned long long track;  // global address of the track slab, 0 if none
  int32_t n;                 // accepted tokens
  int32_t step;              // token after which the track copy is taken (valid if track != 0)
  uint32_t flags;
  uint32_t unused;
};
static_assert(sizeof(Desc) == kDescBytes, "descriptor size");
constexpr uint32_t kFlagEnd = 1u;

// Arena layout of one item with n tokens: slab | k rows (n x 256 B) |
// v (n x 64 B: the slab's rows) | g (n x 4 B) | beta (n x 4 B).
struct Item {
  uint32_t off_k, off_v, off_g, off_beta, bytes;
};
__host__ __device__ constexpr Item item_layout(int n) {
  const uint32_t off_k = kSlabBytes;
  const uint32_t off_v = off_k + static_cast<uint32_t>(n) * kDK * 2u;
  const uint32_t off_g = off_v + static_cast<uint32_t>(n) * kSlabRows * 2u;
  const uint32_t off_beta = off_g + static_cast<uint32_t>(n) * 4u;
  return Item{off_k, off_v, off_g, off_beta, round_up(off_beta + static_cast<uint32_t>(n) * 4u, 128u)};
}

struct Params {
  float* state;
  const uint16_t* rawv;
  const uint16_t* rawk;
  const float* g;
  const float* beta;
  const int32_t* state_indices;
  const int32_t* accept_lens;
  const int32_t* track_indices;  // NULL: no tracking
  const int32_t* track_steps;
  uint32_t* status;
  int32_t L, SL, HV, H, T, B, l2norm, null_id;
  uint32_t arena_bytes, slots;
};

// Address of the kernel (defined in gdn_inst.cu).
const void* commit_kernel();

// ---------------------------------------------------------------------------
// The tcgen05 backend (gdn_tc_kernel.cuh): TF32 tensor-core contractions for
// normalised K, windows of 4 to 8 tokens, without tracking (GDN page,
// Parameters: backend).  One CTA per SM: a loader warp, a builder warp and
// four epilogue warps; a work item is one value head's whole 128 x 128 state.
// ---------------------------------------------------------------------------
constexpr int kTcMinT = 4, kTcMaxT = 8;
constexpr int kTcWarps = 6;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr uint32_t kTcHeadBytes = kDV * kDK * 4;  // 64 KiB of fp32 state
constexpr uint32_t kTcBoxBytes = kDV * 32 * 4;    // one tensor-map box: 128 rows x 32 columns
// shared memory: [full][empty] mbarriers | abort flag | item descriptors (as
// above, to 1024) | the backend's mbarriers | coefficient tables | two
// operand buffers | the arena (1024-byte aligned items)
constexpr uint32_t kTcBar = 1024;
constexpr uint32_t kTcMma1Done = kTcBar;        // [2] S0 k^ in the small accumulator (commit)
constexpr uint32_t kTcTabReady = kTcBar + 16;   // [2] the builder's tables and operands (1 arrival)
constexpr uint32_t kTcA2Ready = kTcBar + 32;    // [2] the epilogue's U operand (4 warps)
constexpr uint32_t kTcMma2Done = kTcBar + 48;   // [2] the update in the large accumulator (commit)
constexpr uint32_t kTcStReady = kTcBar + 64;    // [2] the new state written over S0 in the slot (4 warps)
constexpr uint32_t kTcDFree = kTcBar + 80;      // [2] the epilogue is done with both accumulators (4 warps)
constexpr uint32_t kTcExit = kTcBar + 96;       // every consumer warp is done with TMEM (5 warps)
constexpr uint32_t kTcTmemSlot = kTcBar + 104;  // TMEM base address written by tcgen05.alloc
constexpr uint32_t kTcTabOff = 2048;            // [2] x kTcTabFloats: gamma[8], coef[8], L[8][8]
constexpr uint32_t kTcTabFloats = 96;
constexpr uint32_t kTcOpOff = 4096;             // [2] x 16 KiB: B1 (8 KiB), B2 (4 KiB), A2 (4 KiB)
constexpr uint32_t kTcOpBytes = 16384;
constexpr uint32_t kTcB1 = 0, kTcB2 = 8192, kTcA2 = 12288;
constexpr uint32_t kTcArenaOff = kTcOpOff + 2 * kTcOpBytes;  // 36864
constexpr uint32_t kTcTmemCols = 512;           // D1[2] at 0, 32; D2[2] at 64, 192
static_assert(kTcTmemSlot + 4 <= kTcTabOff && kTcTabOff + 2 * kTcTabFloats * 4 <= kTcOpOff, "tc smem head");
static_assert(kMaxSlots * kDescBytes + kDescOff <= kTcBar, "descriptor table");

struct alignas(16) TcDesc {
  int32_t row0;    // the head's first row in the [rows, 128] view of checkpoint_state
  int32_t n;       // accepted tokens, 1 .. window
  uint32_t flags;
  uint32_t unused[5];
};
static_assert(sizeof(TcDesc) == kDescBytes, "descriptor size");

// Arena layout of one item with n tokens: state (64 KiB, swizzled) | k rows
// (n x 256 B) | v rows (n x 256 B) | g (8 floats) | beta (8 floats).
struct TcItem {
  uint32_t off_k, off_v, off_g, off_beta, bytes;
};
__host__ __device__ constexpr TcItem tc_item_layout(int n) {
  const uint32_t off_k = kTcHeadBytes;
  const uint32_t off_v = off_k + static_cast<uint32_t>(n) * kDK * 2u;
  const uint32_t off_g = off_v + static_cast<uint32_t>(n) * kDV * 2u;
  const uint32_t off_beta = off_g + kTcMaxT * 4u;
  return TcItem{off_k, off_v, off_g, off_beta, round_up(off_beta + kTcMaxT * 4u, 1024u)};
}

struct TcParams {
  CUtensorMap tmap;  // checkpoint_state as [layers*slots*HV*128 rows, 128] fp32, boxes of 128 x 32, 128-byte swizzle
  Params p;
};

// Address of the tcgen05-backend kernel (gdn_inst.cu).
const void* commit_tc_kernel();

}  // namespace gdn
