// gdn_params.h -- constants, descriptor, arena item layout and launch
// parameters of the gated-delta-rule commit kernel, shared by the host
// launcher and the kernel.
#pragma once
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

}  // namespace gdn
