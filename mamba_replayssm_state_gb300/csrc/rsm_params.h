// rsm_params.h -- launch parameters and the shared-memory plan of the
// materialization kernel, shared by the host launcher and the kernel.
#pragma once
#include <cstdint>

namespace rsm {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kThreads = 32 + kConsumerThreads;
constexpr int kMaxWindow = 64;
constexpr int kMaxStages = 16;
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s: never reached by a correct run

// Shared memory head: [full mbarriers][empty mbarriers] | abort flag | per-warp
// decay weights | stages...
constexpr uint32_t kAbortOff = 2 * 8 * kMaxStages;
constexpr uint32_t kWeightOff = 512;
constexpr uint32_t kWeightStride = kMaxWindow + 4;  // floats per consumer warp: w_0..w_63, P
constexpr uint32_t kStageBase = 3072;
static_assert(kWeightOff + kConsumerWarps * kWeightStride * 4 <= kStageBase, "smem head overflow");

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
  // shared-memory plan (see make_plan)
  uint32_t stages, stage_bytes, off_state, off_scale, off_x, off_B, off_dt;
};

struct Plan {
  uint32_t stage_bytes, off_state, off_scale, off_x, off_B, off_dt;
};

__host__ __device__ constexpr uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Byte layout of one pipeline stage.
__host__ __device__ inline Plan make_plan(int dim, int dstate, int state_bytes, bool quant, int in_bytes,
                                          int max_window) {
  Plan p{};
  p.off_state = 128;
  p.off_scale = round_up(p.off_state + dim * dstate * state_bytes, 128);
  p.off_x = round_up(p.off_scale + (quant ? dim * 4 : 0), 128);
  p.off_B = round_up(p.off_x + max_window * dim * in_bytes, 128);
  p.off_dt = round_up(p.off_B + max_window * dstate * in_bytes, 128);
  p.stage_bytes = round_up(p.off_dt + max_window * 4, 128);
  return p;
}

}  // namespace rsm
