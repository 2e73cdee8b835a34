// gdn_tc_kernel.cuh -- the tcgen05 backend of the gated-delta-rule commit
// (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit, API page:
// Parameters, backend: TF32 tensor-core contractions for normalised K,
// windows of 4 to 8 tokens, without tracking).
//
// For one value head with state S_0 (128 value rows x 128 key columns), n
// accepted tokens with normalised keys k^_t, values v_t, decays a_t = exp(g_t)
// and beta_t, the sequential update
//   S_t = a_t S_{t-1} + beta_t u_t k^_t^T,   u_t = v_t - a_t S_{t-1} k^_t,
// unrolls (g_t = a_0 ... a_t) into
//   S_n = g_{n-1} S_0 + sum_s c_s u_s k^_s^T,        c_s = beta_s g_{n-1} / g_s,
//   u_t = v_t - g_t (S_0 k^_t) - sum_{s<t} L_st u_s, L_st = beta_s (g_t / g_s) (k^_s . k^_t):
// two contractions with the whole state, W = S_0 K^ (128 x n) and the rank-n
// update U K^^T (128 x 128), and a triangular solve of n <= 8 unknowns per row
// in between.  The contractions run on the tensor cores with TF32 operands
// (tcgen05.mma kind::tf32), the solve and g_{n-1} S_0 in fp32 on the CUDA cores.
//
// A work item is one value head.  One CTA per SM: a loader warp, a builder
// warp and four epilogue warps (one per TMEM lane quarter, a thread per value
// row), joined by the slot/arena pipeline of the fp32 kernel:
//   loader: the head's state through the tensor map (four boxes of 128 rows x
//     32 columns, 128-byte swizzle: the K-major SW128 layout the MMA reads),
//     the accepted k and v rows (bulk copies), g and beta (4-byte copies);
//   builder: k^ (rsqrt of |k|^2 + 1e-6, as the fp32 kernel), the MMA operands
//     K^ (16 token rows, K-major SW128) and K^^T (K-major, no swizzle), the
//     coefficient table (g_t, c_t, L_st), then the 16 MMAs of W = S_0 K^
//     (M = 128, N = 16, K = 8 each) into the small accumulator of buffer n % 2;
//   epilogue: W from TMEM, the solve for its row, U (its row of c_s u_s) into
//     the second A operand; one thread issues the update MMA (M = N = 128,
//     K = 8) into the large accumulator; then each thread writes
//     g_{n-1} S_0 + update over its row of S_0 in the slot, and one thread
//     stores the head back in place through the tensor map and releases the
//     slot once the store has read it.
// Operands, tables and accumulators are double-buffered by item parity.
// Every wait is bounded in wall time; TMEM (512 columns) is allocated by the
// builder warp and freed by it after an exit barrier.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "../../include/replayssm.h"
#include "gdn_params.h"
#include "rsm_ptx.cuh"
#include "rsm_tc.cuh"

namespace gdn {

using rsm::arena_next;
using rsm::bulk_g2s;
using rsm::cp_async_4;
using rsm::cp_async_mbar_arrive;
using rsm::fence_proxy_async_smem;
using rsm::mbar_arrive;
using rsm::mbar_expect_tx;
using rsm::mbar_init;
using rsm::mbar_wait;
using rsm::smem_addr;

__device__ __forceinline__ void tc_flag(uint32_t* status, uint32_t bits) {
  if (status != nullptr && bits != 0u) atomicOr(status, bits);
}

__device__ __forceinline__ void tc_abort(const Params& p, volatile int* abort_flag, int lane) {
  if (lane == 0) {
    *abort_flag = 1;
    tc_flag(p.status, RSM_STATUS_WAIT_TIMEOUT);
  }
}

// bounded wait with the whole warp agreeing; false on time-out or abort
__device__ __forceinline__ bool tc_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, kWaitTimeoutNs) && !*abort_flag;
  return __all_sync(0xFFFFFFFFu, ok);
}

// tensor-map copies (2-D tile mode): global -> shared completing on an
// mbarrier's transaction count, and shared -> global in a bulk group
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the bulk groups of this thread have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and their writes are done
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Instruction descriptor of kind::tf32: TF32 A and B, fp32 accumulator, both
// operands K-major, an M x N tile.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int m, int n) {
  return (1u << 4) |                              // D format: fp32
         (2u << 7) |                              // A format: tf32
         (2u << 10) |                             // B format: tf32
         (static_cast<uint32_t>(n >> 3) << 17) |  // N / 8
         (static_cast<uint32_t>(m >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor without swizzle, K-major: core matrices of 8 rows x
// 16 bytes (128 contiguous bytes); `lbo` = bytes between core matrices
// adjacent along K, `sbo` = along M/N.
__device__ __forceinline__ uint64_t smem_desc_noswizzle(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
         (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// ---------------------------------------------------------------------------
// loader warp
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_run_loader(const TcParams& tp, unsigned char* smem, int lane) {
  const Params& p = tp.p;
  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8u * kMaxSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);

  // units: (request b, layer l, a run of `chunk` value heads), request-major,
  // dealt to the CTAs round-robin
  const int64_t heads = static_cast<int64_t>(p.B) * p.L * p.HV;
  const int chunk = static_cast<int>(
      min(static_cast<int64_t>(8), max(static_cast<int64_t>(1), heads / (16 * static_cast<int64_t>(gridDim.x)))));
  const int units_per_seg = (p.HV + chunk - 1) / chunk;
  const int64_t total_units = static_cast<int64_t>(p.B) * p.L * units_per_seg;
  const int per_kh = p.HV / p.H;

  uint32_t stage = 0, phase = 0, fills = 0;
  bool aborted = false;
  const uint32_t item_max = tc_item_layout(p.T).bytes;
  uint32_t head = 0, tail = 0, n_out = 0;
  bool wrapped = false;
  uint32_t slot_start = 0;
  uint32_t oldest = 0, oldest_phase = 0;
  auto free_oldest = [&]() -> bool {
    if (!mbar_wait(empty0 + 8u * oldest, oldest_phase, kWaitTimeoutNs)) return false;
    if (++oldest == p.slots) {
      oldest = 0;
      oldest_phase ^= 1u;
    }
    --n_out;
    const uint32_t next = __shfl_sync(0xFFFFFFFFu, slot_start, static_cast<int>(oldest));
    if (n_out == 0) {
      tail = head;
      wrapped = false;
    } else {
      if (next < tail) wrapped = false;
      tail = next;
    }
    return true;
  };
  auto alloc = [&](uint32_t bytes, uint32_t& off) -> bool {
    off = arena_next(head, item_max, p.arena_bytes);
    for (;;) {
      if (n_out == 0) break;
      if (n_out < p.slots) {
        if (off == head) {
          if (!wrapped || head + bytes <= tail) break;
        } else if (!wrapped && bytes <= tail) {
          break;
        }
      }
      if (!free_oldest()) return false;
    }
    if (n_out == 0) {
      tail = off;
      wrapped = false;
    } else if (off != head) {
      wrapped = true;
    }
    return true;
  };

  int cur_b = -1, s = 0, n = 0;
  bool ok = false;
  for (int64_t u = blockIdx.x; u < total_units && !aborted; u += gridDim.x) {
    const int64_t seg = u / units_per_seg;
    const int b = static_cast<int>(seg / p.L);
    const int l = static_cast<int>(seg - static_cast<int64_t>(b) * p.L);
    const int hv0 = static_cast<int>(u - seg * units_per_seg) * chunk;
    const int hv_end = min(p.HV, hv0 + chunk);
    if (b != cur_b) {
      cur_b = b;
      s = __ldg(p.state_indices + b);
      n = __ldg(p.accept_lens + b);
      uint32_t bad = 0;
      ok = s > p.null_id && n != 0;
      if (ok && (s >= p.SL || n < 0 || n > p.T)) {
        bad |= s >= p.SL ? RSM_STATUS_BAD_SLOT : RSM_STATUS_BAD_PREFIX_LEN;
        ok = false;
      }
      if (lane == 0) tc_flag(p.status, bad);
    }
    if (!ok) continue;
    const TcItem it = tc_item_layout(n);
    const int64_t lay_slot = static_cast<int64_t>(l) * p.SL + s;
    for (int hv = hv0; hv < hv_end; ++hv) {
      const int hk = hv / per_kh;
      uint32_t off = 0;
      if (!alloc(it.bytes, off)) {
        aborted = true;
        break;
      }
      unsigned char* sb = smem + kTcArenaOff + off;
      const uint32_t sba = smem_addr(sb);
      const uint32_t fullb = full0 + 8u * stage;
      TcDesc* desc = reinterpret_cast<TcDesc*>(smem + kDescOff) + stage;
      const int row0 = static_cast<int>((lay_slot * p.HV + hv) * kDV);
      const uint16_t* krows = p.rawk + (lay_slot * p.H + hk) * p.T * kDK;
      const uint16_t* vrows = p.rawv + (lay_slot * p.HV + hv) * p.T * kDV;
      const float* grow = p.g + (lay_slot * p.HV + hv) * p.T;
      const float* brow = p.beta + (lay_slot * p.HV + hv) * p.T;
      if (lane == 0) {
        desc->row0 = row0;
        desc->n = n;
        desc->flags = 0u;
        fence_proxy_async_smem();
        mbar_expect_tx(fullb, kTcHeadBytes + static_cast<uint32_t>(n) * (kDK + kDV) * 2u);
      }
      __syncwarp();
      if (lane < 4) tma_load_2d(sba + lane * kTcBoxBytes, &tp.tmap, 32 * lane, row0, fullb);
      if (lane == 4) bulk_g2s(sba + it.off_k, krows, static_cast<uint32_t>(n) * kDK * 2u, fullb);
      if (lane == 5) bulk_g2s(sba + it.off_v, vrows, static_cast<uint32_t>(n) * kDV * 2u, fullb);
      if (lane < n) {
        cp_async_4(sba + it.off_g + 4u * lane, grow + lane);
        cp_async_4(sba + it.off_beta + 4u * lane, brow + lane);
      }
      cp_async_mbar_arrive(fullb);
      __syncwarp();
      if (lane == 0) mbar_arrive(fullb);
      if (lane == static_cast<int>(stage)) slot_start = off;
      head = off + it.bytes;
      ++n_out;
      ++fills;
      if (++stage == p.slots) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }

  bool ended = false;
  if (!aborted) {
    bool fine = true;
    while (fine && n_out >= p.slots) fine = free_oldest();
    if (fine) {
      if (lane == 0) (reinterpret_cast<TcDesc*>(smem + kDescOff) + stage)->flags = kFlagEnd;
      __syncwarp();
      if (lane == 0) mbar_arrive(full0 + 8u * stage);
      ended = true;
    }
  }
  if (!ended) {
    if (lane == 0) {
      *abort_flag = 1;
      tc_flag(p.status, RSM_STATUS_WAIT_TIMEOUT);
    }
    // let copies already issued into the arena land before the CTA exits
    for (uint32_t q = 0; q < p.slots; ++q) {
      if (q < stage)
        (void)mbar_wait(full0 + 8u * q, phase, 1000000ull);
      else if (fills >= p.slots)
        (void)mbar_wait(full0 + 8u * q, phase ^ 1u, 1000000ull);
    }
  }
}

// ---------------------------------------------------------------------------
// builder warp: k^, the operands K^ and K^^T, the coefficient table, W = S_0 K^
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_run_builder(const TcParams& tp, unsigned char* smem, int lane, uint32_t tmem) {
  const Params& p = tp.p;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  constexpr uint32_t kIdesc1 = idesc_tf32_f32(128, 16);
  const uint32_t item_max = tc_item_layout(p.T).bytes;
  uint32_t arena_head = 0, stage = 0, phase = 0, n_it = 0;
  for (;;) {
    if (!tc_wait_warp(full0 + 8u * stage, phase, abort_flag)) {
      tc_abort(p, abort_flag, lane);
      break;
    }
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    const unsigned char* sb = smem + kTcArenaOff + off;
    const TcDesc* desc = reinterpret_cast<const TcDesc*>(smem + kDescOff) + stage;
    if (desc->flags & kFlagEnd) break;
    const int n = desc->n;
    const TcItem it = tc_item_layout(n);
    arena_head = off + it.bytes;
    if (++stage == p.slots) {
      stage = 0;
      phase ^= 1u;
    }
    const uint32_t buf = n_it & 1u;
    unsigned char* op = smem + kTcOpOff + buf * kTcOpBytes;
    float* tab = reinterpret_cast<float*>(smem + kTcTabOff) + buf * kTcTabFloats;
    // this buffer's operands and accumulators are free once the epilogue is
    // done with the item two back (its update MMA read them before)
    if (n_it >= 2 && !tc_wait_warp(sbase + kTcDFree + 8u * buf, ((n_it - 2) >> 1) & 1u, abort_flag)) {
      tc_abort(p, abort_flag, lane);
      break;
    }
    // k^: this lane's keys 4 lane .. 4 lane + 3 of every accepted token
    float kh[kTcMaxT][4];
#pragma unroll
    for (int t = 0; t < kTcMaxT; ++t) {
      const uint2 w = t < n ? *reinterpret_cast<const uint2*>(sb + it.off_k + t * kDK * 2 + lane * 8) : make_uint2(0u, 0u);
      kh[t][0] = __uint_as_float(w.x << 16);
      kh[t][1] = __uint_as_float(w.x & 0xFFFF0000u);
      kh[t][2] = __uint_as_float(w.y << 16);
      kh[t][3] = __uint_as_float(w.y & 0xFFFF0000u);
      float ss = kh[t][0] * kh[t][0] + kh[t][1] * kh[t][1] + kh[t][2] * kh[t][2] + kh[t][3] * kh[t][3];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      const float r = rsqrtf(ss + 1e-6f);
#pragma unroll
      for (int e = 0; e < 4; ++e) kh[t][e] *= r;
    }
    // B1 = K^ (16 token rows x 128 keys, K-major, 128-byte swizzle): key block
    // kb = lane / 8 (32 keys), chunk c = lane % 8 of token row t at
    // kb * 2048 + t * 128 + (c ^ t % 8) * 16; rows n .. 15 zero
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int kb = lane >> 3, c = lane & 7;
      const float4 v = t < kTcMaxT ? make_float4(kh[t < kTcMaxT ? t : 0][0], kh[t < kTcMaxT ? t : 0][1],
                                                 kh[t < kTcMaxT ? t : 0][2], kh[t < kTcMaxT ? t : 0][3])
                                   : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      *reinterpret_cast<float4*>(op + kTcB1 + kb * 2048 + t * 128 + (((c ^ t) & 7) << 4)) = v;
    }
    // B2 = K^^T (128 keys x 8 tokens, K-major without swizzle): key j's tokens
    // 4g .. 4g + 3 at g * 2048 + (j / 8) * 128 + (j % 8) * 16
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * lane + e;
#pragma unroll
      for (int g = 0; g < 2; ++g)
        *reinterpret_cast<float4*>(op + kTcB2 + g * 2048 + (j >> 3) * 128 + (j & 7) * 16) =
            make_float4(kh[4 * g][e], kh[4 * g + 1][e], kh[4 * g + 2][e], kh[4 * g + 3][e]);
    }
    // coefficients: g_t = prod_{r <= t} exp(g_r) (gamma), c_t = beta_t g_{n-1} / g_t,
    // L_st = beta_s (g_t / g_s) (k^_s . k^_t) for s < t
    const float* gs = reinterpret_cast<const float*>(sb + it.off_g);
    const float* bs = reinterpret_cast<const float*>(sb + it.off_beta);
    float gam[kTcMaxT];
    {
      float acc = 1.0f;
#pragma unroll
      for (int t = 0; t < kTcMaxT; ++t) {
        if (t < n) acc *= expf(gs[t]);
        gam[t] = acc;
      }
    }
    const float gN = gam[kTcMaxT - 1];  // = g_{n-1}: the product stops growing after token n-1
#pragma unroll
    for (int t = 0; t < kTcMaxT; ++t) {
#pragma unroll
      for (int s2 = 0; s2 < t; ++s2) {
        float d = kh[s2][0] * kh[t][0] + kh[s2][1] * kh[t][1] + kh[s2][2] * kh[t][2] + kh[s2][3] * kh[t][3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
        if (lane == 0) tab[16 + s2 * 8 + t] = t < n ? bs[s2] * (gam[t] / gam[s2]) * d : 0.0f;
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kTcMaxT; ++t) {
        tab[t] = gam[t];
        tab[8 + t] = t < n ? bs[t] * (gN / gam[t]) : 0.0f;
      }
    }
    fence_proxy_async_smem();  // B1, B2 written by this thread, before the tensor cores read them
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcTabReady + 8u * buf);
    rsm::tc_fence_before();
    __syncwarp();
    rsm::tc_fence_after();
    if (lane == 0) {
      // W = S_0 K^: A = the slot's state (four 16 KiB blocks of 32 keys), B =
      // B1 (four 2 KiB blocks); K = 8 tf32 (32 bytes) per MMA
      const uint32_t a0 = smem_addr(sb), b0 = sbase + kTcOpOff + buf * kTcOpBytes + kTcB1;
      for (int kb = 0; kb < 4; ++kb)
        for (int ks = 0; ks < 4; ++ks)
          tc_mma_tf32(tmem + buf * 32u, rsm::smem_desc_mn_sw128(a0 + kb * kTcBoxBytes + ks * 32, 16u, 1024u),
                      rsm::smem_desc_mn_sw128(b0 + kb * 2048 + ks * 32, 16u, 1024u), kIdesc1,
                      (kb | ks) != 0 ? 1u : 0u);
      rsm::tc_commit(sbase + kTcMma1Done + 8u * buf);
    }
    __syncwarp();
    ++n_it;
  }
}

// ---------------------------------------------------------------------------
// epilogue warps: thread = value row v (TMEM lane)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_run_epilogue(const TcParams& tp, unsigned char* smem, int ew, int warp, int lane,
                                                uint32_t tmem) {
  const Params& p = tp.p;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * kMaxSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  const int quarter = warp & 3;
  const int v = 32 * quarter + lane;  // value row = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
  constexpr uint32_t kIdesc2 = idesc_tf32_f32(128, 128);
  const bool leader = ew == 0 && lane == 0;  // issues the update MMA and the stores
  const uint32_t item_max = tc_item_layout(p.T).bytes;
  uint32_t arena_head = 0, stage = 0, phase = 0, n_it = 0;
  for (;;) {
    if (!tc_wait_warp(full0 + 8u * stage, phase, abort_flag)) {
      tc_abort(p, abort_flag, lane);
      break;
    }
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    unsigned char* sb = smem + kTcArenaOff + off;
    const TcDesc* desc = reinterpret_cast<const TcDesc*>(smem + kDescOff) + stage;
    if (desc->flags & kFlagEnd) break;
    const int n = desc->n, row0 = desc->row0;
    const TcItem it = tc_item_layout(n);
    arena_head = off + it.bytes;
    const uint32_t empty_bar = empty0 + 8u * stage;
    if (++stage == p.slots) {
      stage = 0;
      phase ^= 1u;
    }
    const uint32_t buf = n_it & 1u, par = (n_it >> 1) & 1u;
    unsigned char* op = smem + kTcOpOff + buf * kTcOpBytes;
    const float* tab = reinterpret_cast<const float*>(smem + kTcTabOff) + buf * kTcTabFloats;
    if (!tc_wait_warp(sbase + kTcTabReady + 8u * buf, par, abort_flag) ||
        !tc_wait_warp(sbase + kTcMma1Done + 8u * buf, par, abort_flag)) {
      tc_abort(p, abort_flag, lane);
      break;
    }
    rsm::tc_fence_after();
    // W[v][t] = (S_0 k^_t)[v], then u_t = v_t[v] - g_t W - sum_{s<t} L_st u_s
    float w16[16];
    rsm::tmem_ld16(lane_base + buf * 32u, w16);
    const uint16_t* vrows = reinterpret_cast<const uint16_t*>(sb + it.off_v);
    float u[kTcMaxT];
#pragma unroll
    for (int t = 0; t < kTcMaxT; ++t) {
      float r = 0.0f;
      if (t < n) {
        r = bf16f(vrows[t * kDV + v]) - tab[t] * w16[t];
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) r -= tab[16 + s2 * 8 + t] * u[s2];
      }
      u[t] = r;
    }
    // A2 = U (128 rows x 8 tokens, K-major without swizzle): row v's tokens
    // 4g .. 4g + 3 at g * 2048 + (v / 8) * 128 + (v % 8) * 16
#pragma unroll
    for (int g = 0; g < 2; ++g)
      *reinterpret_cast<float4*>(op + kTcA2 + g * 2048 + (v >> 3) * 128 + (v & 7) * 16) =
          make_float4(tab[8 + 4 * g] * u[4 * g], tab[8 + 4 * g + 1] * u[4 * g + 1], tab[8 + 4 * g + 2] * u[4 * g + 2],
                      tab[8 + 4 * g + 3] * u[4 * g + 3]);
    fence_proxy_async_smem();
    rsm::tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcA2Ready + 8u * buf);
    if (leader) {
      // the update MMA, once every epilogue warp has written its rows of U
      bool ok = mbar_wait(sbase + kTcA2Ready + 8u * buf, par, kWaitTimeoutNs) && !*abort_flag;
      if (ok) {
        rsm::tc_fence_after();
        const uint32_t ob = sbase + kTcOpOff + buf * kTcOpBytes;
        tc_mma_tf32(tmem + 64u + buf * 128u, smem_desc_noswizzle(ob + kTcA2, 2048u, 128u),
                    smem_desc_noswizzle(ob + kTcB2, 2048u, 128u), kIdesc2, 0u);
        rsm::tc_commit(sbase + kTcMma2Done + 8u * buf);
      } else {
        *abort_flag = 1;
        tc_flag(p.status, RSM_STATUS_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
    if (!tc_wait_warp(sbase + kTcMma2Done + 8u * buf, par, abort_flag)) {
      tc_abort(p, abort_flag, lane);
      break;
    }
    rsm::tc_fence_after();
    // S_n = g_{n-1} S_0 + update, written over this thread's row of S_0 in the
    // slot (row v of key block kb at kb * 16 KiB + v * 128, chunk c at c ^ v % 8)
    const float gN = tab[kTcMaxT - 1];
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      float d[32];
      rsm::tmem_ld32(lane_base + 64u + buf * 128u + 32u * kb, d);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float4* q = reinterpret_cast<float4*>(sb + kb * kTcBoxBytes + v * 128 + (((c ^ v) & 7) << 4));
        const float4 s0 = *q;
        *q = make_float4(fmaf(gN, s0.x, d[4 * c]), fmaf(gN, s0.y, d[4 * c + 1]), fmaf(gN, s0.z, d[4 * c + 2]),
                         fmaf(gN, s0.w, d[4 * c + 3]));
      }
    }
    // both accumulators of this buffer go back to the builder
    rsm::tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcDFree + 8u * buf);
    // the new state, in the slot, goes back in place through the tensor map
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcStReady + 8u * buf);
    if (leader) {
      bool ok = mbar_wait(sbase + kTcStReady + 8u * buf, par, kWaitTimeoutNs) && !*abort_flag;
      if (ok) {
        const uint32_t sa = smem_addr(sb);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) tma_store_2d(&tp.tmap, 32 * kb, row0, sa + kb * kTcBoxBytes);
        bulk_commit();
      } else {
        *abort_flag = 1;
        tc_flag(p.status, RSM_STATUS_WAIT_TIMEOUT);
      }
      bulk_wait_read();  // the stores have read the slot: the loader may reuse it
      mbar_arrive(empty_bar);
    }
    __syncwarp();
    ++n_it;
  }
  if (leader) bulk_wait_all();
}

__global__ void __launch_bounds__(kTcThreads, 1) gdn_commit_tc_kernel(const __grid_constant__ TcParams tp) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Params& p = tp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  if (warp == 1) {
    rsm::tmem_alloc(sbase + kTcTmemSlot, kTcTmemCols);
    rsm::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (uint32_t q = 0; q < p.slots; ++q) {
      mbar_init(sbase + 8u * q, 1u);
      mbar_init(sbase + 8u * kMaxSlots + 8u * q, 1u);  // the epilogue's leader, after the store has read the slot
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(sbase + kTcMma1Done + 8u * b, 1u);
      mbar_init(sbase + kTcTabReady + 8u * b, 1u);
      mbar_init(sbase + kTcA2Ready + 8u * b, 4u);
      mbar_init(sbase + kTcMma2Done + 8u * b, 1u);
      mbar_init(sbase + kTcStReady + 8u * b, 4u);
      mbar_init(sbase + kTcDFree + 8u * b, 4u);
    }
    mbar_init(sbase + kTcExit, 5u);
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    rsm::fence_mbar_init();
  }
  rsm::tc_fence_before();
  __syncthreads();
  rsm::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTcTmemSlot);
  // the swizzled state boxes need 1024-byte alignment: a shared-memory base
  // without it (never seen) ends the CTA with a status bit
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) tc_flag(p.status, RSM_STATUS_WAIT_TIMEOUT);
    if (warp == 1) rsm::tmem_dealloc(tmem, kTcTmemCols);
    return;
  }
  if (warp == 0) {
    tc_run_loader(tp, smem, lane);
  } else {
    if (warp == 1)
      tc_run_builder(tp, smem, lane, tmem);
    else
      tc_run_epilogue(tp, smem, warp - 2, warp, lane, tmem);
    rsm::tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcExit);
    if (warp == 1) {
      (void)mbar_wait(sbase + kTcExit, 0u, 3ull * kWaitTimeoutNs);
      rsm::tc_fence_after();
      rsm::tmem_dealloc(tmem, kTcTmemCols);
    }
  }
}

}  // namespace gdn
