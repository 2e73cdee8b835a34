// gdn_kernel.cuh -- the persistent sm_103a kernel that commits accepted
// ReplaySSM prefixes into gated-delta-rule checkpoints
// (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit, API page:
// signature, Parameters, Notes).
//
// Per accepted token t of request b, every (layer, value head) checkpoint
// S [128 value rows x 128 key columns] (fp32, K-last) is updated in place:
//   k^ = k_t / sqrt(|k_t|^2 + 1e-6)     (use_qk_l2norm; else k^ = k_t)
//   S  = exp(g_t) S
//   S  = S + beta_t (v_t - S k^) k^T
// Every value row evolves on its own given k^, its v entry, g and beta, so the
// work item is a slab of 64 rows of one head (32 KiB): a row's dot product is
// a reduction over the 8 lanes that hold it (each lane holds two rows).  The normalisation is folded into
// two scalars per token (S k^ = r * S k, k^ k^T update = (u r) k), so k is
// used raw, and the decay into a running scale of the whole slab, so that each
// element costs two FMAs per token.
//
// One CTA = 1 loader warp + 8 consumer warps joined by pipeline slots (full /
// empty mbarrier pairs and descriptors) and a byte arena, as in the
// materialization kernel: the loader bulk-copies the slab, the request's
// accepted rows of k (one copy), the slab's part of the accepted v rows and
// the accepted g and beta values; the consumers apply the tokens in registers,
// write the track copy at the tracked step and the slab back in place.
// Every wait is bounded in wall time.
#pragma once
#include <cstdint>

#include "../../include/replayssm.h"
#include "gdn_params.h"
#include "rsm_ptx.cuh"

namespace gdn {

using rsm::arena_next;
using rsm::bulk_g2s;
using rsm::bulk_g2s_hint;
using rsm::cp_async_4;
using rsm::cp_async_mbar_arrive;
using rsm::fence_proxy_async_smem;
using rsm::l2_policy_evict_first;
using rsm::mbar_arrive;
using rsm::mbar_expect_tx;
using rsm::mbar_init;
using rsm::mbar_wait;
using rsm::smem_addr;

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bits) {
  if (status != nullptr && bits != 0u) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// loader warp
// ---------------------------------------------------------------------------
__device__ __forceinline__ void run_loader(const Params& p, unsigned char* smem, int lane) {
  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8u * kMaxSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  const uint64_t policy = l2_policy_evict_first();

  // units: (request b, layer l, a run of `chunk` value heads), request-major,
  // dealt to the CTAs round-robin; each unit's heads x slabs are its items
  const int64_t heads = static_cast<int64_t>(p.B) * p.L * p.HV;
  int chunk = static_cast<int>(min(static_cast<int64_t>(8), max(static_cast<int64_t>(1), heads / (16 * static_cast<int64_t>(gridDim.x)))));
  const int units_per_seg = (p.HV + chunk - 1) / chunk;
  const int64_t total_units = static_cast<int64_t>(p.B) * p.L * units_per_seg;
  const int per_kh = p.HV / p.H;

  uint32_t stage = 0, phase = 0, fills = 0;
  bool aborted = false;
  // arena bookkeeping: see the materialization kernel's loader
  const uint32_t item_max = item_layout(p.T).bytes;
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

  int cur_b = -1, s = 0, n = 0, ts = -1, step = -1;
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
      ts = -1;
      step = -1;
      uint32_t bad = 0;
      ok = s > p.null_id && n != 0;
      if (ok && (s >= p.SL || n < 0 || n > p.T)) {
        bad |= s >= p.SL ? RSM_STATUS_BAD_SLOT : RSM_STATUS_BAD_PREFIX_LEN;
        ok = false;
      }
      if (ok && p.track_indices != nullptr) {
        const int t = __ldg(p.track_indices + b);
        if (t > p.null_id) {
          if (t >= p.SL) {
            bad |= RSM_STATUS_BAD_SLOT;
          } else {
            const int st = __ldg(p.track_steps + b);
            if (st >= 0 && st < n) {
              ts = t;
              step = st;
            }
          }
        }
      }
      if (lane == 0) flag_status(p.status, bad);
    }
    if (!ok) continue;
    const Item it = item_layout(n);
    const int64_t lay_slot = static_cast<int64_t>(l) * p.SL + s;
    for (int hv = hv0; hv < hv_end && !aborted; ++hv) {
      const int hk = hv / per_kh;
      float* head_state = p.state + (lay_slot * p.HV + hv) * (kDV * kDK);
      float* head_track =
          ts >= 0 ? p.state + ((static_cast<int64_t>(l) * p.SL + ts) * p.HV + hv) * (kDV * kDK) : nullptr;
      const uint16_t* krows = p.rawk + (lay_slot * p.H + hk) * p.T * kDK;
      const uint16_t* vrows = p.rawv + (lay_slot * p.HV + hv) * p.T * kDV;
      const float* grow = p.g + (lay_slot * p.HV + hv) * p.T;
      const float* brow = p.beta + (lay_slot * p.HV + hv) * p.T;
      for (int r = 0; r < kSlabs; ++r) {
        uint32_t off = 0;
        if (!alloc(it.bytes, off)) {
          aborted = true;
          break;
        }
        unsigned char* sb = smem + kArenaOff + off;
        const uint32_t sba = smem_addr(sb);
        const uint32_t fullb = full0 + 8u * stage;
        Desc* desc = reinterpret_cast<Desc*>(smem + kDescOff) + stage;
        float* slab = head_state + r * kSlabRows * kDK;
        if (lane == 0) {
          const unsigned long long ga = reinterpret_cast<unsigned long long>(slab);
          const unsigned long long gt =
              head_track ? reinterpret_cast<unsigned long long>(head_track + r * kSlabRows * kDK) : 0ull;
          uint4* d4 = reinterpret_cast<uint4*>(desc);
          d4[0] = make_uint4(static_cast<uint32_t>(ga), static_cast<uint32_t>(ga >> 32), static_cast<uint32_t>(gt),
                             static_cast<uint32_t>(gt >> 32));
          d4[1] = make_uint4(static_cast<uint32_t>(n), static_cast<uint32_t>(step), 0u, 0u);
          fence_proxy_async_smem();
          mbar_expect_tx(fullb, kSlabBytes + static_cast<uint32_t>(n) * (kDK * 2u + kSlabRows * 2u));
        }
        __syncwarp();
        if (lane == 0) {
          bulk_g2s_hint(sba, slab, kSlabBytes, fullb, policy);
          bulk_g2s(sba + it.off_k, krows, static_cast<uint32_t>(n) * kDK * 2u, fullb);
        }
        for (int t = lane; t < n; t += 32) {
          bulk_g2s(sba + it.off_v + static_cast<uint32_t>(t) * kSlabRows * 2u,
                   vrows + static_cast<int64_t>(t) * kDV + r * kSlabRows, kSlabRows * 2u, fullb);
          cp_async_4(sba + it.off_g + 4u * t, grow + t);
          cp_async_4(sba + it.off_beta + 4u * t, brow + t);
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
  }

  bool ended = false;
  if (!aborted) {
    bool fine = true;
    while (fine && n_out >= p.slots) fine = free_oldest();
    if (fine) {
      if (lane == 0) (reinterpret_cast<Desc*>(smem + kDescOff) + stage)->flags = kFlagEnd;
      __syncwarp();
      if (lane == 0) mbar_arrive(full0 + 8u * stage);
      ended = true;
    }
  }
  if (!ended) {
    if (lane == 0) {
      *abort_flag = 1;
      flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
    }
    for (uint32_t q = 0; q < p.slots; ++q) {
      if (q < stage)
        (void)mbar_wait(full0 + 8u * q, phase, 1000000ull);
      else if (fills >= p.slots)
        (void)mbar_wait(full0 + 8u * q, phase ^ 1u, 1000000ull);
    }
  }
}

// ---------------------------------------------------------------------------
// consumer warps: lane (lr = lane / 8, column group lc = lane % 8) holds
// S[row][q*32 + lc*4 + e], q, e = 0..3, for its two rows cw*8 + lr and
// cw*8 + lr + 4 (each key value it loads serves both)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void run_consumer(const Params& p, unsigned char* smem, int cw, int lane) {
  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8u * kMaxSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  const int lr = lane >> 3, lc = lane & 7;
  const int rowa = cw * 8 + lr, rowb = rowa + 4;  // this lane's rows inside the slab
  const uint32_t item_max = item_layout(p.T).bytes;
  const bool l2norm = p.l2norm != 0;
  uint32_t arena_head = 0;
  uint32_t stage = 0, phase = 0;
  for (;;) {
    if (!mbar_wait(full0 + 8u * stage, phase, kWaitTimeoutNs) || *abort_flag) {
      if (lane == 0) {
        *abort_flag = 1;
        flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
      }
      break;
    }
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    const unsigned char* sb = smem + kArenaOff + off;
    const Desc* desc = reinterpret_cast<const Desc*>(smem + kDescOff) + stage;
    if (desc->flags & kFlagEnd) break;
    const int n = desc->n;
    const int step = desc->step;
    float* slab = reinterpret_cast<float*>(desc->slab);
    float* track = reinterpret_cast<float*>(desc->track);
    const Item it = item_layout(n);
    arena_head = off + it.bytes;

    // per-token scalars, once per item and warp, four lanes per token:
    // exp(g), beta, r = 1/sqrt(|k|^2 + 1e-6) (1 without normalisation), exp(-g)
    float4* tok = reinterpret_cast<float4*>(smem + kTokOff + cw * kTokBytes);
    for (int t0 = 0; t0 < n; t0 += 8) {
      const int t = t0 + (lane >> 2), part = lane & 3;
      float ss = 0.0f;
      if (t < n && l2norm) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // columns (q*4 + part)*8 .. +7
          const uint4 w = *reinterpret_cast<const uint4*>(sb + it.off_k + t * kDK * 2 + (q * 4 + part) * 16);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16lo(ws[e]), hi = bf16hi(ws[e]);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
      }
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
      if (t < n && part == 0) {
        const float g = reinterpret_cast<const float*>(sb + it.off_g)[t];
        tok[t] = make_float4(expf(g), reinterpret_cast<const float*>(sb + it.off_beta)[t],
                             l2norm ? rsqrtf(ss + 1e-6f) : 1.0f, expf(-g));
      }
    }
    __syncwarp();

    // The decay is kept as a scale: the state is c * S.  Per token, with
    // ca = c * exp(g): S k^ after the decay is ca * r * (S k), and the update
    // (u r) k adds (u r / ca) k to S.  Rescaling is exact up to rounding
    // (it scales every term alike); S is renormalised before c gets small.
    // this lane's state values as packed pairs: Sa/Sb[2q], [2q+1] = columns
    // q*32 + lc*4 + {0,1}, {2,3} of rows rowa / rowb
    float2 Sa[8], Sb[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 va = *reinterpret_cast<const float4*>(sb + (rowa * kDK + q * 32 + lc * 4) * 4);
      const float4 vb = *reinterpret_cast<const float4*>(sb + (rowb * kDK + q * 32 + lc * 4) * 4);
      Sa[2 * q] = make_float2(va.x, va.y);
      Sa[2 * q + 1] = make_float2(va.z, va.w);
      Sb[2 * q] = make_float2(vb.x, vb.y);
      Sb[2 * q + 1] = make_float2(vb.z, vb.w);
    }
    float c = 1.0f, inv_c = 1.0f;
    const uint16_t* vcol = reinterpret_cast<const uint16_t*>(sb + it.off_v);
    for (int t = 0; t < n; ++t) {
      const float4 tp = tok[t];
      float2 k2[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint2 w = *reinterpret_cast<const uint2*>(sb + it.off_k + (t * kDK + q * 32 + lc * 4) * 2);
        k2[2 * q] = make_float2(bf16lo(w.x), bf16hi(w.x));
        k2[2 * q + 1] = make_float2(bf16lo(w.y), bf16hi(w.y));
      }
      float2 da = __fmul2_rn(Sa[0], k2[0]), db = __fmul2_rn(Sb[0], k2[0]);
#pragma unroll
      for (int e = 1; e < 8; ++e) {
        da = __ffma2_rn(Sa[e], k2[e], da);
        db = __ffma2_rn(Sb[e], k2[e], db);
      }
      float dota = da.x + da.y, dotb = db.x + db.y;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        dota += __shfl_xor_sync(0xFFFFFFFFu, dota, o);
        dotb += __shfl_xor_sync(0xFFFFFFFFu, dotb, o);
      }
      const float v_a = __uint_as_float(static_cast<uint32_t>(vcol[t * kSlabRows + rowa]) << 16);
      const float v_b = __uint_as_float(static_cast<uint32_t>(vcol[t * kSlabRows + rowb]) << 16);
      const float ca = c * tp.x, inv_ca = inv_c * tp.w;
      const float rs = tp.z * inv_ca;
      const float wa = tp.y * (v_a - ca * (tp.z * dota)) * rs;
      const float wb = tp.y * (v_b - ca * (tp.z * dotb)) * rs;
      const float2 wa2 = make_float2(wa, wa), wb2 = make_float2(wb, wb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        Sa[e] = __ffma2_rn(wa2, k2[e], Sa[e]);
        Sb[e] = __ffma2_rn(wb2, k2[e], Sb[e]);
      }
      c = ca;
      inv_c = inv_ca;
      if (c < 0x1p-30f) {  // the same in every lane of the item
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          Sa[e] = __fmul2_rn(Sa[e], c2);
          Sb[e] = __fmul2_rn(Sb[e], c2);
        }
        c = 1.0f;
        inv_c = 1.0f;
      }
      if (track != nullptr && t == step) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __stcs(reinterpret_cast<float4*>(track + rowa * kDK + q * 32 + lc * 4),
                 make_float4(c * Sa[2 * q].x, c * Sa[2 * q].y, c * Sa[2 * q + 1].x, c * Sa[2 * q + 1].y));
          __stcs(reinterpret_cast<float4*>(track + rowb * kDK + q * 32 + lc * 4),
                 make_float4(c * Sb[2 * q].x, c * Sb[2 * q].y, c * Sb[2 * q + 1].x, c * Sb[2 * q + 1].y));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * stage);  // nothing more is read from the slot
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __stcs(reinterpret_cast<float4*>(slab + rowa * kDK + q * 32 + lc * 4),
             make_float4(c * Sa[2 * q].x, c * Sa[2 * q].y, c * Sa[2 * q + 1].x, c * Sa[2 * q + 1].y));
      __stcs(reinterpret_cast<float4*>(slab + rowb * kDK + q * 32 + lc * 4),
             make_float4(c * Sb[2 * q].x, c * Sb[2 * q].y, c * Sb[2 * q + 1].x, c * Sb[2 * q + 1].y));
    }
    if (++stage == p.slots) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) gdn_commit_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const uint32_t full0 = smem_addr(smem);
    for (uint32_t q = 0; q < p.slots; ++q) {
      mbar_init(full0 + 8u * q, 1u);
      mbar_init(full0 + 8u * kMaxSlots + 8u * q, kConsumerWarps);
    }
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    rsm::fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0)
    run_loader(p, smem, lane);
  else
    run_consumer(p, smem, warp - 1, lane);
}

}  // namespace gdn
