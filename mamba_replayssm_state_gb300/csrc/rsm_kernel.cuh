// rsm_kernel.cuh -- the persistent sm_103a kernel for ReplaySSM prefix
// materialization (flashinfer.mamba.replayssm_materialize, API page; the
// persistent work-queue design of FlashInfer PR #4815, Description).
//
// Work item = (active request i, layer l, head h): one [dim, dstate] state tile.
// Items are numbered request-major -> layer -> head; runs of up to 32 heads of
// one (request, layer) form units dealt to the CTAs round-robin, so that every
// CTA gets a mix of requests (and of replay lengths) while the items of a unit
// share their metadata and stream through contiguous state memory.
//
// One CTA = 1 loader warp + 8 consumer warps, joined by S pipeline slots (a
// full/empty mbarrier pair and a descriptor each) and a byte arena in shared
// memory that holds the slots' data, each item taking only the bytes of its
// own replay length:
//   loader   : finds n (the first -1 of the active list), resolves the slot
//              and pointer tables once per (request, layer), and per item
//              issues bulk asynchronous copies (cp.async.bulk) of the source
//              state tile (+ its scales), the k ring rows of x and of B, and
//              4-byte cp.async copies of the k dt values and of A[h], all
//              completing on the stage's "full" mbarrier.  Pads, out-of-range
//              metadata and misaligned addresses are handled here.
//   consumers: wait for "full", compute the decay of every token once per
//              warp (exp(dt*A) with a shuffle suffix-product scan), apply the
//              whole prefix to the tile in registers, requantize, store with
//              16-byte streaming stores, and release the slot ("empty").
// Every state element is read once and written once; the ring is only read.
// Every wait is bounded in wall time (a logic error ends the kernel with a
// status bit instead of hanging).
//
// The prefix is applied in closed form, which is the sequential recurrence
// S <- a_t*S + dt_t x_t B_t^T unrolled exactly:
//   S_k = P * S_0 + sum_t w_t x_t B_t^T,  P = prod_t a_t,  w_t = dt_t prod_{s>t} a_s,
// costing one FFMA per element per token (plus one FMUL per element).
#pragma once
#include <cfloat>
#include <cstdint>

#include "rsm_formats.cuh"
#include "rsm_params.h"
#include "rsm_ptx.cuh"

namespace rsm {

struct alignas(16) ItemDesc {
  unsigned long long dst_state;  // global address of the destination head tile
  unsigned long long dst_scale;  // global address of the destination head's scales
  int32_t k;                     // ring entries to apply; 0 = exact copy
  uint32_t flags;
  int32_t layer;
  int32_t dst_slot;
  int32_t head;                  // the item's (first) head
  float A[2];                    // A of the item's heads; landed by cp.async
  uint32_t unused;
};
static_assert(sizeof(ItemDesc) == kDescBytes, "descriptor size");
constexpr uint32_t kFlagEnd = 1u, kFlagDstAligned = 2u, kFlagScaleAligned = 4u;
// An item whose head continues the previous item's B group (same request and
// layer): its B rows are not copied.  The tensor-core kernel reuses the MMA
// operand it built from the previous item's; the one-byte kernel (prefixes of
// at most kTokChunk tokens) its warps' fp32 copies of them.
constexpr uint32_t kFlagSameB = 8u;

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bits) {
  if (status != nullptr && bits != 0u) atomicOr(status, bits);
}

// Warp-cooperative byte copy global -> shared for the rare misaligned item.
__device__ __forceinline__ void copy_bytes_warp(unsigned char* dst, const unsigned char* src, uint32_t n,
                                                int lane) {
  for (uint32_t o = lane; o < n; o += 32) dst[o] = src[o];
}

template <int IF>
struct In {
  static constexpr int bytes = IF == RSM_F32 ? 4 : 2;
};

// CNT consecutive input elements (bf16 or fp32) from shared memory -> fp32.
template <int IF, int CNT>
__device__ __forceinline__ void load_inputs(const unsigned char* p, float* out) {
  constexpr int bytes = CNT * In<IF>::bytes;
  if constexpr (IF == RSM_F32) {
    if constexpr (bytes % 16 == 0) {
#pragma unroll
      for (int q = 0; q < CNT / 4; ++q) {
        const float4 v = reinterpret_cast<const float4*>(p)[q];
        out[4 * q] = v.x;
        out[4 * q + 1] = v.y;
        out[4 * q + 2] = v.z;
        out[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < CNT; ++q) out[q] = reinterpret_cast<const float*>(p)[q];
    }
  } else {  // bf16
    if constexpr (bytes % 16 == 0) {
#pragma unroll
      for (int q = 0; q < CNT / 8; ++q) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          out[8 * q + 2 * e] = bf16lo(w[e]);
          out[8 * q + 2 * e + 1] = bf16hi(w[e]);
        }
      }
    } else if constexpr (bytes == 8) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      out[0] = bf16lo(v.x);
      out[1] = bf16hi(v.x);
      out[2] = bf16lo(v.y);
      out[3] = bf16hi(v.y);
    } else if constexpr (bytes == 4) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      out[0] = bf16lo(v);
      out[1] = bf16hi(v);
    } else {
#pragma unroll
      for (int q = 0; q < CNT; ++q)
        out[q] = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[q]) << 16);
    }
  }
}

// ---------------------------------------------------------------------------
// loader warp
// ---------------------------------------------------------------------------
// kChunked: long prefixes' ring rows as 16-byte cp.async chunks (the
// tensor-core kernel, whose windows reach 64 tokens); otherwise every ring row
// is one bulk copy, which keeps the other kernels' loader small.
// HPI: heads per item (1, or 2 for the one-byte tensor-core kernel, whose
// items are two consecutive heads of one B group: their tiles, scales and x
// rows are adjacent in memory, so they move as one tile of 2D rows; dt and A
// take one value per head).  Requires heads_per_group % HPI == 0.
template <int SF, int IF, int D, int N, bool kChunked = false, int HPI = 1, bool kExactFit = false>
__device__ __forceinline__ void run_loader(const Params& p, unsigned char* smem, int lane) {
  constexpr int ES = Fmt<SF>::bytes;
  constexpr int IE = In<IF>::bytes;
  constexpr bool Q = Fmt<SF>::quant;
  constexpr int DI = HPI * D;  // tile rows of one item
  constexpr uint32_t kTileBytes = DI * N * ES;
  static_assert(HPI == 1 || HPI == 2, "one or two heads per item");
  static_assert(kTileBytes % 16 == 0 && (DI * IE) % 16 == 0 && (N * IE) % 16 == 0, "bulk copy sizes");

  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  constexpr int XC = DI * IE / 16, BC = N * IE / 16;  // 16-byte chunks per item x row and per B row
  static_assert(kChunkedRingMinK <= 32, "ring rows by bulk copies: one token per lane");
  static_assert(XC >= 1 && XC <= 32 && 32 % XC == 0 && BC >= 1 && BC <= 32 && 32 % BC == 0, "ring row chunks");

  // n = position of the first -1 (entries after it are ignored)
  int n = p.Bt;
  for (int base = 0; base < p.Bt; base += 256) {
    int v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int idx = base + 32 * q + lane;
      v[q] = idx < p.Bt ? __ldg(p.active + idx) : 0;
    }
    int pos = -1;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, v[q] == -1 && base + 32 * q + lane < p.Bt);
      if (pos < 0 && m != 0u) pos = base + 32 * q + __ffs(m) - 1;
    }
    if (pos >= 0) {
      n = pos;
      break;
    }
  }

  // Work units: (request i, layer l, a run of `chunk` consecutive heads), in
  // request -> layer -> head order, dealt to the CTAs round-robin.  Each CTA
  // thus sees every part of the batch (replay lengths differ per request, so
  // contiguous ranges would leave the CTAs of long-prefix requests last),
  // while a unit still shares one metadata lookup and a run of B rows.
  // Smaller batches get shorter runs so that every CTA still has ~16 units.
  // (heads counted in items of HPI heads)
  const int HI = p.H / HPI, hpg_i = p.hpg / HPI;
  const int64_t total = static_cast<int64_t>(n) * p.L * HI;
  int chunk = static_cast<int>(min(static_cast<int64_t>(32),
                                   max(static_cast<int64_t>(4), total / (16 * static_cast<int64_t>(gridDim.x)))));
  if (chunk > HI) chunk = HI;
  const int units_per_seg = (HI + chunk - 1) / chunk;
  const int64_t total_units = static_cast<int64_t>(n) * p.L * units_per_seg;
  const int G = p.H / p.hpg;
  const uint64_t policy = l2_policy_evict_first();

  uint32_t stage = 0, phase = 0, fills = 0;
  bool aborted = false;

  // Arena bookkeeping (warp-uniform).  The n_out items not yet released by
  // the consumers sit in the n_out slots before `stage` and occupy
  // [tail, head) of the arena, or [tail, wrap point) + [0, head) once
  // allocation has wrapped.  Releases complete in slot order (every consumer
  // warp takes the items in order), so freeing is first in, first out.
  // Placement depends on the item sizes alone (arena_next), so the consumers
  // follow it without reading it from the descriptor: an item goes at the
  // head if the bytes from there to the arena's end hold item_max (or, with
  // kExactFit, the item itself), else at offset 0.
  const uint32_t item_max = item_layout(DI, N, ES, Q, IE, p.W, true, HPI).bytes;
  uint32_t head = 0, tail = 0, n_out = 0;
  bool wrapped = false;
  uint32_t slot_start = 0;  // lane s: arena offset of the item in slot s
  uint32_t oldest = 0, oldest_phase = 0;  // slot of the oldest outstanding item and its lap parity

  // waits until the consumers released the oldest outstanding item, frees it
  auto free_oldest = [&]() -> bool {
    if (!mbar_wait(empty0 + 8u * oldest, oldest_phase, kWaitTimeoutNs)) return false;
    if (++oldest == p.stages) {
      oldest = 0;
      oldest_phase ^= 1u;
    }
    --n_out;
    const uint32_t next = __shfl_sync(0xFFFFFFFFu, slot_start, static_cast<int>(oldest));
    if (n_out == 0) {
      tail = head;
      wrapped = false;
    } else {
      if (next < tail) wrapped = false;  // the oldest item is now past the wrap point
      tail = next;
    }
    return true;
  };
  // the item's place, then a free slot and free bytes [off, off + bytes) there
  auto alloc = [&](uint32_t bytes, uint32_t& off) -> bool {
    off = arena_next(head, kExactFit ? bytes : item_max, p.arena_bytes);
    for (;;) {
      if (n_out == 0) break;
      if (n_out < p.stages) {
        if (off == head) {
          if (!wrapped || head + bytes <= tail) break;  // [head, arena end) holds item_max
        } else if (!wrapped && bytes <= tail) {
          break;  // wrapping to 0: [0, tail) is free
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
  int cur_i = -1, b = 0;
  for (int64_t u = blockIdx.x; u < total_units && !aborted; u += gridDim.x) {
    const int64_t seg = u / units_per_seg;
    const int i = static_cast<int>(seg / p.L);
    const int l = static_cast<int>(seg - static_cast<int64_t>(i) * p.L);
    int h = static_cast<int>(u - seg * units_per_seg) * chunk;  // item index: heads h*HPI .. h*HPI+HPI-1
    const int h_end = min(HI, h + chunk);

    // per-layer table entries, one per lane, fetched together
    int64_t tab = 0;
    {
      const int64_t* t = nullptr;
      switch (lane) {
        case 0: t = p.state_ptrs; break;
        case 1: t = p.state_strides; break;
        case 2: t = p.x_ptrs; break;
        case 3: t = p.x_strides; break;
        case 4: t = p.B_ptrs; break;
        case 5: t = p.B_strides; break;
        case 6: t = p.dt_ptrs; break;
        case 7: t = p.dt_strides; break;
        case 8: t = p.A_ptrs; break;
        case 9: t = Q ? p.scale_ptrs : nullptr; break;
        case 10: t = Q ? p.scale_strides : nullptr; break;
        default: break;
      }
      if (t != nullptr) tab = __ldg(t + l);
    }
    if (i != cur_i) {
      b = __ldg(p.active + i);
      cur_i = i;
    }
    uint32_t bad = 0;
    bool ok = true;
    int src = p.pad, dst = p.pad, k = 0, rs = 0;
    if (b < 0 || b >= p.Bt) {
      bad |= RSM_STATUS_BAD_ACTIVE_INDEX;
      ok = false;
    } else {
      src = __ldg(p.src_slots + static_cast<int64_t>(l) * p.Bt + b);
      dst = __ldg(p.dst_slots + static_cast<int64_t>(l) * p.Bt + b);
      k = __ldg(p.prefix_len + b);
      rs = __ldg(p.ring_start + b);
      if (k < 0 || k > p.W) {
        bad |= RSM_STATUS_BAD_PREFIX_LEN;
        ok = false;
      }
      if (rs < 0 || rs >= p.R) {
        bad |= RSM_STATUS_BAD_RING_START;
        ok = false;
      }
      if (src == p.pad || dst == p.pad) {
        ok = false;
      } else if (src < 0 || dst < 0 || (p.num_slots > 0 && (src >= p.num_slots || dst >= p.num_slots))) {
        bad |= RSM_STATUS_BAD_SLOT;
        ok = false;
      }
    }
    if (lane == 0) flag_status(p.status, bad);
    if (!ok) continue;
    const unsigned char* state_base = reinterpret_cast<const unsigned char*>(__shfl_sync(0xFFFFFFFFu, tab, 0));
    const int64_t state_stride = __shfl_sync(0xFFFFFFFFu, tab, 1);
    const unsigned char* x_base = reinterpret_cast<const unsigned char*>(__shfl_sync(0xFFFFFFFFu, tab, 2));
    const int64_t x_stride = __shfl_sync(0xFFFFFFFFu, tab, 3);
    const unsigned char* B_base = reinterpret_cast<const unsigned char*>(__shfl_sync(0xFFFFFFFFu, tab, 4));
    const int64_t B_stride = __shfl_sync(0xFFFFFFFFu, tab, 5);
    const float* dt_base = reinterpret_cast<const float*>(__shfl_sync(0xFFFFFFFFu, tab, 6));
    const int64_t dt_stride = __shfl_sync(0xFFFFFFFFu, tab, 7);
    const float* A_base = reinterpret_cast<const float*>(__shfl_sync(0xFFFFFFFFu, tab, 8));
    float* scale_base = reinterpret_cast<float*>(__shfl_sync(0xFFFFFFFFu, tab, 9));
    const int64_t scale_stride = __shfl_sync(0xFFFFFFFFu, tab, 10);

    const unsigned char* src_slot = state_base + static_cast<int64_t>(src) * state_stride * ES;
    unsigned char* dst_slot = const_cast<unsigned char*>(state_base) + static_cast<int64_t>(dst) * state_stride * ES;
    const unsigned char* x_slot = x_base + static_cast<int64_t>(src) * x_stride * IE;
    const unsigned char* B_slot = B_base + static_cast<int64_t>(src) * B_stride * IE;
    const float* dt_slot = dt_base + static_cast<int64_t>(src) * dt_stride;
    const float* src_sc_slot = nullptr;
    float* dst_sc_slot = nullptr;
    if constexpr (Q) {
      src_sc_slot = scale_base + static_cast<int64_t>(src) * scale_stride;
      dst_sc_slot = scale_base + static_cast<int64_t>(dst) * scale_stride;
    }
    // Every tile, row and scale block of the segment starts a whole number of
    // 16-byte units after its slot base (D*N*ES, D*IE, N*IE and D*4 are
    // multiples of 16), so alignment is a property of the segment.
    static_assert((D * IE) % 16 == 0 && (N * IE) % 16 == 0 && (D * 4) % 16 == 0, "row granularity");
    const bool seg_aligned =
        ((reinterpret_cast<uintptr_t>(src_slot) | reinterpret_cast<uintptr_t>(x_slot) |
          reinterpret_cast<uintptr_t>(B_slot) | reinterpret_cast<uintptr_t>(src_sc_slot)) & 15u) == 0u &&
        ((reinterpret_cast<uintptr_t>(dt_slot) | reinterpret_cast<uintptr_t>(A_base)) & 3u) == 0u;
    const uint32_t dst_flags = ((reinterpret_cast<uintptr_t>(dst_slot) & 15u) == 0u ? kFlagDstAligned : 0u) |
                               ((reinterpret_cast<uintptr_t>(dst_sc_slot) & 3u) == 0u ? kFlagScaleAligned : 0u);

    // this lane's ring rows for the whole segment: tokens t = lane and lane + 32
    // (row p_t = (ring_start + t) mod R, the same for every head of the segment)
    int ring_row[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int t = lane + 32 * q;
      ring_row[q] = t < k ? (rs + t) % p.R : 0;
    }
    int g = h * HPI / p.hpg;                         // B group of item h, advanced incrementally
    int g_left = hpg_i - (h - g * hpg_i);            // items left in group g, h included
    const uint4 desc_tail = make_uint4(static_cast<uint32_t>(k), dst_flags, static_cast<uint32_t>(l),
                                       static_cast<uint32_t>(dst));
    const ItemLayout il_full = item_layout(DI, N, ES, Q, IE, k, true, HPI);
    const ItemLayout il_noB = item_layout(DI, N, ES, Q, IE, k, false, HPI);
    const bool tc_items = p.tc_min_k > 0 && k >= p.tc_min_k;  // the tensor-core kernel's MMA path
    const int unit_h0 = h;

    for (; h < h_end; ++h) {
      // B rows reused from the previous item (same unit, same group): the
      // tensor-core kernel keeps the operand it built; the one-byte kernel
      // keeps its fp32 B rows when the whole prefix fits one token chunk
      const bool b_reuse = tc_items || (Q && k > 0 && k <= kTokChunk);
      const bool same_B = b_reuse && h != unit_h0 && g_left != hpg_i;
      const ItemLayout il = same_B ? il_noB : il_full;
      uint32_t off = 0;
      if (!alloc(il.bytes, off)) {
        aborted = true;
        break;
      }
      unsigned char* sb = smem + p.arena0 + off;
      const uint32_t sba = smem_addr(sb);
      const uint32_t fullb = full0 + 8u * stage;
      ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + p.desc0) + stage;
      const uint32_t desca = smem_addr(desc);

      const int64_t tile_off = static_cast<int64_t>(h) * DI * N * ES;
      const unsigned char* src_tile = src_slot + tile_off;
      unsigned char* dst_tile = dst_slot + tile_off;
      const float* src_sc = nullptr;
      float* dst_sc = nullptr;
      if constexpr (Q) {
        src_sc = src_sc_slot + static_cast<int64_t>(h) * DI;
        dst_sc = dst_sc_slot + static_cast<int64_t>(h) * DI;
      }
      const float* A_ptr = A_base + h * HPI;
      const bool aligned = seg_aligned;

      if (lane == 0) {
        uint4* d4 = reinterpret_cast<uint4*>(desc);
        const unsigned long long ds = reinterpret_cast<unsigned long long>(dst_tile);
        const unsigned long long dc = reinterpret_cast<unsigned long long>(dst_sc);
        d4[0] = make_uint4(static_cast<uint32_t>(ds), static_cast<uint32_t>(ds >> 32), static_cast<uint32_t>(dc),
                           static_cast<uint32_t>(dc >> 32));
        d4[1] = make_uint4(desc_tail.x, desc_tail.y | (same_B ? kFlagSameB : 0u), desc_tail.z,
                           desc_tail.w);  // k, flags, layer, dst_slot
        desc->head = h * HPI;
      }
      if (aligned) {
        const bool row_copies = !kChunked || k < kChunkedRingMinK;  // ring rows by bulk copies (see below)
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_expect_tx(fullb, kTileBytes + (Q ? DI * 4u : 0u) +
                                    (row_copies ? static_cast<uint32_t>(k) * (DI + (same_B ? 0 : N)) * IE : 0u));
        }
        __syncwarp();
        if (lane == 0) {
          bulk_g2s_hint(sba, src_tile, kTileBytes, fullb, policy);
          if constexpr (Q) bulk_g2s(sba + il.off_scale, src_sc, DI * 4u, fullb);
          if (k > 0) {
#pragma unroll
            for (int j = 0; j < HPI; ++j)
              cp_async_4(desca + static_cast<uint32_t>(offsetof(ItemDesc, A) + 4 * j), A_ptr + j);
          }
        }
        // Ring rows: up to kChunkedRingMinK tokens, one bulk copy per row by
        // the lanes in parallel.  Longer prefixes as 16-byte cp.async chunks
        // spread over the lanes, through the load/store units: one small bulk
        // copy per row queues behind the tile copies on the bulk-copy engine
        // (measured 15% slower at 64 tokens, while at 16 tokens and less the
        // chunks cost the loader more than they save).  Lane l copies chunk
        // l % XC of tokens l / XC, then every 32 / XC tokens further; the
        // chunk's ring row follows modulo R.
        if (row_copies) {
#pragma unroll
          for (int q = 0; q < (kChunked ? 1 : 2); ++q) {
            const int t = lane + 32 * q;
            if (t < k) {
              const int64_t xr = static_cast<int64_t>(ring_row[q]) * p.H + h * HPI;
              bulk_g2s(sba + il.off_x + static_cast<uint32_t>(t) * DI * IE, x_slot + xr * (D * IE), DI * IE, fullb);
              if (!same_B)
                bulk_g2s(sba + il.off_B + static_cast<uint32_t>(t) * N * IE,
                         B_slot + (static_cast<int64_t>(ring_row[q]) * G + g) * (N * IE), N * IE, fullb);
            }
          }
        } else if constexpr (kChunked) {
          const int x_t0 = lane / XC, x_part = lane % XC;
          int pr = rs + x_t0 - (rs + x_t0 >= p.R ? p.R : 0);
          while (pr >= p.R) pr -= p.R;
          const int64_t row_bytes = static_cast<int64_t>(p.H) * (D * IE);
          const unsigned char* xp = x_slot + static_cast<int64_t>(h) * (DI * IE) + 16 * x_part;
          const unsigned char* xq = xp + static_cast<int64_t>(pr) * row_bytes;
          const unsigned char* x_end = xp + static_cast<int64_t>(p.R) * row_bytes;
          const int64_t step = (32 / XC) * row_bytes, wrap = static_cast<int64_t>(p.R) * row_bytes;
          uint32_t sdst = sba + il.off_x + static_cast<uint32_t>(x_t0 * DI * IE + 16 * x_part);
          for (int t = x_t0; t < k; t += 32 / XC) {
            cp_async_16(sdst, xq);
            sdst += (32 / XC) * DI * IE;
            xq += step;
            while (xq >= x_end) xq -= wrap;  // rings shorter than the step wrap more than once
          }
          if (!same_B) {
            const int b_t0 = lane / BC, b_part = lane % BC;
            int pb = rs + b_t0 - (rs + b_t0 >= p.R ? p.R : 0);
            while (pb >= p.R) pb -= p.R;
            for (int t = b_t0; t < k; t += 32 / BC) {
              cp_async_16(sba + il.off_B + static_cast<uint32_t>(t * N * IE + 16 * b_part),
                          B_slot + (static_cast<int64_t>(pb) * G + g) * (N * IE) + 16 * b_part);
              pb += 32 / BC;
              while (pb >= p.R) pb -= p.R;
            }
          }
        }
        // dt of this lane's tokens t = lane and t = lane + 32 (head j's k values
        // at off_dt + 4 j k)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int t = lane + 32 * q;
          if (t < k) {
#pragma unroll
            for (int j = 0; j < HPI; ++j)
              cp_async_4(sba + il.off_dt + 4u * (j * k + t),
                         dt_slot + static_cast<int64_t>(ring_row[q]) * p.H + h * HPI + j);
          }
        }
        cp_async_mbar_arrive(fullb);
      } else {
        // any alignment: plain byte copies by the whole warp
        copy_bytes_warp(sb, src_tile, kTileBytes, lane);
        if constexpr (Q)
          copy_bytes_warp(sb + il.off_scale, reinterpret_cast<const unsigned char*>(src_sc), DI * 4u, lane);
        for (int t = 0; t < k; ++t) {
          const int pr = (rs + t) % p.R;
          copy_bytes_warp(sb + il.off_x + t * DI * IE,
                          x_slot + (static_cast<int64_t>(pr) * p.H + h * HPI) * D * IE, DI * IE, lane);
          if (!same_B)
            copy_bytes_warp(sb + il.off_B + t * N * IE, B_slot + (static_cast<int64_t>(pr) * G + g) * N * IE,
                            N * IE, lane);
          for (int j = 0; j < HPI; ++j)
            copy_bytes_warp(sb + il.off_dt + 4 * (j * k + t),
                            reinterpret_cast<const unsigned char*>(dt_slot + static_cast<int64_t>(pr) * p.H + h * HPI + j),
                            4, lane);
        }
        if (k > 0)
          copy_bytes_warp(reinterpret_cast<unsigned char*>(desc) + offsetof(ItemDesc, A),
                          reinterpret_cast<const unsigned char*>(A_ptr), 4 * HPI, lane);
        __threadfence_block();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(fullb);
      if (--g_left == 0) {
        ++g;
        g_left = hpg_i;
      }
      // the item now occupies [off, off + il.bytes) of the arena, in slot `stage`
      if (lane == static_cast<int>(stage)) slot_start = off;
      head = off + il.bytes;
      ++n_out;
      ++fills;
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }

  // end marker for the consumers, in the next slot once it is free
  bool ended = false;
  if (!aborted) {
    bool ok = true;
    while (ok && n_out >= p.stages) ok = free_oldest();
    if (ok) {
      if (lane == 0) (reinterpret_cast<ItemDesc*>(smem + p.desc0) + stage)->flags = kFlagEnd;
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
    // let copies already issued into the arena land before the CTA exits: the
    // last fill of slot s completed the full-barrier phase of parity `phase`
    // (s < stage) or `phase ^ 1` (s >= stage, if the slots went round once)
    for (uint32_t s = 0; s < p.stages; ++s) {
      if (s < stage)
        (void)mbar_wait(full0 + 8u * s, phase, 1000000ull);
      else if (fills >= p.stages)
        (void)mbar_wait(full0 + 8u * s, phase ^ 1u, 1000000ull);
    }
  }
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
// Decay of a prefix of k <= 64 tokens, once per warp: a_t = exp(dt_t*A),
// w_t = dt_t * prod_{s>t} a_s into wbuf, and P = prod_t a_t returned (the same
// in every lane).  Suffix products by shuffles over 32-token chunks; the two
// chunks of a longer prefix are scanned side by side, the first one's weights
// then scaled by the second one's product.
__device__ __forceinline__ float decay_scan(const float* dts, float A, int k, int lane, float* wbuf) {
  const float dt0 = lane < k ? dts[lane] : 0.0f;
  float i0 = lane < k ? expf(dt0 * A) : 1.0f;
  if (k <= 32) {
    // after the level with offset `off` lane t holds the product over
    // [t, t + 2*off); levels past the prefix would only multiply by the 1.0
    // of lanes >= k, so they are skipped (k is warp-uniform)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      if (off >= k) break;
      const float v0 = __shfl_down_sync(0xFFFFFFFFu, i0, off);
      if (lane + off < 32) i0 *= v0;
    }
    float e0 = __shfl_down_sync(0xFFFFFFFFu, i0, 1);
    if (lane == 31) e0 = 1.0f;
    if (lane < k) wbuf[lane] = dt0 * e0;
    return __shfl_sync(0xFFFFFFFFu, i0, 0);
  }
  const int t1 = 32 + lane;
  const float dt1 = t1 < k ? dts[t1] : 0.0f;
  float i1 = t1 < k ? expf(dt1 * A) : 1.0f;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float v0 = __shfl_down_sync(0xFFFFFFFFu, i0, off);
    const float v1 = __shfl_down_sync(0xFFFFFFFFu, i1, off);
    if (lane + off < 32) {
      i0 *= v0;
      i1 *= v1;
    }
  }
  float e0 = __shfl_down_sync(0xFFFFFFFFu, i0, 1);
  float e1 = __shfl_down_sync(0xFFFFFFFFu, i1, 1);
  if (lane == 31) e0 = e1 = 1.0f;
  const float p1 = __shfl_sync(0xFFFFFFFFu, i1, 0);  // product of the second chunk
  if (t1 < k) wbuf[t1] = dt1 * e1;
  if (lane < k) wbuf[lane] = dt0 * (e0 * p1);
  return p1 * __shfl_sync(0xFFFFFFFFu, i0, 0);
}

// (Tensor-core kernels.)  Sets the abort flag and the status bit (lane 0), so that the other warps
// leave at their next wait.
__device__ __forceinline__ void tc_give_up(const Params& p, volatile int* abort_flag, int lane) {
  if (lane == 0) {
    *abort_flag = 1;
    flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
  }
}

// Waits for the phase of parity `parity` of `bar` (bounded) with the whole
// warp agreeing on the outcome; false on time-out or abort.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, kWaitTimeoutNs) && !*abort_flag;
  return __all_sync(0xFFFFFFFFu, ok);
}

// Byte-wise store of a vector to a destination that is not 16-byte aligned
// (out of line: the aligned path is the one every ordinary call runs).
static __device__ __noinline__ void store_bytes(unsigned char* dst, uint4 v) {
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&v);
  for (int q = 0; q < 16; ++q) dst[q] = b[q];
}
static __device__ __noinline__ void store_bytes(unsigned char* dst, uint2 v) {
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&v);
  for (int q = 0; q < 8; ++q) dst[q] = b[q];
}

// Stochastic rounding of 8 consecutive 16-bit elements (one Philox call,
// counter (e/8, dst_slot, layer, 0) with e the first element's index; word i
// rounds elements 2i and 2i + 1) into their 16 bytes.
template <int SF>
__device__ __forceinline__ uint4 sr_words8(float2 a0, float2 a1, float2 a2, float2 a3, uint4 r) {
  return make_uint4(sr_pack2<SF>(a0.x, a0.y, r.x), sr_pack2<SF>(a1.x, a1.y, r.y), sr_pack2<SF>(a2.x, a2.y, r.z),
                    sr_pack2<SF>(a3.x, a3.y, r.w));
}

// Kept out of line, so that the code of the rounding-to-nearest path, which
// every call without Philox runs, stays compact.
template <int SF>
__device__ __noinline__ uint4 sr_pack8(float2 a0, float2 a1, float2 a2, float2 a3, uint32_t blk, uint32_t slot,
                                       uint32_t layer, uint32_t key0, uint32_t key1, int rounds) {
  return sr_words8<SF>(a0, a1, a2, a3, philox4x32(make_uint4(blk, slot, layer, 0u), key0, key1, rounds));
}

// The same for two rows of 8 elements (calls blk_a and blk_b): two independent
// Philox chains side by side.
struct RawPair {
  uint4 a, b;
};

template <int SF>
__device__ __noinline__ RawPair sr_pack8x2(float2 a0, float2 a1, float2 a2, float2 a3, float2 b0, float2 b1, float2 b2,
                                           float2 b3, uint32_t blk_a, uint32_t blk_b, uint32_t slot, uint32_t layer,
                                           uint32_t key0, uint32_t key1, int rounds) {
  uint4 r[2] = {make_uint4(blk_a, slot, layer, 0u), make_uint4(blk_b, slot, layer, 0u)};
  philox4x32_n<2>(r, key0, key1, rounds);
  return RawPair{sr_words8<SF>(a0, a1, a2, a3, r[0]), sr_words8<SF>(b0, b1, b2, b3, r[1])};
}

// One item with a non-empty prefix on the CUDA cores: the decay scan, the
// prefix applied to this thread's [RPT rows x VEC columns] of the tile in
// closed form (the tokens converted kTokChunk at a time into the warp's fp32
// buffer `cbuf`), requantization and the store.  The slot is released (empty
// barrier) as soon as the warp holds all it still needs.
template <int SF, int IF, int D, int N>
__device__ __forceinline__ void replay_ffma(const Params& p, const unsigned char* sb, const ItemLayout& il,
                                            const ItemDesc* desc, int k, float* wbuf, float* cbuf, int cw, int lane,
                                            uint32_t empty_bar, uint32_t key0, uint32_t key1, bool sr) {
  constexpr int ES = Fmt<SF>::bytes;
  constexpr int IE = In<IF>::bytes;
  constexpr bool Q = Fmt<SF>::quant;
  constexpr ThreadLayout TL = thread_layout(D, N, ES);
  constexpr int VEC = TL.vec, LPR = TL.lpr, CT = TL.ct, SLAB_ROWS = TL.slab_rows, RPT = TL.rpt, COLS = TL.cols;
  constexpr int V2 = VEC / 2;
  using Raw = typename Vec<SF>::Raw;
  constexpr int XW = SLAB_ROWS % 4 == 0 ? 4 : (SLAB_ROWS % 2 == 0 ? 2 : 1);
  static_assert(RPT == 1 || RPT % 2 == 0, "rows per thread");
  float* bbuf = cbuf + kTokChunk * SLAB_ROWS;  // after c of kTokChunk tokens
  const int lane_row = lane / LPR, lane_col = lane % LPR;
  const int slab_row0 = (cw / CT) * SLAB_ROWS;
  const int tile_col0 = (cw % CT) * COLS;
  const int rrow = lane_row * RPT;
  const int row0 = slab_row0 + rrow;
  const int ccol = lane_col * VEC;
  const int col0 = tile_col0 + ccol;
  const bool worker = rrow < SLAB_ROWS;
  (void)ccol;
  const uint32_t flags = desc->flags;
  unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
  float* dst_sc = reinterpret_cast<float*>(desc->dst_scale);
  const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
  const int h = desc->head;
  const uint32_t dst_slot_id = static_cast<uint32_t>(desc->dst_slot);
  const uint32_t layer_id = static_cast<uint32_t>(desc->layer);
  auto release = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);
  };
    // decay of each token, once per warp: a_t = exp(dt_t*A), then
    // w_t = dt_t * prod_{s>t} a_s and P = prod_t a_t by a suffix-product scan
    const float P = decay_scan(reinterpret_cast<const float*>(sb + il.off_dt), desc->A[0], k, lane, wbuf);

    // this thread's [RPT rows x VEC columns] of the tile, dequantized, times P
    float2 acc[RPT][V2];
    if (worker) {
      const float2 P2 = make_float2(P, P);
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const Raw raw = *reinterpret_cast<const Raw*>(sb + ((row0 + r) * N + col0) * ES);
        unpack_vec<SF>(raw, acc[r]);
        if constexpr (Q) {
          // code * (scale * P): the row's scale folded into the decay product
          const float sp = reinterpret_cast<const float*>(sb + il.off_scale)[row0 + r] * P;
          const float2 sp2 = make_float2(sp, sp);
#pragma unroll
          for (int u = 0; u < V2; ++u) acc[r][u] = __fmul2_rn(acc[r][u], sp2);
        } else {
#pragma unroll
          for (int u = 0; u < V2; ++u) acc[r][u] = __fmul2_rn(acc[r][u], P2);
        }
      }
    }
    __syncwarp();  // wbuf visible to the whole warp

    // the prefix, kTokChunk tokens at a time: convert this warp's share of
    // the tokens to fp32 (c = w*x for its rows, B for its columns), then one
    // rank-1 update per token with packed fp32x2 FMAs.  (c is stored once and
    // paired in registers: storing (c, c) pairs made the 48-layer bf16 shape
    // 0.7% slower, 6% at 8 requests.)
    const unsigned char* xs = sb + il.off_x;
    const unsigned char* Bs = sb + il.off_B;
    for (int t0 = 0; t0 < k; t0 += kTokChunk) {
      const int tn = min(kTokChunk, k - t0);
      for (int u = lane; u < tn * (SLAB_ROWS / XW); u += 32) {
        const int t = u / (SLAB_ROWS / XW), rx = (u % (SLAB_ROWS / XW)) * XW;
        float xv[XW];
        load_inputs<IF, XW>(xs + ((t0 + t) * D + slab_row0 + rx) * IE, xv);
        const float wt = wbuf[t0 + t];
        float* dst = cbuf + t * SLAB_ROWS + rx;
        if constexpr (XW == 4) {
          *reinterpret_cast<float4*>(dst) = make_float4(xv[0] * wt, xv[1] * wt, xv[2] * wt, xv[3] * wt);
        } else if constexpr (XW == 2) {
          *reinterpret_cast<float2*>(dst) = make_float2(xv[0] * wt, xv[1] * wt);
        } else {
          dst[0] = xv[0] * wt;
        }
      }
      for (int u = lane; u < tn * (COLS / 8); u += 32) {
        const int t = u / (COLS / 8), j8 = (u % (COLS / 8)) * 8;
        float bv[8];
        load_inputs<IF, 8>(Bs + ((t0 + t) * N + tile_col0 + j8) * IE, bv);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = j8 + 4 * h, lc = j / VEC, o = j % VEC;  // o is a multiple of 4
          *reinterpret_cast<float4*>(bbuf + t * COLS + (o / 4) * (LPR * 4) + lc * 4) =
              make_float4(bv[4 * h], bv[4 * h + 1], bv[4 * h + 2], bv[4 * h + 3]);
        }
      }
      __syncwarp();
      if (t0 + kTokChunk >= k) release();  // the last chunk: nothing more is read from the stage
      if (worker) {
#pragma unroll 2
        for (int t = 0; t < tn; ++t) {
          float c[RPT];
          float2 b2[V2];
          const float* cp = cbuf + t * SLAB_ROWS + rrow;
          if constexpr (RPT % 4 == 0) {
#pragma unroll
            for (int r = 0; r < RPT; r += 4) {
              const float4 v = *reinterpret_cast<const float4*>(cp + r);
              c[r] = v.x; c[r + 1] = v.y; c[r + 2] = v.z; c[r + 3] = v.w;
            }
          } else if constexpr (RPT % 2 == 0) {
#pragma unroll
            for (int r = 0; r < RPT; r += 2) {
              const float2 v = *reinterpret_cast<const float2*>(cp + r);
              c[r] = v.x; c[r + 1] = v.y;
            }
          } else {
#pragma unroll
            for (int r = 0; r < RPT; ++r) c[r] = cp[r];
          }
#pragma unroll
          for (int g = 0; g < VEC / 4; ++g) {
            const float4 v = *reinterpret_cast<const float4*>(bbuf + t * COLS + g * (LPR * 4) + lane_col * 4);
            b2[2 * g] = make_float2(v.x, v.y);
            b2[2 * g + 1] = make_float2(v.z, v.w);
          }
#pragma unroll
          for (int r = 0; r < RPT; ++r) {
#pragma unroll
            for (int u = 0; u < V2; ++u) acc[r][u] = __ffma2_rn(make_float2(c[r], c[r]), b2[u], acc[r][u]);
          }
        }
      }
      __syncwarp();  // the chunk buffer is rewritten by the next chunk
    }

    // requantize + store
    // one-byte formats: lanes with lane_col % RSPAN == 0 own row row0 + lane_col / RSPAN
    constexpr int RSPAN = LPR / RPT;
    float scale_own = 0.0f;
    bool zero_rows[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) zero_rows[r] = false;
    if constexpr (Q) {
      // symmetric per-(head, row) scale.  The row amax is a transpose
      // reduction over the LPR lanes of the row group: at each of the first
      // log2(RPT) levels a lane keeps half of its rows and trades the other
      // half with its partner, so that afterwards each lane holds one row,
      // row lane_col / RSPAN, reduced over a RSPAN-lane span; the remaining
      // levels reduce that span.  Each lane divides its row's inverse and
      // scale once, and the inverses are shuffled to the rest.
      static_assert(RPT <= LPR && (RPT & (RPT - 1)) == 0 && (LPR & (LPR - 1)) == 0, "row reduction shape");
      float amax[RPT];
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        amax[r] = 0.0f;
#pragma unroll
        for (int u = 0; u < V2; ++u) amax[r] = fmaxf(amax[r], fmaxf(fabsf(acc[r][u].x), fabsf(acc[r][u].y)));
      }
#pragma unroll
      for (int s = 0; (RPT >> s) > 1; ++s) {
        const int half = (RPT >> s) / 2, off = LPR >> (s + 1);
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = upper ? amax[i] : amax[i + half];
          const float keep = upper ? amax[i + half] : amax[i];
          amax[i] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, off));
        }
      }
      float am = amax[0];
#pragma unroll
      for (int off = RSPAN / 2; off >= 1; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
      constexpr float qmax = SF == RSM_I8 ? 127.0f : 448.0f;
      const float inv_own = __fdiv_rn(qmax, am);
      scale_own = inv_own <= FLT_MAX ? __fdiv_rn(am, qmax) : 0.0f;
      const int row_lane0 = lane & ~(LPR - 1);
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const float inv = __shfl_sync(0xFFFFFFFFu, inv_own, row_lane0 + r * RSPAN);
        // a row whose qmax/amax is not finite (amax == 0 or tiny) becomes zero
        // codes: its packed words are cleared after the (then meaningless)
        // scaling and rounding
        zero_rows[r] = !(inv <= FLT_MAX);
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int u = 0; u < V2; ++u) acc[r][u] = __fmul2_rn(acc[r][u], inv2);
      }
    }
    auto store_row = [&](int r, Raw out) {
      if constexpr (Q) {
        if (zero_rows[r]) out = Raw{};
      }
      const uint32_t off = ((row0 + r) * N + col0) * ES;
      if (dst_aligned)
        stg_stream(dst_tile + off, out);
      else
        store_bytes(dst_tile + off, out);
    };
    bool use_sr = false;
    if constexpr (Fmt<SF>::bytes == 2) use_sr = sr;  // one-byte state rounds in its own kernel
    if (worker) {
      if (use_sr) {
        if constexpr (Fmt<SF>::bytes == 2) {
          // Philox counter of element e: (e / 8, dst_slot, layer, 0); a row's
          // 8 elements start on a multiple of 8, so they are one block
          static_assert(V2 == 4, "stochastic rounding works on 8-element vectors");
          const uint32_t blk0 = static_cast<uint32_t>(((static_cast<int64_t>(h) * D + row0) * N + col0) >> 3);
          constexpr uint32_t kRowBlocks = N / 8;
          if constexpr (RPT % 2 == 0) {
#pragma unroll
            for (int r = 0; r < RPT; r += 2) {
              const RawPair o = sr_pack8x2<SF>(acc[r][0], acc[r][1], acc[r][2], acc[r][3], acc[r + 1][0],
                                                   acc[r + 1][1], acc[r + 1][2], acc[r + 1][3], blk0 + r * kRowBlocks,
                                                   blk0 + (r + 1) * kRowBlocks, dst_slot_id, layer_id, key0, key1,
                                                   p.philox_rounds);
              store_row(r, o.a);
              store_row(r + 1, o.b);
            }
          } else {
#pragma unroll
            for (int r = 0; r < RPT; ++r)
              store_row(r, sr_pack8<SF>(acc[r][0], acc[r][1], acc[r][2], acc[r][3], blk0 + r * kRowBlocks,
                                        dst_slot_id, layer_id, key0, key1, p.philox_rounds));
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < RPT; ++r) store_row(r, pack_vec_rne<SF>(acc[r]));
      }
    }
    if constexpr (Q) {
      if (lane_col % RSPAN == 0) {
        const int srow = row0 + lane_col / RSPAN;
        if (flags & kFlagScaleAligned) {
          dst_sc[srow] = scale_own;
        } else {
          const unsigned char* vb = reinterpret_cast<const unsigned char*>(&scale_own);
          unsigned char* db = reinterpret_cast<unsigned char*>(dst_sc + srow);
          for (int q = 0; q < 4; ++q) db[q] = vb[q];
        }
      }
    }
}

template <int SF, int IF, int D, int N>
__device__ __forceinline__ void run_consumer(const Params& p, unsigned char* smem, int cw, int lane) {
  constexpr int ES = Fmt<SF>::bytes;
  constexpr int IE = In<IF>::bytes;
  constexpr bool Q = Fmt<SF>::quant;
  constexpr ThreadLayout TL = thread_layout(D, N, ES);
  constexpr int VEC = TL.vec, LPR = TL.lpr, CT = TL.ct, SLAB_ROWS = TL.slab_rows, RPT = TL.rpt, COLS = TL.cols;
  static_assert(VEC == Vec<SF>::N && VEC % 2 == 0, "vector width");
  using Raw = typename Vec<SF>::Raw;
  static_assert(TL.tct % LPR == 0 && kConsumerWarps % CT == 0 && D % TL.slabs == 0, "thread layout");
  static_assert(SLAB_ROWS % TL.rpw == 0 || SLAB_ROWS < TL.rpw, "rows must split evenly");
  static_assert(!Q || SLAB_ROWS >= TL.rpw, "one-byte formats need every consumer lane busy");
  static_assert(COLS % 8 == 0, "token-chunk buffer vectors");

  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* wbuf = reinterpret_cast<float*>(smem + kWeightOff) + cw * kWeightStride;
  // this warp's fp32 token chunk: c[t][r] = w_t * x_t[slab row r] and the B_t
  // values of its column tile.  B is stored in float4 groups interleaved by
  // lane: column o of lane column lc sits at t*COLS + (o/4)*LPR*4 + lc*4 + o%4,
  // so that the eight lanes of a quarter-warp read 128 contiguous bytes.
  float* cbuf = reinterpret_cast<float*>(smem + kWarpBufOff) + cw * warp_buf_floats(D, N, ES);
  static_assert(VEC % 4 == 0, "B chunk groups");

  const int lane_row = lane / LPR, lane_col = lane % LPR;
  const int slab_row0 = (cw / CT) * SLAB_ROWS;  // first tile row of this warp's slab
  const int tile_col0 = (cw % CT) * COLS;       // first tile column of this warp's column tile
  const int rrow = lane_row * RPT;              // this thread's first row inside the slab
  const int row0 = slab_row0 + rrow;
  const int ccol = lane_col * VEC;              // this thread's first column inside the column tile
  const int col0 = tile_col0 + ccol;
  const bool worker = rrow < SLAB_ROWS;

  uint32_t key0 = 0, key1 = 0;
  const bool sr = p.philox_rounds > 0;
  if (sr) {
    const uint64_t s = static_cast<uint64_t>(__ldg(p.rand_seed));
    key0 = static_cast<uint32_t>(s);
    key1 = static_cast<uint32_t>(s >> 32);
  }

  const uint32_t item_max = item_layout(D, N, ES, Q, IE, p.W).bytes;
  uint32_t arena_head = 0;  // where the loader's next item goes (arena_next)
  uint32_t stage = 0, phase = 0;
  for (;;) {
    if (!mbar_wait(full0 + 8u * stage, phase, kWaitTimeoutNs) || *abort_flag) {
      if (lane == 0) {
        *abort_flag = 1;
        flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
      }
      break;
    }
    // the item's data (tile, scales, x rows, B rows, dt), placed as the loader places it
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    const unsigned char* sb = smem + p.arena0 + off;
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = desc->flags;
    if (flags & kFlagEnd) break;
    // everything the item needs from its descriptor, read before the slot is released
    const int k = desc->k;
    const ItemLayout il = item_layout(D, N, ES, Q, IE, k);
    arena_head = off + il.bytes;
    unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
    float* dst_sc = reinterpret_cast<float*>(desc->dst_scale);
    const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
    // A warp releases the stage as soon as it holds all it still needs (in
    // registers or in its private chunk buffer), so that the loader refills it
    // while this warp computes and stores.
    const uint32_t empty_bar = empty0 + 8u * stage;
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    };

    if (k == 0) {
      // exact copy of the source tile (and scales)
      Raw raw[RPT];
      float scv = 0.0f;
      if (worker) {
#pragma unroll
        for (int r = 0; r < RPT; ++r)
          raw[r] = *reinterpret_cast<const Raw*>(sb + ((row0 + r) * N + col0) * ES);
      }
      const int sr_row = cw * 32 + lane;  // one scale per consumer thread (D <= 256)
      if constexpr (Q) {
        if (sr_row < D) scv = reinterpret_cast<const float*>(sb + il.off_scale)[sr_row];
      }
      release();
      if (worker) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const uint32_t off = ((row0 + r) * N + col0) * ES;
          if (dst_aligned)
            stg_stream(dst_tile + off, raw[r]);
          else
            store_bytes(dst_tile + off, raw[r]);
        }
      }
      if constexpr (Q) {
        if (sr_row < D) {
          if (flags & kFlagScaleAligned) {
            dst_sc[sr_row] = scv;
          } else {
            const unsigned char* vb = reinterpret_cast<const unsigned char*>(&scv);
            unsigned char* db = reinterpret_cast<unsigned char*>(dst_sc + sr_row);
            for (int q = 0; q < 4; ++q) db[q] = vb[q];
          }
        }
      }
    } else {
      replay_ffma<SF, IF, D, N>(p, sb, il, desc, k, wbuf, cbuf, cw, lane, empty_bar, key0, key1, sr);
    }
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

template <int SF, int IF, int D, int N>
__global__ void __launch_bounds__(kThreads, 2) materialize_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  // empty active list: one load, then out
  if (__ldg(p.active) == -1) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const uint32_t full0 = smem_addr(smem);
    for (uint32_t s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8u * s, 1u);
      mbar_init(full0 + 8u * kMaxStages + 8u * s, kConsumerWarps);
    }
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0)
    run_loader<SF, IF, D, N>(p, smem, lane);
  else
    run_consumer<SF, IF, D, N>(p, smem, warp - 1, lane);
}

// The one-byte kernel (rsm_q8_kernel.cuh): rounding to nearest, or
// stochastic rounding (SR).
template <int SF, int IF, bool SR>
const void* q8_kernel();

// Instantiation hook: each translation unit that includes this header (and,
// for one-byte state, rsm_q8_kernel.cuh) provides kernel_for<...>() for its
// formats: the kernel a call with philox_rounds == 0 launches, and for 16-bit
// and fp32 state the one for every call.
template <int SF, int IF, int D, int N>
const void* kernel_for() {
  if constexpr (Fmt<SF>::quant) {
    static_assert(D == 64 && N == 128, "one-byte state is 64 x 128");
    return q8_kernel<SF, IF, false>();
  } else {
    return reinterpret_cast<const void*>(&materialize_kernel<SF, IF, D, N>);
  }
}

// One-byte state with stochastic rounding: the one-byte kernel's instance
// that draws the Philox words.
template <int SF, int IF, int D, int N>
const void* kernel_for_sr() {
  static_assert(Fmt<SF>::quant && D == 64 && N == 128, "the stochastic-rounding instance is one-byte state");
  return q8_kernel<SF, IF, true>();
}

}  // namespace rsm
