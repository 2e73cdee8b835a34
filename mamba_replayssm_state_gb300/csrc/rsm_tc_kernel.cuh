// rsm_tc_kernel.cuh -- the long-window variant of the materialization kernel:
// the replayed prefix applied as a dense contraction on the tensor cores.
//
// In closed form a head's replay is S_k = P * S_0 + C B with C[i][t] =
// w_t x_t[i] (64 x k) and B[t][j] = B_t[j] (k x 128): a rank-k update.  For
// long prefixes that is a matrix product worth the tensor cores.  Per item the
// consumer warps write both operands into shared memory as bf16 K-major core
// matrices (A = B^T: 128 x k, from the bf16 ring rows exactly; the second
// operand = C^T: 64 x k, w_t x_t rounded to bf16), one thread issues
// ceil(k/16) tcgen05.mma (M = 128 dstate columns, N = 64 dim rows, K = 16)
// accumulating S^T - P S_0^T in TMEM (fp32), and every consumer thread reads
// its TMEM lane (one dstate column j, 32 dim rows), adds P S_0, rounds and
// stores its elements straight to global memory (a warp writes 64 contiguous
// bytes per tile row).  The item's slot is released as soon as the operands
// are built: S_0 and P are in registers by then, so the loader refills the
// slot while the MMA and the epilogue run.
//
// The loader warp, the arena and the slots are the materialization kernel's.
// Prefixes shorter than p.tc_min_k tokens take the CUDA-core path of the
// materialization kernel (its fixed cost is lower), with its token buffers in
// the operand region.
// The consumer warps synchronise on mbarriers with bounded waits (never an
// unbounded bar.sync), so a broken run ends with a status bit.  TMEM (64
// columns) is allocated by consumer warp 0 before the loop and freed by it at
// the end.
#pragma once
#include "rsm_kernel.cuh"
#include "rsm_tc.cuh"

namespace rsm {

template <int SF>
__device__ __forceinline__ float to_f32_16(uint32_t bits) {
  if constexpr (SF == RSM_BF16) {
    return __uint_as_float(bits << 16);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
  }
}

template <int SF>
__device__ __forceinline__ uint32_t from_f32_16(float v) {
  // round to nearest even (values already rounded stochastically stay exact)
  return SF == RSM_BF16 ? (pack_bf16x2(v, 0.0f) & 0xFFFFu) : (pack_f16x2(v, 0.0f) & 0xFFFFu);
}

// The epilogue for stochastic rounding or a misaligned destination, out of
// line (rare paths): S = P S_0 + acc for this thread's column j, rows i0..i0+31.
template <int SF>
__device__ __noinline__ void tc_epilogue_slow(const Params& p, uint32_t taddr, uint32_t s00, uint32_t s01,
                                              uint32_t s02, uint32_t s03, uint32_t s04, uint32_t s05, uint32_t s06,
                                              uint32_t s07, uint32_t s08, uint32_t s09, uint32_t s10, uint32_t s11,
                                              uint32_t s12, uint32_t s13, uint32_t s14, uint32_t s15, float P,
                                              unsigned char* out_col, bool dst_aligned, bool sr, int h, int i0, int j,
                                              uint32_t dst_slot_id, uint32_t layer_id, uint32_t key0,
                                              uint32_t key1) {
  constexpr int D = 64, N = 128;
  const uint32_t s0[16] = {s00, s01, s02, s03, s04, s05, s06, s07, s08, s09, s10, s11, s12, s13, s14, s15};
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    float acc[16];
    tmem_ld16(taddr + 16u * part, acc);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t pair = s0[8 * part + c / 2];
      const float x0 = to_f32_16<SF>(c & 1 ? pair >> 16 : pair & 0xFFFFu);
      float y = fmaf(P, x0, acc[c]);
      if (sr) {
        const int64_t e = (static_cast<int64_t>(h) * D + i0 + 16 * part + c) * N + j;
        const uint4 rnd = philox4x32(make_uint4(static_cast<uint32_t>(e >> 2), dst_slot_id, layer_id, 0u), key0,
                                     key1, p.philox_rounds);
        const uint32_t wsel = (e & 3) == 0 ? rnd.x : (e & 3) == 1 ? rnd.y : (e & 3) == 2 ? rnd.z : rnd.w;
        y = sr_fmt<SF>(y, wsel);
      }
      const uint32_t v = from_f32_16<SF>(y);
      unsigned char* q = out_col + static_cast<uint32_t>(i0 + 16 * part + c) * (N * 2u);
      if (dst_aligned) {
        stg16_stream(q, static_cast<uint16_t>(v));
      } else {
        q[0] = static_cast<unsigned char>(v);
        q[1] = static_cast<unsigned char>(v >> 8);
      }
    }
  }
}

template <int SF>
__device__ __forceinline__ void run_consumer_tc(const Params& p, unsigned char* smem, int cw, int lane,
                                                uint32_t tmem) {
  static_assert(SF == RSM_BF16 || SF == RSM_F16, "16-bit state only");
  constexpr int D = 64, N = 128, ES = 2, IE = 2;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * kMaxStages;
  const uint32_t mma_bar = sbase + kTcBarOff;
  const uint32_t xbar1 = mma_bar + 8u, xbar2 = mma_bar + 16u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* wbuf = reinterpret_cast<float*>(smem + kWeightOff) + cw * kWeightStride;
  unsigned char* aop = smem + kTcAOff;  // A operand
  unsigned char* bop = smem + kTcBOff;
  // short prefixes run on the CUDA cores with per-warp token buffers inside the operand region
  float* cbuf = reinterpret_cast<float*>(smem + kTcAOff) + cw * warp_buf_floats(D, N, ES);
  static_assert(kConsumerWarps * warp_buf_floats(64, 128, 2) * 4 <= kTcDescBase - kTcAOff, "token buffers");
  const int tid = cw * 32 + lane;       // 0 .. 255 over the consumer warps
  const int quarter = (cw + 1) & 3;     // TMEM lane quarter this warp may access (CTA warp id % 4)
  const int half = cw >> 2;             // which 32 of the 64 accumulator columns
  const int j = 32 * quarter + lane;    // this thread's dstate column = its TMEM lane
  const int i0 = 32 * half;             // its first dim row
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 64);

  uint32_t key0 = 0, key1 = 0;
  const bool sr = p.philox_rounds > 0;
  if (sr) {
    const uint64_t s = static_cast<uint64_t>(__ldg(p.rand_seed));
    key0 = static_cast<uint32_t>(s);
    key1 = static_cast<uint32_t>(s >> 32);
  }
  auto give_up = [&]() {
    if (lane == 0) {
      *abort_flag = 1;
      flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
    }
  };
  uint32_t xpar = 0, x1par = 0, mpar = 0;
  bool prev_tc = false;  // the last item with a prefix went through the MMA
  // every consumer warp arrives, then all wait (bounded)
  // (every exit decision is taken by the whole warp: the warp-wide tcgen05
  // instructions below must never see a partial warp)
  auto xsync = [&](uint32_t bar) -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, xpar, kWaitTimeoutNs) && !*abort_flag;
    return __all_sync(0xFFFFFFFFu, ok);
  };

  const uint32_t item_max = item_layout(D, N, ES, false, IE, p.W).bytes;
  uint32_t arena_head = 0;
  uint32_t stage = 0, phase = 0;
  for (;;) {
    const bool full_ok = mbar_wait(full0 + 8u * stage, phase, kWaitTimeoutNs) && !*abort_flag;
    if (!__all_sync(0xFFFFFFFFu, full_ok)) {
      give_up();
      break;
    }
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    const unsigned char* sb = smem + p.arena0 + off;
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = __shfl_sync(0xFFFFFFFFu, desc->flags, 0);
    if (flags & kFlagEnd) break;
    const int k = __shfl_sync(0xFFFFFFFFu, desc->k, 0);
    const bool same_B = (flags & kFlagSameB) != 0u;  // the A operand of the previous item still holds
    const ItemLayout il = item_layout(D, N, ES, false, IE, k, !same_B);
    arena_head = off + il.bytes;
    unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
    const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
    const int h = desc->head;
    const uint32_t dst_slot_id = static_cast<uint32_t>(desc->dst_slot);
    const uint32_t layer_id = static_cast<uint32_t>(desc->layer);
    const uint32_t empty_bar = empty0 + 8u * stage;

    if (k == 0) {
      // exact copy of the source tile: 1024 vectors of 16 bytes over 256 threads
      uint4 v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = reinterpret_cast<const uint4*>(sb)[tid + 256 * r];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t o = static_cast<uint32_t>(tid + 256 * r) * 16u;
        if (dst_aligned) {
          stg128_stream(dst_tile + o, v[r]);
        } else {
          const unsigned char* b = reinterpret_cast<const unsigned char*>(&v[r]);
          for (int q = 0; q < 16; ++q) dst_tile[o + q] = b[q];
        }
      }
    } else if (k < p.tc_min_k) {
      replay_ffma<SF, RSM_BF16, 64, 128, true>(p, sb, il, desc, k, wbuf, cbuf, cw, lane, empty_bar, key0, key1, sr);
      prev_tc = false;
    } else {
      // decay of each token, once per warp (as in the materialization kernel)
      const float P = decay_scan(reinterpret_cast<const float*>(sb + il.off_dt), desc->A, k, lane, wbuf);
      __syncwarp();  // wbuf visible to the whole warp

      // S_0 at this thread's (dim rows i0 .. i0+31, dstate column j), kept as
      // packed 16-bit pairs until the epilogue
      uint32_t s0[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        s0[c] = static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[(i0 + 2 * c) * N + j]) |
                (static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[(i0 + 2 * c + 1) * N + j]) << 16);

      // after a CUDA-core item, every warp is done with its token buffer (inside
      // the operand region) before the operands are written
      if (!prev_tc) {
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar1);
        const bool ok = mbar_wait(xbar1, x1par, kWaitTimeoutNs) && !*abort_flag;
        x1par ^= 1u;
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          give_up();
          break;
        }
      }
      const int kp = (k + 15) & ~15;  // K padded to whole MMAs; tokens k .. kp-1 are zero
      const uint16_t* Brows = reinterpret_cast<const uint16_t*>(sb + il.off_B);
      const uint16_t* xrows = reinterpret_cast<const uint16_t*>(sb + il.off_x);
      for (int u = same_B ? 128 * (kp / 8) : tid; u < 128 * (kp / 8); u += 256) {  // A = B^T (unless reused)
        const int jj = u & 127, tg = u >> 7;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 8 * tg + 2 * e;
          const uint32_t lo = t < k ? Brows[t * N + jj] : 0u;
          const uint32_t hi = t + 1 < k ? Brows[(t + 1) * N + jj] : 0u;
          w[e] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(aop + (jj >> 3) * kTcSbo + tg * 128 + (jj & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      for (int u = tid; u < 64 * (kp / 8); u += 256) {
        const int ii = u & 63, tg = u >> 6;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 8 * tg + 2 * e;
          const float lo = t < k ? wbuf[t] * __uint_as_float(static_cast<uint32_t>(xrows[t * D + ii]) << 16) : 0.0f;
          const float hi =
              t + 1 < k ? wbuf[t + 1] * __uint_as_float(static_cast<uint32_t>(xrows[(t + 1) * D + ii]) << 16) : 0.0f;
          w[e] = pack_bf16x2(lo, hi);
        }
        *reinterpret_cast<uint4*>(bop + (ii >> 3) * kTcSbo + tg * 128 + (ii & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();  // the operands, written by this thread, before the tensor cores read them
      // the warp holds all it still needs from the item (S_0 and P in
      // registers, the operands in their own buffers): the slot goes back to
      // the loader while the MMA and the epilogue run
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
      tc_fence_before();
      if (!xsync(xbar2)) {
        give_up();
        break;
      }
      tc_fence_after();
      if (tid == 0) {
        const uint64_t adesc0 = smem_desc_kmajor(sbase + kTcAOff, 128u, kTcSbo);
        const uint64_t bdesc0 = smem_desc_kmajor(sbase + kTcBOff, 128u, kTcSbo);
        for (int kc = 0; kc < kp / 16; ++kc)  // the start address field counts 16-byte units: +256 B per step
          tc_mma_bf16(tmem, adesc0 + static_cast<uint64_t>(16 * kc), bdesc0 + static_cast<uint64_t>(16 * kc), kIdesc,
                      kc > 0 ? 1u : 0u);
        tc_commit(mma_bar);
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(mma_bar, mpar, kWaitTimeoutNs))) {
        give_up();
        break;
      }
      mpar ^= 1u;
      tc_fence_after();
      // S = P S_0 + (C B), rounded and stored straight from registers, 16
      // accumulator columns at a time.  Rounding to nearest into an aligned
      // tile is the common path, kept inline; stochastic rounding and
      // misaligned tiles go out of line, which keeps this kernel's registers
      // and code small (measured 6-15% faster at every prefix length than
      // with both paths inline)
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(i0);
      unsigned char* out_col = dst_tile + static_cast<uint32_t>(j) * 2u;
      if (!sr && dst_aligned) {
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float acc[16];
          tmem_ld16(taddr + 16u * part, acc);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint32_t pair = s0[8 * part + c / 2];
            const float x0 = to_f32_16<SF>(c & 1 ? pair >> 16 : pair & 0xFFFFu);
            stg16_stream(out_col + static_cast<uint32_t>(i0 + 16 * part + c) * (N * 2u),
                         static_cast<uint16_t>(from_f32_16<SF>(fmaf(P, x0, acc[c]))));
          }
        }
      } else {
        tc_epilogue_slow<SF>(p, taddr, s0[0], s0[1], s0[2], s0[3], s0[4], s0[5], s0[6], s0[7], s0[8], s0[9], s0[10],
                             s0[11], s0[12], s0[13], s0[14], s0[15], P, out_col, dst_aligned, sr, h, i0, j,
                             dst_slot_id, layer_id, key0, key1);
      }
      // (every warp's TMEM reads end before the next MMA overwrites the
      // accumulator: they precede its arrival at the next operand barrier)
      xpar ^= 1u;
      prev_tc = true;
    }
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

template <int SF>
__global__ void __launch_bounds__(kThreads, 2) materialize_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (__ldg(p.active) == -1) return;  // empty active list: one load, then out

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  if (warp == 1) {
    tmem_alloc(sbase + kTcTmemSlot, kTcTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.stages; ++s) {
      mbar_init(sbase + 8u * s, 1u);
      mbar_init(sbase + 8u * kMaxStages + 8u * s, kConsumerWarps);
    }
    mbar_init(sbase + kTcBarOff, 1u);  // MMA completion
    for (uint32_t b = 1; b <= 4; ++b) mbar_init(sbase + kTcBarOff + 8u * b, kConsumerWarps);  // x1, x2, spare, exit
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTcTmemSlot);
  if (warp == 0) {
    run_loader<SF, RSM_BF16, 64, 128>(p, smem, lane);
  } else {
    run_consumer_tc<SF>(p, smem, warp - 1, lane, tmem);
    // every consumer warp is done with TMEM before the allocating warp frees it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcBarOff + 32u);
    if (warp == 1) {
      (void)mbar_wait(sbase + kTcBarOff + 32u, 0u, 3ull * kWaitTimeoutNs);
      tc_fence_after();
      tmem_dealloc(tmem, kTcTmemCols);
    }
  }
}

template <int SF>
const void* kernel_for_tc() {
  return reinterpret_cast<const void*>(&materialize_tc_kernel<SF>);
}

}  // namespace rsm
