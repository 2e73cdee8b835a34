// rsm_q8tc_kernel.cuh -- one-byte state (int8 or fp8 e4m3 codes with one fp32
// scale per (head, dim row); API page, Parameters: state_dtype,
// state_scale_ptrs; one-byte state is 64 x 128) with the replayed prefix on
// the tensor cores.
//
// In closed form a head's replay is S_k = P S_0 + C B with C[i][t] = w_t x_t[i]
// and B[t][j] the ring rows: a rank-k contraction.  On the CUDA cores it costs
// k FMAs per element, and for one-byte state, whose bytes carry a decode, a row
// maximum and a requantization on top, the kernel is then bound by
// instruction issue rather than by memory.  Here the contraction runs on the
// tensor cores and the CUDA cores keep only the per-element format work.
//
// An item is a pair of consecutive heads of one B group (the loader's HPI = 2:
// their tiles, scales and x rows are adjacent in memory).  Its accumulator is
// M = 128 rows (head pair x 64 dim rows, the TMEM lanes) x N = 128 dstate
// columns, so that one epilogue thread holds one whole tile row and the row's
// maximum needs no exchange between threads.  Operands, MN-major with the
// 128-byte swizzle (a token's 128-element row is a row of two swizzle atoms):
//   C = w x, split into two bf16 operands, hi = bf16(c) and lo = bf16(c - hi),
//     so that hi + lo carries 16 significant bits of c (the CUDA-core kernels
//     keep c in fp32; plain bf16 would round it to 8);
//   B, the bf16 ring rows, exact.
// Both are padded with zero tokens to a multiple of 16; the accumulator
// receives C_hi B + C_lo B from 2 ceil(k/16) MMAs of K = 16.
//
// CTA: the loader warp (the materialization kernel's, two heads per item),
// two builder warps and four epilogue warps.
//   builder warp j (head j of the item): the decay weights of head j, then,
//     once the previous item's MMAs have completed (the operands are
//     single-buffered), its head's half of C_hi and C_lo and its half of B's
//     columns (B only for the first item of a B group); warp 0 issues the MMAs
//     into accumulator n mod 2 once the epilogue has handed it back, and
//     commits them to that accumulator's mbarrier.
//   epilogue warp q (TMEM lane quarter q, tile rows 32q .. 32q + 31; a thread
//     per row): the warp's 32 rows of codes, read coalesced into a swizzled
//     staging buffer, from which each thread then reads its own row without
//     bank conflicts; the slot goes back to the loader.  Once the MMAs are
//     done: S = fl(code * (scale P) + acc), one fma (the decoded state
//     code * scale, decayed, plus the replay, rounded once), written back to
//     TMEM while the row's amax is taken, then read again, requantized (round
//     to nearest even, or Philox stochastic rounding), and stored through the
//     staging buffer as coalesced 16-byte vectors; the accumulator goes back
//     to the builders.
// With two accumulators the MMAs of item n + 1 run while the epilogue drains
// item n.  Every wait is an mbarrier wait bounded in wall time, every exit
// decision is warp-uniform, TMEM (256 columns) is allocated by warp 1 before
// the loop and freed by it after an exit barrier.
#pragma once
#include "rsm_kernel.cuh"
#include "rsm_tc.cuh"

namespace rsm {

// Byte offset of 16-byte chunk c (0..7) of row r in a region of 128-byte rows
// whose chunks are XOR-swizzled by the row (conflict-free both for a warp
// reading four whole rows and for 32 threads reading one chunk of their own row).
__device__ __forceinline__ uint32_t qt_swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// max(m, |a|, |b|) in one instruction (sm_100 three-input maximum of
// absolute values); a NaN operand is ignored, as by fmaxf
__device__ __forceinline__ float absmax3(float m, float a, float b) {
  float r;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(a), "f"(b));
  return r;
}

template <int SF>
__device__ __forceinline__ void run_builder_qt(const Params& p, unsigned char* smem, int bw, int lane, uint32_t tmem) {
  constexpr int D = 64, N = 128, DI = kQtHeads * D, IE = 2;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* wbuf = reinterpret_cast<float*>(smem + kWeightOff) + bw * kWeightStride;  // head bw's weights
  const uint32_t opb = qt_op_bytes(p.W);
  unsigned char* chi = smem + kQtOpOff;
  unsigned char* clo = chi + opb;
  unsigned char* bop = chi + 2 * opb;
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, true, true);

  const uint32_t item_max = item_layout(DI, N, 1, true, IE, p.W, true, kQtHeads).bytes;
  uint32_t arena_head = 0;
  uint32_t stage = 0, phase = 0;
  uint32_t n_tc = 0;  // items with a replay so far
  // C rows (tokens) t >= c_dirty are zero in both C operands: rows k .. kp-1
  // of an item must be zero (or at least finite: B's are zero), so only rows
  // that an earlier, longer item wrote are cleared.  Nothing is known at the
  // start (the shared memory holds anything).
  int c_dirty = static_cast<int>(qt_kpad(p.W));
  for (;;) {
    if (!tc_wait(full0 + 8u * stage, phase, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    const unsigned char* sb = smem + p.arena0 + off;
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = __shfl_sync(0xFFFFFFFFu, desc->flags, 0);
    if (flags & kFlagEnd) break;
    const int k = __shfl_sync(0xFFFFFFFFu, desc->k, 0);
    const bool same_B = (flags & kFlagSameB) != 0u;  // the B operand of the previous item still holds
    const ItemLayout il = item_layout(DI, N, 1, true, IE, k, !same_B, kQtHeads);
    arena_head = off + il.bytes;
    const uint32_t empty_bar = empty0 + 8u * stage;
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }
    if (k == 0) {  // a copy: the epilogue group's alone
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
      continue;
    }
    // decay weights w_t of head bw
    (void)decay_scan(reinterpret_cast<const float*>(sb + il.off_dt) + bw * k, desc->A[bw], k, lane, wbuf);
    __syncwarp();  // wbuf visible to the whole warp
    // the operands are free once the previous item's MMAs have completed
    if (n_tc > 0 && !tc_wait(sbase + kQtMmaDone + 8u * ((n_tc - 1) & 1u), ((n_tc - 1) >> 1) & 1u, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    const int kp = (k + 15) & ~15;  // K padded to whole MMAs; tokens k .. kp-1 are zero
    // token t's row of an operand: 16 chunks of 8 bf16 along MN; chunk c is in
    // atom column c / 8 of token group t / 8, at chunk (c % 8) ^ (t % 8) of the
    // atom's row t % 8.  This warp writes chunks 8 bw .. 8 bw + 7: its head's
    // 64 rows of C (rows k .. c_dirty-1 cleared), and half of B's columns
    // (rows k .. kp-1 zero).
    const int c_rows = max(k, min(c_dirty, kp));
    const int rows = same_B ? c_rows : kp;
    c_dirty = c_dirty > kp ? c_dirty : k;
    for (int u = lane; u < rows * 8; u += 32) {
      const int t = u >> 3, c = 8 * bw + (u & 7);
      const uint32_t o = static_cast<uint32_t>((t >> 3) * kQtGroup + (c >> 3) * 1024 + (t & 7) * 128 +
                                               (((c & 7) ^ (t & 7)) << 4));
      uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
      if (t < k) {
        const uint4 xv = *reinterpret_cast<const uint4*>(sb + il.off_x + t * (DI * 2) + c * 16);
        const float w = wbuf[t];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v0 = bf16lo(xw[e]) * w, v1 = bf16hi(xw[e]) * w;
          hw[e] = pack_bf16x2(v0, v1);
          // v - hi is exact in fp32; its bf16 rounding is the second operand
          lw[e] = pack_bf16x2(v0 - bf16lo(hw[e]), v1 - bf16hi(hw[e]));
        }
        hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      if (t < c_rows) {
        *reinterpret_cast<uint4*>(chi + o) = hi;
        *reinterpret_cast<uint4*>(clo + o) = lo;
      }
      if (!same_B) {
        const uint4 bv = t < k ? *reinterpret_cast<const uint4*>(sb + il.off_B + t * (N * 2) + c * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(bop + o) = bv;
      }
    }
    fence_proxy_async_smem();  // the operands, written by this thread, before the tensor cores read them
    // the builders are done with the slot's x, B and dt
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);
    // both builder warps have written their halves
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kQtBuildBar);
    if (!tc_wait(sbase + kQtBuildBar, n_tc & 1u, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    tc_fence_after();
    const uint32_t buf = n_tc & 1u;
    if (bw == 0) {
      // the accumulator is free once the epilogue is done with it (two items back)
      const bool ok = n_tc < 2 || tc_wait(sbase + kQtTmemFree + 8u * buf, ((n_tc - 2) >> 1) & 1u, abort_flag);
      if (!ok) {
        tc_give_up(p, abort_flag, lane);
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t dh = smem_desc_mn_sw128(sbase + kQtOpOff, 1024u, kQtGroup);
        const uint64_t dl = smem_desc_mn_sw128(sbase + kQtOpOff + opb, 1024u, kQtGroup);
        const uint64_t db = smem_desc_mn_sw128(sbase + kQtOpOff + 2 * opb, 1024u, kQtGroup);
        // per 16 tokens (two token groups) C_hi B then C_lo B; the start
        // address field counts 16-byte units
        for (int kc = 0; kc < kp / 16; ++kc) {
          const uint64_t step = static_cast<uint64_t>(kc * 2 * kQtGroup / 16);
          tc_mma_bf16(tmem + buf * kQtAccCols, dh + step, db + step, kIdesc, kc > 0 ? 1u : 0u);
          tc_mma_bf16(tmem + buf * kQtAccCols, dl + step, db + step, kIdesc, 1u);
        }
        tc_commit(sbase + kQtMmaDone + 8u * buf);
      }
      __syncwarp();
    }
    ++n_tc;
  }
  // the issuing warp leaves only once its last MMAs have completed, so that
  // TMEM is never freed under them (the epilogue waits for them too, unless a
  // wait ran out)
  if (bw == 0 && n_tc > 0)
    (void)mbar_wait(sbase + kQtMmaDone + 8u * ((n_tc - 1) & 1u), ((n_tc - 1) >> 1) & 1u, kWaitTimeoutNs);
}

// Requantizes 32 consecutive values of a row, times inv = qmax / amax, into 8
// words of codes.  Stochastic rounding: Philox counters c0 and c0 + 1 cover
// columns 0-15 and 16-31 of the 32; word q of a call rounds its columns
// 4q .. 4q + 3.  fp8 values are v * inv + 0, so that a row quantized with
// inv = 0 gets +0 codes even where v is negative.
template <int SF, bool SR>
__device__ __forceinline__ void qt_quantize32(const float (&a)[32], float inv, uint32_t c0, uint32_t dst_slot_id,
                                              uint32_t layer_id, uint32_t key0, uint32_t key1, int rounds,
                                              uint32_t (&w)[8]) {
  const float2 inv2 = make_float2(inv, inv), zero2 = make_float2(0.0f, 0.0f);
  if constexpr (SR) {
    uint4 rw[2] = {make_uint4(c0, dst_slot_id, layer_id, 0u), make_uint4(c0 + 1u, dst_slot_id, layer_id, 0u)};
    philox4x32_n<2>(rw, key0, key1, rounds);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint32_t words[4] = {rw[g].x, rw[g].y, rw[g].z, rw[g].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = 16 * g + 4 * q;
        const float2 v01 = __ffma2_rn(make_float2(a[e], a[e + 1]), inv2, zero2);
        const float2 v23 = __ffma2_rn(make_float2(a[e + 2], a[e + 3]), inv2, zero2);
        if constexpr (SF == RSM_I8) {
          uint32_t r[4];
          sr_r16x4(words[q], r);
          const float2 magic = make_float2(12582912.0f, 12582912.0f);
          const float2 c01 = __fadd2_rn(make_float2(sr_i8(v01.x, r[0]), sr_i8(v01.y, r[1])), magic);
          const float2 c23 = __fadd2_rn(make_float2(sr_i8(v23.x, r[2]), sr_i8(v23.y, r[3])), magic);
          w[4 * g + q] = __byte_perm(__byte_perm(__float_as_uint(c01.x), __float_as_uint(c01.y), 0x0040u),
                                     __byte_perm(__float_as_uint(c23.x), __float_as_uint(c23.y), 0x0040u), 0x5410u);
        } else {
          w[4 * g + q] = sr_e4m3x4(v01.x, v01.y, v23.x, v23.y, words[q]);
        }
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = 4 * q;
      if constexpr (SF == RSM_I8) {
        // round to nearest even in one step: fl(v * inv + 1.5 * 2^23) keeps the
        // exact product's rounding to an integer in its low byte (|v * inv| <= 127.5)
        const float2 magic = make_float2(12582912.0f, 12582912.0f);
        const float2 c01 = __ffma2_rn(make_float2(a[e], a[e + 1]), inv2, magic);
        const float2 c23 = __ffma2_rn(make_float2(a[e + 2], a[e + 3]), inv2, magic);
        w[q] = __byte_perm(__byte_perm(__float_as_uint(c01.x), __float_as_uint(c01.y), 0x0040u),
                           __byte_perm(__float_as_uint(c23.x), __float_as_uint(c23.y), 0x0040u), 0x5410u);
      } else {
        const float2 v01 = __ffma2_rn(make_float2(a[e], a[e + 1]), inv2, zero2);
        const float2 v23 = __ffma2_rn(make_float2(a[e + 2], a[e + 3]), inv2, zero2);
        w[q] = __byte_perm(f32x2_to_e4m3x2(v01.x, v01.y), f32x2_to_e4m3x2(v23.x, v23.y), 0x5410u);
      }
    }
  }
}

template <int SF, bool SR>
__device__ __forceinline__ void run_epilogue_qt(const Params& p, unsigned char* smem, int ew, int warp, int lane,
                                                uint32_t tmem) {
  constexpr int D = 64, N = 128, DI = kQtHeads * D, IE = 2;
  constexpr float qmax = SF == RSM_I8 ? 127.0f : 448.0f;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  const int tid = ew * 32 + lane;    // 0 .. 127 over the epilogue group
  const int quarter = warp & 3;      // TMEM lane quarter this warp may access (CTA warp id % 4)
  const int m = 32 * quarter + lane; // this thread's tile row of the item = its TMEM lane
  const int hj = quarter >> 1;       // the row's head within the item
  const int row_i = m & (D - 1);     // the row's dim index within its head
  unsigned char* stg = smem + qt_stage_off(p.W) + ew * kQtStageBytes;  // this warp's staging (32 rows)
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quarter) << 16);

  uint32_t key0 = 0, key1 = 0;
  if constexpr (SR) {
    const uint64_t s = static_cast<uint64_t>(__ldg(p.rand_seed));
    key0 = static_cast<uint32_t>(s);
    key1 = static_cast<uint32_t>(s >> 32);
  }
  const uint32_t item_max = item_layout(DI, N, 1, true, IE, p.W, true, kQtHeads).bytes;
  uint32_t arena_head = 0;
  uint32_t stage = 0, phase = 0;
  uint32_t n_tc = 0;
  for (;;) {
    if (!tc_wait(full0 + 8u * stage, phase, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    const uint32_t off = arena_next(arena_head, item_max, p.arena_bytes);
    const unsigned char* sb = smem + p.arena0 + off;
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = __shfl_sync(0xFFFFFFFFu, desc->flags, 0);
    if (flags & kFlagEnd) break;
    const int k = __shfl_sync(0xFFFFFFFFu, desc->k, 0);
    const bool same_B = (flags & kFlagSameB) != 0u;
    const ItemLayout il = item_layout(DI, N, 1, true, IE, k, !same_B, kQtHeads);
    arena_head = off + il.bytes;
    unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
    float* dst_sc = reinterpret_cast<float*>(desc->dst_scale);
    const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
    const bool sc_aligned = (flags & kFlagScaleAligned) != 0u;
    const uint32_t empty_bar = empty0 + 8u * stage;
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }

    if (k == 0) {
      // exact copy of the two tiles (1024 vectors of 16 bytes) and their 128 scales
      uint4 v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) v[r] = reinterpret_cast<const uint4*>(sb)[tid + 128 * r];
      const float scv = reinterpret_cast<const float*>(sb + il.off_scale)[tid];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        unsigned char* d = dst_tile + static_cast<uint32_t>(tid + 128 * r) * 16u;
        if (dst_aligned)
          stg128_stream(d, v[r]);
        else
          store_bytes(d, v[r]);
      }
      if (sc_aligned) {
        dst_sc[tid] = scv;
      } else {
        const unsigned char* vb = reinterpret_cast<const unsigned char*>(&scv);
        unsigned char* db = reinterpret_cast<unsigned char*>(dst_sc + tid);
        for (int q = 0; q < 4; ++q) db[q] = vb[q];
      }
      continue;
    }

    // the Philox counter words of this row, read before the slot is released
    const uint32_t dst_slot_id = static_cast<uint32_t>(desc->dst_slot);
    const uint32_t layer_id = static_cast<uint32_t>(desc->layer);
    const uint32_t row_ctr = static_cast<uint32_t>(((desc->head + hj) * D + row_i) * (N / 16));
    // P of the row's head: the product of exp(dt_t A) over the prefix
    float P;
    {
      const float* dts = reinterpret_cast<const float*>(sb + il.off_dt) + hj * k;
      const float A = desc->A[hj];
      float a = lane < k ? expf(dts[lane] * A) : 1.0f;
      if (lane + 32 < k) a *= expf(dts[lane + 32] * A);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a *= __shfl_xor_sync(0xFFFFFFFFu, a, o);
      P = a;
    }
    const float sc = reinterpret_cast<const float*>(sb + il.off_scale)[m];
    // this warp's 32 rows of codes, read four rows at a time (coalesced) into
    // the staging buffer, swizzled: from there each thread reads its own row
    // without bank conflicts, and writes its codes back in the same place
    {
      const unsigned char* rows = sb + 32 * quarter * N;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int r = 4 * s + (lane >> 3), c = lane & 7;
        *reinterpret_cast<uint4*>(stg + qt_swz(r, c)) = *reinterpret_cast<const uint4*>(rows + r * N + c * 16);
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(empty_bar);  // the epilogue is done with the slot

    const uint32_t buf = n_tc & 1u;
    const uint32_t taddr = lane_base + buf * kQtAccCols;
    if (!tc_wait(sbase + kQtMmaDone + 8u * buf, (n_tc >> 1) & 1u, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    tc_fence_after();
    // S = fl(code * (scale P) + acc): the decoded state code * scale, decayed
    // and replayed, rounded once; back into TMEM, and the row's amax
    float am = 0.0f;
    {
      const float sp = sc * P;
      const float2 sp2 = make_float2(sp, sp);
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) {
        float a[32];
        tmem_ld32(taddr + 32u * c2, a);
        const uint4 c0 = *reinterpret_cast<const uint4*>(stg + qt_swz(lane, 2 * c2));
        const uint4 c1 = *reinterpret_cast<const uint4*>(stg + qt_swz(lane, 2 * c2 + 1));
        const uint32_t code[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // four codes a word
          float f[4];
          unpack_words<SF, 1>(code + q, f);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float2 y = __ffma2_rn(make_float2(f[2 * u], f[2 * u + 1]), sp2,
                                        make_float2(a[4 * q + 2 * u], a[4 * q + 2 * u + 1]));
            a[4 * q + 2 * u] = y.x;
            a[4 * q + 2 * u + 1] = y.y;
          }
        }
#pragma unroll
        for (int u = 0; u < 32; u += 2) am = absmax3(am, a[u], a[u + 1]);
        tmem_st32(taddr + 32u * c2, a);
      }
      tmem_st_wait();
    }
    // a row whose qmax / amax is not finite (amax 0 or tiny) gets scale 0 and
    // zero codes: it is quantized with inv = 0 (its values are all finite and
    // tiny, so every product is 0).  The stored scale is the correctly rounded
    // amax / qmax; the multiplier qmax / amax that codes are computed with is a
    // fast division (within 2 ulps: a code moves only where v * qmax / amax
    // lies within 2 ulps of a rounding boundary, and |v| * inv stays below
    // 127.5 for int8)
    float inv = __fdividef(qmax, am);
    const bool finite = inv <= FLT_MAX;
    const float scale = finite ? __fdiv_rn(am, qmax) : 0.0f;
    if (!finite) inv = 0.0f;
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2) {
      float a[32];
      tmem_ld32(taddr + 32u * c2, a);
      uint32_t w[8];
      qt_quantize32<SF, SR>(a, inv, row_ctr + 2u * c2, dst_slot_id, layer_id, key0, key1, p.philox_rounds, w);
      *reinterpret_cast<uint4*>(stg + qt_swz(lane, 2 * c2)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(stg + qt_swz(lane, 2 * c2 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    // the accumulator goes back to the builders
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kQtTmemFree + 8u * buf);
    // the warp's 32 rows out, four whole rows (512 contiguous bytes) per store
    __syncwarp();
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int r = 4 * s + (lane >> 3), c = lane & 7;
      const uint4 v = *reinterpret_cast<const uint4*>(stg + qt_swz(r, c));
      unsigned char* d = dst_tile + static_cast<uint32_t>((32 * quarter + r) * N + c * 16);
      if (dst_aligned)
        stg128_stream(d, v);
      else
        store_bytes(d, v);
    }
    if (sc_aligned) {
      dst_sc[m] = scale;
    } else {
      const unsigned char* vb = reinterpret_cast<const unsigned char*>(&scale);
      unsigned char* db = reinterpret_cast<unsigned char*>(dst_sc + m);
      for (int q = 0; q < 4; ++q) db[q] = vb[q];
    }
    __syncwarp();  // the staging buffer is rewritten by the next item
    ++n_tc;
  }
}

template <int SF, bool SR>
__global__ void __maxnreg__(kQtMaxRegs) materialize_q8tc_kernel(const __grid_constant__ Params p) {
  static_assert(SF == RSM_I8 || SF == RSM_FP8_E4M3, "one-byte state only");
  static_assert(kQtEpilogueWarps == 4, "epilogue warps cover the four lane quarters");
  extern __shared__ __align__(128) unsigned char smem[];
  if (__ldg(p.active) == -1) return;  // empty active list: one load, then out

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  if (warp == 1) {
    tmem_alloc(sbase + kQtTmemSlot, kQtTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.stages; ++s) {
      mbar_init(sbase + 8u * s, 1u);
      mbar_init(sbase + 8u * kMaxStages + 8u * s, kQtConsumerWarps);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(sbase + kQtMmaDone + 8u * b, 1u);
      mbar_init(sbase + kQtTmemFree + 8u * b, kQtEpilogueWarps);
    }
    mbar_init(sbase + kQtBuildBar, kQtBuilderWarps);
    mbar_init(sbase + kQtExitBar, kQtConsumerWarps);
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kQtTmemSlot);
  // the swizzled operands need 1024-byte aligned atoms: a shared-memory base
  // without that alignment (never seen) ends the CTA with a status bit
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, kQtTmemCols);
    return;
  }
  if (warp == 0) {
    run_loader<SF, RSM_BF16, 64, 128, false, kQtHeads>(p, smem, lane);
  } else {
    if (warp <= kQtBuilderWarps)
      run_builder_qt<SF>(p, smem, warp - 1, lane, tmem);
    else
      run_epilogue_qt<SF, SR>(p, smem, warp - 1 - kQtBuilderWarps, warp, lane, tmem);
    // every consumer warp is done with TMEM before the allocating warp frees it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kQtExitBar);
    if (warp == 1) {
      (void)mbar_wait(sbase + kQtExitBar, 0u, 3ull * kWaitTimeoutNs);
      tc_fence_after();
      tmem_dealloc(tmem, kQtTmemCols);
    }
  }
}

template <int SF, bool SR>
const void* kernel_for_q8tc() {
  return reinterpret_cast<const void*>(&materialize_q8tc_kernel<SF, SR>);
}

}  // namespace rsm
