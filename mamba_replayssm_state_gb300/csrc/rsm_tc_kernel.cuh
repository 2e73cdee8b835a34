// rsm_tc_kernel.cuh -- the long-window variant of the materialization kernel:
// the replayed prefix applied as a dense contraction on the tensor cores.
//
// In closed form a head's replay is S_k = P * S_0 + C B with C[i][t] =
// w_t x_t[i] (64 x k) and B[t][j] = B_t[j] (k x 128): a rank-k update, worth
// the tensor cores for long prefixes.  The accumulator is S^T - P S_0^T in
// TMEM: M = 128 dstate columns (TMEM lanes) x N = 64 dim rows (columns).
//
// The loader warp, the arena and the slots are the materialization kernel's.
// The seven consumer warps form two groups that work on consecutive items at
// the same time:
//   builder group (warps 1-3): decay weights of the item's tokens, the MMA
//     operands in shared memory, MN-major with the 128-byte swizzle, so that
//     a ring row is a row of the operand (A = B^T: 128 x k_pad, the bf16 ring
//     rows of B copied exactly, rebuilt only for the first head of a B group;
//     the second operand C^T: 64 x k_pad, w_t x_t rounded to bf16, or for
//     fp16 state split into two bf16 operands hi + lo), 16 bytes
//     a thread at a time, then one thread issues ceil(k/16) tcgen05.mma
//     (K = 16) into one of two TMEM accumulators and commits them to that
//     accumulator's mbarrier.  (K-major operands had each 16-byte chunk
//     gathered from 8 rows; that build was the kernel's critical path);
//   epilogue group (warps 4-7): the item's S_0 column (one dstate column j per
//     thread, all 64 dim rows) into registers, the slot released, then after
//     the MMA the accumulator column read from TMEM lane j, P S_0 added,
//     rounded and stored straight to global memory (a warp writes 64
//     contiguous bytes per tile row), and the accumulator handed back.
//     (Writing the result over S_0 in shared memory and storing the tile with
//     one bulk copy measured slower at every prefix length: the slot then
//     stays taken until the copy has read it.)
// With two accumulators the builder prepares item n+1 while the epilogue
// drains item n.  Operands are single-buffered: the builder writes them only
// after the previous MMA has completed.  Copies (prefix 0) are done by the
// epilogue group alone.
// Every wait is an mbarrier wait bounded in wall time, every exit decision is
// warp-uniform (the tcgen05 loads, allocation and deallocation are warp-wide),
// and TMEM (128 columns) is allocated by warp 1 before the loop and freed by it
// after an exit barrier.
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

__device__ __forceinline__ void stg32_stream(void* p, uint32_t v) {
  asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int SF>
__device__ __forceinline__ uint32_t from_f32_16(float v) {
  // round to nearest even (values already rounded stochastically stay exact)
  return SF == RSM_BF16 ? (pack_bf16x2(v, 0.0f) & 0xFFFFu) : (pack_f16x2(v, 0.0f) & 0xFFFFu);
}

// The epilogue for stochastic rounding or a misaligned destination, out of
// line (rare paths): S = P S_0 + acc for this thread's column j, with S_0 read
// from the item's tile in shared memory.
template <int SF>
__device__ __noinline__ void tc_epilogue_general(int philox_rounds, uint32_t taddr, bool split_n, const uint16_t* s0_col,
                                                 float P, unsigned char* out_col, bool dst_aligned, bool sr, int h,
                                                 int j, uint32_t dst_slot_id, uint32_t layer_id, uint32_t key0,
                                                 uint32_t key1) {
  constexpr int D = 64, N = 128;
#pragma unroll 1
  for (int part = 0; part < D / 16; ++part) {
    float acc[16];
    tmem_ld16(taddr + 16u * part, acc);
    if (split_n) {  // hi and lo products in the accumulator's two halves
      float lo16[16];
      tmem_ld16(taddr + kTcLoCols + 16u * part, lo16);
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] += lo16[c];
    }
#pragma unroll 1
    for (int c = 0; c < 16; ++c) {
      const int i = 16 * part + c;
      const float y = fmaf(P, to_f32_16<SF>(s0_col[i * N]), acc[c]);
      uint32_t v;
      if (sr) {
        // element e's 16 bits: the low (e even) or high half of word (e >> 1) & 3
        // of call e >> 3, given to the conversion as the random bits of its low result
        const int64_t e = (static_cast<int64_t>(h) * D + i) * N + j;
        const uint4 rnd =
            philox4x32(make_uint4(static_cast<uint32_t>(e >> 3), dst_slot_id, layer_id, 0u), key0, key1, philox_rounds);
        const int q = static_cast<int>((e >> 1) & 3);
        const uint32_t wsel = q == 0 ? rnd.x : q == 1 ? rnd.y : q == 2 ? rnd.z : rnd.w;
        v = sr_pack2<SF>(y, 0.0f, (e & 1) ? (wsel >> 16) : (wsel & 0xFFFFu)) & 0xFFFFu;
      } else {
        v = from_f32_16<SF>(y);
      }
      unsigned char* q = out_col + static_cast<uint32_t>(i) * (N * 2u);
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
__device__ __forceinline__ void run_builder_tc(const Params& p, unsigned char* smem, int bw, int lane, uint32_t tmem) {
  constexpr int D = 64, N = 128, ES = 2, IE = 2;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* wbuf = reinterpret_cast<float*>(smem + kWeightOff) + bw * kWeightStride;
  constexpr bool kSplit = tc_split_c(SF);
  constexpr uint32_t kCGroup = tc_c_group(SF);  // bytes between token groups of C^T
  unsigned char* aop = smem + tc_a_off(SF);
  unsigned char* bop = smem + kTcBOff;
  const int tid = bw * 32 + lane;  // over the builder group
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 64, true, true);
  constexpr uint32_t kIdescN128 = idesc_bf16_f32(128, 128, true, true);

  uint32_t arena_head = 0;
  uint32_t stage = 0, phase = 0;
  uint32_t n_tc = 0;  // tensor-core items so far
  int c_dirty = kTcKMax;  // leading token rows of C^T (and C_lo^T) that may hold nonzero values
  for (;;) {
    if (!tc_wait(full0 + 8u * stage, phase, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = __shfl_sync(0xFFFFFFFFu, desc->flags, 0);
    if (flags & kFlagEnd) break;
    const int k = __shfl_sync(0xFFFFFFFFu, desc->k, 0);
    const bool same_B = (flags & kFlagSameB) != 0u;  // the A operand of the previous item still holds
    const ItemLayout il = item_layout(D, N, ES, false, IE, k, !same_B);
    const uint32_t off = arena_next(arena_head, il.bytes, p.arena_bytes);  // the loader's exact-fit placement
    const unsigned char* sb = smem + p.arena0 + off;
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
    // decay weights w_t of the item's tokens, once per warp
    (void)decay_scan(reinterpret_cast<const float*>(sb + il.off_dt), desc->A[0], k, lane, wbuf);
    __syncwarp();  // wbuf visible to the whole warp
    // the operands are free once the previous item's MMAs have completed
    if (n_tc > 0 && !tc_wait(sbase + kTcMmaDone + 8u * ((n_tc - 1) & 1u), ((n_tc - 1) >> 1) & 1u, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    const int kp = (k + 15) & ~15;  // K padded to whole MMAs; tokens k .. kp-1 are zero
    constexpr int kStep = 32 * kTcBuilderWarps;
    if (!same_B) {
      // A = B^T: token t's 256-byte B row is row t % 8 of atom column c / 8 of
      // token group t / 8; chunk c % 8 goes to chunk (c % 8) ^ (t % 8)
      for (int u = tid; u < kp * 16; u += kStep) {
        const int t = u >> 4, c = u & 15;
        const uint4 v = t < k ? *reinterpret_cast<const uint4*>(sb + il.off_B + t * (N * 2) + c * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(aop + (t >> 3) * kTcAGroup + (c >> 3) * 1024 + (t & 7) * 128 +
                                  (((c & 7) ^ (t & 7)) << 4)) = v;
      }
    }
    // C^T = (w x)^T: token t's 128-byte row w_t x_t, chunk c to chunk c ^ (t % 8);
    // two chunks a thread at a time, both loaded before either is converted.
    // Rows k .. kq-1 must be zero: only those a longer item left nonzero are
    // cleared (rows past kq are not read by this item's MMAs)
    const int kq = kSplit && k <= 8 ? 8 : kp;  // token rows the MMAs read
    const int rows = max(k, min(c_dirty, kq));
    c_dirty = c_dirty > kq ? c_dirty : k;
    const int n_chunks = rows * 8;
    for (int u0 = tid; u0 < n_chunks; u0 += 2 * kStep) {
      uint4 xv[2];
      float wt[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int u = u0 + r * kStep, t = u >> 3, c = u & 7;
        xv[r] = make_uint4(0u, 0u, 0u, 0u);
        wt[r] = 0.0f;
        if (u < n_chunks && t < k) {
          xv[r] = *reinterpret_cast<const uint4*>(sb + il.off_x + t * (D * 2) + c * 16);
          wt[r] = wbuf[t];
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int u = u0 + r * kStep, t = u >> 3, c = u & 7;
        if (u >= n_chunks) break;
        const uint32_t at = (t >> 3) * kCGroup + (t & 7) * 128 + ((c ^ (t & 7)) << 4);
        const uint32_t xw[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
        const float2 w2 = make_float2(wt[r], wt[r]);
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 cc = __fmul2_rn(make_float2(bf16lo(xw[q]), bf16hi(xw[q])), w2);
          if constexpr (kSplit) {
            // hi = c with its low 16 bits cleared (a bf16 value), lo = c - hi
            // (exact) rounded to bf16: hi + lo is w x within 2^-16 relative
            const uint32_t c0 = __float_as_uint(cc.x), c1 = __float_as_uint(cc.y);
            hw[q] = __byte_perm(c0, c1, 0x7632u);
            const float2 ll = __ffma2_rn(make_float2(__uint_as_float(c0 & 0xFFFF0000u), __uint_as_float(c1 & 0xFFFF0000u)),
                                         make_float2(-1.0f, -1.0f), cc);
            lw[q] = pack_bf16x2(ll.x, ll.y);
          } else {
            hw[q] = pack_bf16x2(cc.x, cc.y);
          }
        }
        *reinterpret_cast<uint4*>(bop + at) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if constexpr (kSplit) *reinterpret_cast<uint4*>(bop + at + 1024) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    fence_proxy_async_smem();  // the operands, written by this thread, before the tensor cores read them
    // the group is done with the slot's x, B and dt
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);
    // every builder warp has written its share of the operands
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcBuildBar);
    if (!tc_wait(sbase + kTcBuildBar, n_tc & 1u, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    tc_fence_after();
    const uint32_t buf = n_tc & 1u;
    if (bw == 0) {
      // the accumulator is free once the epilogue has read it (two items back)
      const bool ok = n_tc < 2 || tc_wait(sbase + kTcTmemFree + 8u * buf, ((n_tc - 2) >> 1) & 1u, abort_flag);
      if (!ok) {
        tc_give_up(p, abort_flag, lane);
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t bdesc0 = smem_desc_mn_sw128(sbase + kTcBOff, 1024u, 1024u);
        if (kSplit && k <= 8) {
          // one MMA: K rows 0-7 of C^T are the tokens' hi rows and 8-15 their
          // lo rows, against the eight A rows read twice (K stride 0); the
          // start address field counts 16-byte units
          tc_mma_bf16(tmem + buf * kTcAccCols, smem_desc_mn_sw128(sbase + tc_a_off(SF), 1024u, 0u), bdesc0, kIdesc,
                      0u);
        } else if (kSplit) {
          // one MMA of N = 128 per 16 tokens: C^T as 128 rows (hi, then lo)
          const uint64_t adesc0 = smem_desc_mn_sw128(sbase + tc_a_off(SF), 1024u, kTcAGroup);
          const uint64_t cdesc0 = smem_desc_mn_sw128(sbase + kTcBOff, 1024u, kCGroup);
          for (int kc = 0; kc < kp / 16; ++kc)
            tc_mma_bf16(tmem + buf * kTcAccCols, adesc0 + static_cast<uint64_t>(kc * 2 * kTcAGroup / 16),
                        cdesc0 + static_cast<uint64_t>(kc * 2 * kCGroup / 16), kIdescN128, kc > 0 ? 1u : 0u);
        } else {
          // one MMA per 16 tokens, i.e. per two token groups
          const uint64_t adesc0 = smem_desc_mn_sw128(sbase + tc_a_off(SF), 1024u, kTcAGroup);
          for (int kc = 0; kc < kp / 16; ++kc)
            tc_mma_bf16(tmem + buf * kTcAccCols, adesc0 + static_cast<uint64_t>(kc * 2 * kTcAGroup / 16),
                        bdesc0 + static_cast<uint64_t>(kc * 2 * kCGroup / 16), kIdesc, kc > 0 ? 1u : 0u);
        }
        tc_commit(sbase + kTcMmaDone + 8u * buf);
      }
      __syncwarp();
    }
    ++n_tc;
  }
}

template <int SF>
__device__ __forceinline__ void run_epilogue_tc(const Params& p, unsigned char* smem, int ew, int warp, int lane,
                                                uint32_t tmem) {
  constexpr int D = 64, N = 128, ES = 2, IE = 2;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* wbuf = reinterpret_cast<float*>(smem + kWeightOff) + (kTcBuilderWarps + ew) * kWeightStride;
  const int tid = ew * 32 + lane;   // 0 .. 127 over the epilogue group
  const int quarter = warp & 3;     // TMEM lane quarter this warp may access (CTA warp id % 4)
  const int j = 32 * quarter + lane;  // this thread's dstate column = its TMEM lane

  uint32_t key0 = 0, key1 = 0;
  const bool sr = p.philox_rounds > 0;
  if (sr) {
    const uint64_t s = static_cast<uint64_t>(__ldg(p.rand_seed));
    key0 = static_cast<uint32_t>(s);
    key1 = static_cast<uint32_t>(s >> 32);
  }
  uint32_t arena_head = 0;
  uint32_t stage = 0, phase = 0;
  uint32_t n_tc = 0;
  for (;;) {
    if (!tc_wait(full0 + 8u * stage, phase, abort_flag)) {
      tc_give_up(p, abort_flag, lane);
      break;
    }
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = __shfl_sync(0xFFFFFFFFu, desc->flags, 0);
    if (flags & kFlagEnd) break;
    const int k = __shfl_sync(0xFFFFFFFFu, desc->k, 0);
    const bool same_B = (flags & kFlagSameB) != 0u;
    const ItemLayout il = item_layout(D, N, ES, false, IE, k, !same_B);
    const uint32_t off = arena_next(arena_head, il.bytes, p.arena_bytes);  // the loader's exact-fit placement
    const unsigned char* sb = smem + p.arena0 + off;
    arena_head = off + il.bytes;
    unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
    const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
    const uint32_t empty_bar = empty0 + 8u * stage;
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }

    if (k == 0) {
      // exact copy of the source tile: 1024 vectors of 16 bytes over 128 threads
      uint4 v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) v[r] = reinterpret_cast<const uint4*>(sb)[tid + 128 * r];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const uint32_t o = static_cast<uint32_t>(tid + 128 * r) * 16u;
        if (dst_aligned) {
          stg128_stream(dst_tile + o, v[r]);
        } else {
          const unsigned char* b = reinterpret_cast<const unsigned char*>(&v[r]);
          for (int q = 0; q < 16; ++q) dst_tile[o + q] = b[q];
        }
      }
      continue;
    }

    const int h = desc->head;
    const uint32_t dst_slot_id = static_cast<uint32_t>(desc->dst_slot);
    const uint32_t layer_id = static_cast<uint32_t>(desc->layer);
    const float P = decay_scan(reinterpret_cast<const float*>(sb + il.off_dt), desc->A[0], k, lane, wbuf);
    const uint32_t buf = n_tc & 1u;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + buf * kTcAccCols;
    const bool split_n = tc_split_c(SF) && k > 8;  // the accumulator's halves hold hi and lo
    unsigned char* out_col = dst_tile + static_cast<uint32_t>(j) * 2u;
    const uint16_t* s0_col = reinterpret_cast<const uint16_t*>(sb) + j;
    if (!sr && dst_aligned) {
      // Columns in pairs: lanes 2m and 2m + 1 own columns j and j ^ 1 (TMEM
      // lanes); of each row pair (i, i + 1) the even lane writes row i and the
      // odd lane row i + 1, both columns, after trading one accumulator value.
      const bool odd = (lane & 1) != 0;
      const int jp = j & ~1;
      // S_0 of the column pair at this lane's rows 2c + odd, as 16-bit pairs;
      // then the slot goes back to the loader while the MMA runs
      const uint32_t* s0p = reinterpret_cast<const uint32_t*>(sb) + jp / 2;
      uint32_t s0[D / 2];
#pragma unroll
      for (int c = 0; c < D / 2; ++c) s0[c] = s0p[(2 * c + (odd ? 1 : 0)) * (N / 2)];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
      if (!tc_wait(sbase + kTcMmaDone + 8u * buf, (n_tc >> 1) & 1u, abort_flag)) {
        tc_give_up(p, abort_flag, lane);
        break;
      }
      tc_fence_after();
      unsigned char* out_pair = dst_tile + static_cast<uint32_t>(jp) * 2u + (odd ? N * 2u : 0u);
#pragma unroll
      for (int part = 0; part < D / 16; ++part) {
        float acc[16];
        tmem_ld16(taddr + 16u * part, acc);
        if (split_n) {  // hi and lo products in the two halves
          float lo16[16];
          tmem_ld16(taddr + kTcLoCols + 16u * part, lo16);
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            const float2 a2 = __fadd2_rn(make_float2(acc[c], acc[c + 1]), make_float2(lo16[c], lo16[c + 1]));
            acc[c] = a2.x;
            acc[c + 1] = a2.y;
          }
        }
#pragma unroll
        for (int c2 = 0; c2 < 8; ++c2) {
          const float a0 = acc[2 * c2], a1 = acc[2 * c2 + 1];
          const float recv = __shfl_xor_sync(0xFFFFFFFFu, odd ? a0 : a1, 1);
          const float lo = odd ? recv : a0, hi = odd ? a1 : recv;
          const uint32_t sp = s0[8 * part + c2];
          const float x0 = to_f32_16<SF>(sp & 0xFFFFu), x1 = to_f32_16<SF>(sp >> 16);
          const float y0 = fmaf(P, x0, lo), y1 = fmaf(P, x1, hi);
          const uint32_t w = SF == RSM_BF16 ? pack_bf16x2(y0, y1) : pack_f16x2(y0, y1);
          stg32_stream(out_pair + static_cast<uint32_t>(16 * part + 2 * c2) * (N * 2u), w);
        }
      }
    } else {
      // stochastic rounding or a misaligned destination: S_0 read from the
      // slot during the epilogue, which releases the slot afterwards
      if (!tc_wait(sbase + kTcMmaDone + 8u * buf, (n_tc >> 1) & 1u, abort_flag)) {
        tc_give_up(p, abort_flag, lane);
        break;
      }
      tc_fence_after();
      tc_epilogue_general<SF>(p.philox_rounds, taddr, split_n, s0_col, P, out_col, dst_aligned, sr, h, j,
                              dst_slot_id, layer_id, key0, key1);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    // the accumulator goes back to the builder group
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcTmemFree + 8u * buf);
    ++n_tc;
  }
}

template <int SF>
__global__ void __launch_bounds__(kTcThreads, 2) materialize_tc_kernel(const __grid_constant__ Params p) {
  static_assert(SF == RSM_BF16 || SF == RSM_F16, "16-bit state only");
  static_assert(kTcEpilogueWarps == 4 && (1 + kTcBuilderWarps) % 4 == 0, "epilogue warps cover the four lane quarters");
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
      mbar_init(sbase + 8u * kMaxStages + 8u * s, kTcConsumerWarps);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(sbase + kTcMmaDone + 8u * b, 1u);
      mbar_init(sbase + kTcTmemFree + 8u * b, kTcEpilogueWarps);
    }
    mbar_init(sbase + kTcBuildBar, kTcBuilderWarps);
    mbar_init(sbase + kTcExitBar, kTcConsumerWarps);
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTcTmemSlot);
  // the swizzled operands need 1024-byte aligned atoms: a shared-memory base
  // without that alignment (never seen) ends the CTA with a status bit
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) flag_status(p.status, RSM_STATUS_WAIT_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, kTcTmemCols);
    return;
  }
  if (warp == 0) {
    run_loader<SF, RSM_BF16, 64, 128, true, 1, true>(p, smem, lane);
  } else {
    if (warp <= kTcBuilderWarps)
      run_builder_tc<SF>(p, smem, warp - 1, lane, tmem);
    else
      run_epilogue_tc<SF>(p, smem, warp - 1 - kTcBuilderWarps, warp, lane, tmem);
    // every consumer warp is done with TMEM (the epilogue waited for every MMA
    // it reads) before the allocating warp frees it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbase + kTcExitBar);
    if (warp == 1) {
      (void)mbar_wait(sbase + kTcExitBar, 0u, 3ull * kWaitTimeoutNs);
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
