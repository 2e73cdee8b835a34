// rsm_q8_kernel.cuh -- the materialization kernel for one-byte state (int8 or
// fp8 e4m3 codes with one fp32 scale per (head, dim-row); API page,
// Parameters: state_dtype, state_scale_ptrs; one-byte state is 64 x 128).
//
// A byte of state carries the arithmetic of two bytes of 16-bit state plus a
// row amax, two divisions per row and the byte packing, so this path is bound
// by instruction issue, not by DRAM.  It therefore spreads the per-item work
// (descriptor, decay scan, token conversion, row reduction) over more elements
// per lane than the 16-bit kernel: four consumer warps per CTA, each lane
// owning 8 rows x 8 codes (64 elements), with three CTAs per SM under a
// 128-register cap.  The loader warp, the arena and the slots are the
// materialization kernel's.
//
// Per item, warp cw owns tile rows [16 cw, 16 cw + 16); lane (lr, lc) =
// (lane / 16, lane % 16) owns rows 16 cw + 8 lr + r (r < 8) x columns
// 8 lc .. 8 lc + 7, so that the 16 lanes of a row group hold whole rows and a
// row's amax is a warp reduction.
//
// Two instances: rounding to nearest even, and Philox stochastic rounding
// (template SR), whose Philox words cover 16 consecutive elements of a row:
// the lanes 2m and 2m + 1 of a row group share one call per row, each drawing
// the call of one row of a row pair and trading the two words the other needs.
#pragma once
#include "rsm_kernel.cuh"

namespace rsm {

// 8 codes (fp32 values on the format's grid, or int8 values already holding
// 1.5 * 2^23 + code) -> 8 bytes
template <int SF>
__device__ __forceinline__ uint2 pack_row8(const float2 (&v)[4]) {
  if constexpr (SF == RSM_I8) {
    // the low byte of 1.5 * 2^23 + code is the two's-complement code
    const uint32_t lo = __byte_perm(__byte_perm(__float_as_uint(v[0].x), __float_as_uint(v[0].y), 0x0040u),
                                    __byte_perm(__float_as_uint(v[1].x), __float_as_uint(v[1].y), 0x0040u), 0x5410u);
    const uint32_t hi = __byte_perm(__byte_perm(__float_as_uint(v[2].x), __float_as_uint(v[2].y), 0x0040u),
                                    __byte_perm(__float_as_uint(v[3].x), __float_as_uint(v[3].y), 0x0040u), 0x5410u);
    return make_uint2(lo, hi);
  } else {
    return make_uint2(f32x2_to_e4m3x2(v[0].x, v[0].y) | (f32x2_to_e4m3x2(v[1].x, v[1].y) << 16),
                      f32x2_to_e4m3x2(v[2].x, v[2].y) | (f32x2_to_e4m3x2(v[3].x, v[3].y) << 16));
  }
}

// Packs one row vector and stores its 8 bytes; a row whose qmax/amax (inv) is
// not finite (amax == 0 or tiny) becomes zero codes.
template <int SF>
__device__ __forceinline__ void store_row8(const float2 (&v)[4], float inv, unsigned char* d, bool dst_aligned) {
  uint2 out = pack_row8<SF>(v);
  if (!(inv <= FLT_MAX)) out = make_uint2(0u, 0u);
  if (dst_aligned)
    stg64_stream(d, out);
  else
    store_bytes(d, out);
}

template <int SF, int IF, bool SR>
__device__ __forceinline__ void replay_q8(const Params& p, const unsigned char* sb, const ItemLayout& il,
                                          const ItemDesc* desc, int k, float* wbuf, float* cbuf, int cw, int lane,
                                          uint32_t empty_bar, uint32_t key0, uint32_t key1) {
  constexpr int D = 64, N = 128, IE = In<IF>::bytes;
  constexpr int RPT = 8;            // rows per lane
  constexpr int SLAB = 16;          // rows per warp
  constexpr float qmax = SF == RSM_I8 ? 127.0f : 448.0f;
  static_assert(kQ8WarpBufFloats == kTokChunk * (2 * SLAB + N), "token buffer plan");
  const int lr = lane >> 4, lc = lane & 15;
  const int row0 = SLAB * cw + RPT * lr;  // this lane's first tile row
  float* bbuf = cbuf + kTokChunk * 2 * SLAB;
  const uint32_t flags = desc->flags;
  const bool same_B = (flags & kFlagSameB) != 0u;  // bbuf still holds this item's B rows
  unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
  float* dst_sc = reinterpret_cast<float*>(desc->dst_scale);
  const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
  // the Philox counter words of this item, read before the slot is released
  const uint32_t dst_slot_id = static_cast<uint32_t>(desc->dst_slot);
  const uint32_t layer_id = static_cast<uint32_t>(desc->layer);
  const int head = desc->head;

  const float P = decay_scan(reinterpret_cast<const float*>(sb + il.off_dt), desc->A[0], k, lane, wbuf);

  // this lane's 8 x 8 codes, decoded and multiplied by scale * P
  float2 acc[RPT][4];
  {
    const float* scs = reinterpret_cast<const float*>(sb + il.off_scale) + row0;
    const float4 s0 = *reinterpret_cast<const float4*>(scs);
    const float4 s1 = *reinterpret_cast<const float4*>(scs + 4);
    const float sc[RPT] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const uint2* src = reinterpret_cast<const uint2*>(sb + row0 * N + 8 * lc);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      unpack_vec<SF>(src[r * (N / 8)], acc[r]);
      const float sp = sc[r] * P;
      const float2 sp2 = make_float2(sp, sp);
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[r][u] = __fmul2_rn(acc[r][u], sp2);
    }
  }
  __syncwarp();  // wbuf visible to the whole warp

  // the prefix, kTokChunk tokens at a time: (c, c) pairs of c = w x for the
  // warp's 16 rows and B for all 128 columns in fp32, then one rank-1 update
  // per token with packed fp32x2 FMAs
  const unsigned char* xs = sb + il.off_x;
  const unsigned char* Bs = sb + il.off_B;
  for (int t0 = 0; t0 < k; t0 += kTokChunk) {
    const int tn = min(kTokChunk, k - t0);
    for (int u = lane; u < tn * SLAB; u += 32) {
      const int t = u >> 4, r = u & 15;
      float xv[1];
      load_inputs<IF, 1>(xs + ((t0 + t) * D + SLAB * cw + r) * IE, xv);
      const float c = xv[0] * wbuf[t0 + t];
      *reinterpret_cast<float2*>(cbuf + t * 2 * SLAB + 2 * r) = make_float2(c, c);
    }
    // B: lane column l8's 8 columns as two float4 groups, 64 floats apart, so
    // that eight lanes reading one group read 128 contiguous bytes.  An item of
    // the previous item's B group (one chunk) finds its rows already there.
    if (!same_B)
    for (int u = lane; u < tn * (N / 8); u += 32) {
      const int t = u >> 4, l8 = u & 15;
      float bv[8];
      load_inputs<IF, 8>(Bs + ((t0 + t) * N + 8 * l8) * IE, bv);
      float* d = bbuf + t * N + 4 * l8;
      *reinterpret_cast<float4*>(d) = make_float4(bv[0], bv[1], bv[2], bv[3]);
      *reinterpret_cast<float4*>(d + N / 2) = make_float4(bv[4], bv[5], bv[6], bv[7]);
    }
    __syncwarp();
    if (t0 + kTokChunk >= k) {  // the last chunk: nothing more is read from the slot
      if (lane == 0) mbar_arrive(empty_bar);
    }
    const float* cp = cbuf + 2 * RPT * lr;
    const float* bp = bbuf + 4 * lc;
    // two tokens per pass when rounding to nearest; one with stochastic
    // rounding, whose instance needs the registers (measured on GB300: fp8 SR
    // 18% faster, the nearest-rounding instances unchanged)
    constexpr int kTokUnroll = SR ? 1 : 2;
#pragma unroll kTokUnroll
    for (int t = 0; t < tn; ++t) {
      float2 c2[RPT];
#pragma unroll
      for (int r = 0; r < RPT; r += 2) {
        const float4 v = *reinterpret_cast<const float4*>(cp + t * 2 * SLAB + 2 * r);
        c2[r] = make_float2(v.x, v.y);
        c2[r + 1] = make_float2(v.z, v.w);
      }
      const float4 b0 = *reinterpret_cast<const float4*>(bp + t * N);
      const float4 b1 = *reinterpret_cast<const float4*>(bp + t * N + N / 2);
      const float2 b2[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                            make_float2(b1.z, b1.w)};
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[r][u] = __ffma2_rn(c2[r], b2[u], acc[r][u]);
      }
    }
    __syncwarp();  // the chunk buffers are rewritten by the next chunk
  }

  // requantization: the row amax by a transpose reduction over the 16 lanes of
  // the row group (at each of the first three levels a lane keeps half of its
  // rows and trades the other half with its partner; afterwards lanes 2m and
  // 2m + 1 of the group hold row m), then one division pair per row
  float amax[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    float m0 = fmaxf(fabsf(acc[r][0].x), fabsf(acc[r][0].y));
    float m1 = fmaxf(fabsf(acc[r][1].x), fabsf(acc[r][1].y));
    float m2 = fmaxf(fabsf(acc[r][2].x), fabsf(acc[r][2].y));
    float m3 = fmaxf(fabsf(acc[r][3].x), fabsf(acc[r][3].y));
    amax[r] = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  }
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int half = (RPT >> s) / 2, off = 8 >> s;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? amax[i] : amax[i + half];
      const float keep = upper ? amax[i + half] : amax[i];
      amax[i] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, off));
    }
  }
  const float am = fmaxf(amax[0], __shfl_xor_sync(0xFFFFFFFFu, amax[0], 1));
  const float inv_own = __fdiv_rn(qmax, am);
  const float scale_own = inv_own <= FLT_MAX ? __fdiv_rn(am, qmax) : 0.0f;

  const int group0 = lane & 16;
  if constexpr (SR) {
    // Philox counter (e / 16, dst_slot, layer, 0) with e = (h * D + row) * N +
    // col: one call per 16 columns of a row, the columns of lanes lc and lc ^ 1.
    // For row pair (2q, 2q + 1) the even lane draws row 2q's call and the odd
    // lane row 2q + 1's; words 0, 1 cover the even lane's 8 columns, 2, 3 the
    // odd lane's.  Two row pairs (two Philox chains) at a time.
    const bool odd = (lc & 1) != 0;
#pragma unroll
    for (int q0 = 0; q0 < RPT / 2; q0 += 2) {
      uint4 rw[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int row = row0 + 2 * (q0 + q) + (odd ? 1 : 0);
        rw[q] = make_uint4(static_cast<uint32_t>((head * D + row) * (N / 16) + (lc >> 1)), dst_slot_id, layer_id, 0u);
      }
      philox4x32_n<2>(rw, key0, key1, p.philox_rounds);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t g0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? rw[q].x : rw[q].z, 1);
        const uint32_t g1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? rw[q].y : rw[q].w, 1);
        const uint2 words[2] = {odd ? make_uint2(g0, g1) : make_uint2(rw[q].x, rw[q].y),
                                odd ? make_uint2(rw[q].z, rw[q].w) : make_uint2(g0, g1)};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int r = 2 * (q0 + q) + h2;
          const float inv = __shfl_sync(0xFFFFFFFFu, inv_own, group0 + 2 * r);
          const float2 inv2 = make_float2(inv, inv);
          float2 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) v[u] = __fmul2_rn(acc[r][u], inv2);
          uint2 out;
          if constexpr (SF == RSM_I8) {
            uint32_t ra[4], rb[4];
            sr_r16x4(words[h2].x, ra);
            sr_r16x4(words[h2].y, rb);
            const float2 magic = make_float2(12582912.0f, 12582912.0f);
            float2 c[4] = {make_float2(sr_i8(v[0].x, ra[0]), sr_i8(v[0].y, ra[1])),
                           make_float2(sr_i8(v[1].x, ra[2]), sr_i8(v[1].y, ra[3])),
                           make_float2(sr_i8(v[2].x, rb[0]), sr_i8(v[2].y, rb[1])),
                           make_float2(sr_i8(v[3].x, rb[2]), sr_i8(v[3].y, rb[3]))};
#pragma unroll
            for (int u = 0; u < 4; ++u) c[u] = __fadd2_rn(c[u], magic);
            out = pack_row8<SF>(c);
          } else {
            out = make_uint2(sr_e4m3x4(v[0].x, v[0].y, v[1].x, v[1].y, words[h2].x),
                             sr_e4m3x4(v[2].x, v[2].y, v[3].x, v[3].y, words[h2].y));
          }
          if (!(inv <= FLT_MAX)) out = make_uint2(0u, 0u);
          unsigned char* d = dst_tile + (row0 + r) * N + 8 * lc;
          if (dst_aligned)
            stg64_stream(d, out);
          else
            store_bytes(d, out);
        }
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const float inv = __shfl_sync(0xFFFFFFFFu, inv_own, group0 + 2 * r);
      const float2 inv2 = make_float2(inv, inv);
      float2 v[4];
      if constexpr (SF == RSM_I8) {
        // round to nearest even in one step: fl(v * inv + 1.5 * 2^23) keeps the
        // exact product's rounding to an integer in its low byte (|v * inv| <= 127.5)
        const float2 magic = make_float2(12582912.0f, 12582912.0f);
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ffma2_rn(acc[r][u], inv2, magic);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __fmul2_rn(acc[r][u], inv2);
      }
      store_row8<SF>(v, inv, dst_tile + (row0 + r) * N + 8 * lc, dst_aligned);
    }
  }
  if ((lc & 1) == 0) {
    const int srow = row0 + (lc >> 1);
    if (flags & kFlagScaleAligned) {
      dst_sc[srow] = scale_own;
    } else {
      const unsigned char* vb = reinterpret_cast<const unsigned char*>(&scale_own);
      unsigned char* db = reinterpret_cast<unsigned char*>(dst_sc + srow);
      for (int q = 0; q < 4; ++q) db[q] = vb[q];
    }
  }
}

template <int SF, int IF, bool SR>
__device__ __forceinline__ void run_consumer_q8(const Params& p, unsigned char* smem, int cw, int lane) {
  constexpr int D = 64, N = 128, IE = In<IF>::bytes;
  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8u * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* wbuf = reinterpret_cast<float*>(smem + kWeightOff) + cw * kWeightStride;
  float* cbuf = reinterpret_cast<float*>(smem + kWarpBufOff) + cw * kQ8WarpBufFloats;
  const int tid = cw * 32 + lane;  // 0 .. 127

  uint32_t key0 = 0, key1 = 0;
  if constexpr (SR) {
    const uint64_t s = static_cast<uint64_t>(__ldg(p.rand_seed));
    key0 = static_cast<uint32_t>(s);
    key1 = static_cast<uint32_t>(s >> 32);
  }

  const uint32_t item_max = item_layout(D, N, 1, true, IE, p.W).bytes;
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
    const unsigned char* sb = smem + p.arena0 + off;
    const ItemDesc* desc = reinterpret_cast<const ItemDesc*>(smem + p.desc0) + stage;
    const uint32_t flags = desc->flags;
    if (flags & kFlagEnd) break;
    const int k = desc->k;
    const ItemLayout il = item_layout(D, N, 1, true, IE, k, (flags & kFlagSameB) == 0u);
    arena_head = off + il.bytes;
    const uint32_t empty_bar = empty0 + 8u * stage;

    if (k == 0) {
      // exact copy of the 8 KiB of codes (four 16-byte vectors a thread) and the 64 scales
      unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
      float* dst_sc = reinterpret_cast<float*>(desc->dst_scale);
      const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = reinterpret_cast<const uint4*>(sb)[tid + 128 * q];
      const float scv = tid < D ? reinterpret_cast<const float*>(sb + il.off_scale)[tid] : 0.0f;
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        unsigned char* d = dst_tile + static_cast<uint32_t>(tid + 128 * q) * 16u;
        if (dst_aligned)
          stg128_stream(d, v[q]);
        else
          store_bytes(d, v[q]);
      }
      if (tid < D) {
        if (flags & kFlagScaleAligned) {
          dst_sc[tid] = scv;
        } else {
          const unsigned char* vb = reinterpret_cast<const unsigned char*>(&scv);
          unsigned char* db = reinterpret_cast<unsigned char*>(dst_sc + tid);
          for (int q = 0; q < 4; ++q) db[q] = vb[q];
        }
      }
    } else {
      replay_q8<SF, IF, SR>(p, sb, il, desc, k, wbuf, cbuf, cw, lane, empty_bar, key0, key1);
    }
    if (++stage == p.stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

template <int SF, int IF, bool SR>
__global__ void __maxnreg__(kQ8MaxRegs) materialize_q8_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  // empty active list: one load, then out
  if (__ldg(p.active) == -1) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const uint32_t full0 = smem_addr(smem);
    for (uint32_t s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8u * s, 1u);
      mbar_init(full0 + 8u * kMaxStages + 8u * s, kQ8ConsumerWarps);
    }
    *reinterpret_cast<volatile int*>(smem + kAbortOff) = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0)
    run_loader<SF, IF, 64, 128>(p, smem, lane);
  else
    run_consumer_q8<SF, IF, SR>(p, smem, warp - 1, lane);
}

template <int SF, int IF, bool SR>
const void* q8_kernel() {
  return reinterpret_cast<const void*>(&materialize_q8_kernel<SF, IF, SR>);
}

}  // namespace rsm
