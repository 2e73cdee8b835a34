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
// Stochastic rounding is a separate kernel instance (template SR): its Philox
// work is inline there, and the round-to-nearest instance carries none of it.
#pragma once
#include "rsm_kernel.cuh"

namespace rsm {

// fp8 e4m3 stochastic rounding of |y| >= 2^-6 (or y == 0) on the bit pattern:
// adding the complement of the 16 random bits, scaled to the 20 discarded
// bits, carries into the next grid point exactly when r * 2^4 < the discarded
// bits (the rule of sr_round for a word r << 16); saturates at 448.
__device__ __forceinline__ float sr_e4m3_normal(float y, uint32_t r16) {
  const uint32_t bits = __float_as_uint(y);
  const uint32_t sign = bits & 0x80000000u;
  uint32_t r = ((bits ^ sign) + (((r16 ^ 0xFFFFu) << 4) | 0xFu)) & 0xFFF00000u;
  r = min(r, 0x43E00000u);  // 448
  return __uint_as_float(r | sign);
}

__device__ __forceinline__ bool e4m3_normal_or_zero(float y) {
  const uint32_t ab = __float_as_uint(y) & 0x7FFFFFFFu;
  return ab >= 0x3C800000u || ab == 0u;  // |y| >= 2^-6
}

// int8 stochastic rounding on the integer grid in fp32 arithmetic: lo =
// trunc|y| and the fraction f are exact (|y| < 2^23), and the magnitude goes up
// iff r < f * 2^16 (the rule of sr_round for a word r << 16); saturates at 127.
__device__ __forceinline__ float sr_i8_grid(float y, uint32_t r16) {
  const float a = fabsf(y);
  const float lo = truncf(a);
  const float f = (a - lo) * 65536.0f;
  const float rf = __uint_as_float(0x4B000000u | r16) - 8388608.0f;  // r as fp32, exactly
  const float r = fminf(lo + (rf < f ? 1.0f : 0.0f), 127.0f);
  return copysignf(r, y);
}

// The general fp8 rule for a row vector holding a value below 2^-6 (rare):
// out of line, so that the kernel's code stays small.
struct Row8 {
  float2 v[4];
};
static __device__ __noinline__ Row8 sr_e4m3_row8_general(float2 v0, float2 v1, float2 v2, float2 v3, uint32_t w0,
                                                        uint32_t w1, uint32_t w2, uint32_t w3) {
  Row8 o;
  o.v[0] = make_float2(sr_e4m3(v0.x, sr_lo16(w0)), sr_e4m3(v0.y, sr_hi16(w0)));
  o.v[1] = make_float2(sr_e4m3(v1.x, sr_lo16(w1)), sr_e4m3(v1.y, sr_hi16(w1)));
  o.v[2] = make_float2(sr_e4m3(v2.x, sr_lo16(w2)), sr_e4m3(v2.y, sr_hi16(w2)));
  o.v[3] = make_float2(sr_e4m3(v3.x, sr_lo16(w3)), sr_e4m3(v3.y, sr_hi16(w3)));
  return o;
}

// Stochastic rounding of one row vector of 8 scaled values (its Philox block
// gives 16 random bits per element) to the grid of SF, exactly on the grid.
template <int SF>
__device__ __forceinline__ void sr_row8(float2 (&v)[4], const uint4& rnd) {
  const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  if constexpr (SF == RSM_I8) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = make_float2(sr_i8_grid(v[u].x, w[u] & 0xFFFFu), sr_i8_grid(v[u].y, w[u] >> 16));
  } else {
    bool normal = true;
#pragma unroll
    for (int u = 0; u < 4; ++u) normal = normal && e4m3_normal_or_zero(v[u].x) && e4m3_normal_or_zero(v[u].y);
    if (__all_sync(0xFFFFFFFFu, normal)) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = make_float2(sr_e4m3_normal(v[u].x, w[u] & 0xFFFFu), sr_e4m3_normal(v[u].y, w[u] >> 16));
    } else {  // a value below 2^-6 somewhere in the warp: the general rule (rare)
      const Row8 o = sr_e4m3_row8_general(v[0], v[1], v[2], v[3], w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = o.v[u];
    }
  }
}

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

// Stochastic rounding of this lane's 8 row vectors, kSrRows rows at a time so
// that as many independent Philox chains (one block of 8 elements per row) run
// side by side, in a compact round loop.
constexpr int kSrRows = 2;
template <int SF>
__device__ __forceinline__ void requant_rows_sr(float2 (&acc)[8][4], float inv_own, int group0, uint32_t blk0,
                                                uint32_t slot, uint32_t layer, uint32_t key0, uint32_t key1,
                                                int rounds, unsigned char* dst_tile, int row0, int lc,
                                                bool dst_aligned) {
  constexpr int N = 128;
#pragma unroll
  for (int r0 = 0; r0 < 8; r0 += kSrRows) {
    uint4 rnd[kSrRows];
#pragma unroll
    for (int q = 0; q < kSrRows; ++q) rnd[q] = make_uint4(blk0 + (r0 + q) * (N / 8), slot, layer, 0u);
    philox4x32_xc<kSrRows>(rnd, key0, key1, rounds);
#pragma unroll
    for (int q = 0; q < kSrRows; ++q) {
      const int r = r0 + q;
      const float inv = __shfl_sync(0xFFFFFFFFu, inv_own, group0 + 2 * r);
      const float2 inv2 = make_float2(inv, inv);
      float2 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __fmul2_rn(acc[r][u], inv2);
      sr_row8<SF>(v, rnd[q]);
      if constexpr (SF == RSM_I8) {
        const float2 magic = make_float2(12582912.0f, 12582912.0f);
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __fadd2_rn(v[u], magic);
      }
      store_row8<SF>(v, inv, dst_tile + (row0 + r) * N + 8 * lc, dst_aligned);
    }
  }
}

template <int SF, int IF, bool SR>
__device__ __forceinline__ void replay_q8(const Params& p, const unsigned char* sb, const ItemLayout& il,
                                          const ItemDesc* desc, int k, float* wbuf, float* cbuf, int cw, int lane,
                                          uint32_t empty_bar, uint32_t key0, uint32_t key1) {
  constexpr int D = 64, N = 128, IE = In<IF>::bytes;
  constexpr int RPT = 8;            // rows per lane
  constexpr int SLAB = 16;          // rows per warp
  constexpr float qmax = SF == RSM_I8 ? 127.0f : 448.0f;
  static_assert(warp_buf_floats(D, N, 1, kQ8ConsumerWarps) == kTokChunk * (2 * SLAB + N), "token buffer plan");
  const int lr = lane >> 4, lc = lane & 15;
  const int row0 = SLAB * cw + RPT * lr;  // this lane's first tile row
  float* bbuf = cbuf + kTokChunk * 2 * SLAB;
  const uint32_t flags = desc->flags;
  unsigned char* dst_tile = reinterpret_cast<unsigned char*>(desc->dst_state);
  float* dst_sc = reinterpret_cast<float*>(desc->dst_scale);
  const bool dst_aligned = (flags & kFlagDstAligned) != 0u;
  // everything else the item needs from its descriptor, read before the slot is released
  const uint32_t dst_slot_id = static_cast<uint32_t>(desc->dst_slot);
  const uint32_t layer_id = static_cast<uint32_t>(desc->layer);
  // Philox block of this lane's first row vector: element (h * D + row) * N + 8 lc, over 8
  const uint32_t blk0 = static_cast<uint32_t>((static_cast<int64_t>(desc->head) * D + row0) * (N / 8) + lc);

  const float P = decay_scan(reinterpret_cast<const float*>(sb + il.off_dt), desc->A, k, lane, wbuf);

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
    // that eight lanes reading one group read 128 contiguous bytes
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
#pragma unroll 2
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
    requant_rows_sr<SF>(acc, inv_own, group0, blk0, dst_slot_id, layer_id, key0, key1, p.philox_rounds, dst_tile,
                        row0, lc, dst_aligned);
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
  float* cbuf = reinterpret_cast<float*>(smem + kWarpBufOff) + cw * warp_buf_floats(D, N, 1, kQ8ConsumerWarps);
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
    const ItemLayout il = item_layout(D, N, 1, true, IE, k);
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

// One-byte state with stochastic rounding: the eight-warp kernel, whose two
// CTAs per SM keep more Philox chains in flight than the four-warp one.
template <int SF, int IF, int D, int N>
const void* kernel_for_sr() {
  static_assert(Fmt<SF>::quant && D == 64 && N == 128, "the stochastic-rounding instance is one-byte state");
  return reinterpret_cast<const void*>(&materialize_kernel<SF, IF, D, N>);
}

}  // namespace rsm
