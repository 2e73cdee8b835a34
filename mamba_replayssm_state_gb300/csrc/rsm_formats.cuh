// rsm_formats.cuh -- device-side state/input element formats: 16-byte vector
// unpack to fp32, fp32 pack with round-to-nearest-even or stochastic rounding,
// and the Philox-4x32 generator that drives stochastic rounding.
//
// Conversions use the hardware cvt instructions (exact for decoding; RNE with
// IEEE overflow for bf16/fp16, RNE-satfinite for fp8 e4m3).  Stochastic
// rounding is integer arithmetic on the fp32 bit pattern and takes exactly
// the decision "round the magnitude up iff word < frac * 2^32", frac being the
// distance to the lower grid neighbour over the grid spacing.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "../../include/replayssm.h"

namespace rsm {

template <int F> struct Fmt;
template <> struct Fmt<RSM_F32> { static constexpr int bytes = 4; static constexpr bool quant = false; };
template <> struct Fmt<RSM_BF16> { static constexpr int bytes = 2; static constexpr bool quant = false; };
template <> struct Fmt<RSM_F16> { static constexpr int bytes = 2; static constexpr bool quant = false; };
template <> struct Fmt<RSM_I8> { static constexpr int bytes = 1; static constexpr bool quant = true; };
template <> struct Fmt<RSM_FP8_E4M3> { static constexpr int bytes = 1; static constexpr bool quant = true; };

// ---------------------------------------------------------------------------
// scalar helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float2 f16x2_to_f32(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// two e4m3 codes (in the low 16 bits) -> two fp32 values, exactly
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t codes16) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(codes16));
  return f16x2_to_f32(h2);
}

// two fp32 -> two e4m3 codes (low 16 bits), round to nearest even, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n\tcvt.u32.u16 %0, c;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// Philox-4x32 (Salmon, Moraes, Dror, Shaw, SC'11, section 5.2)
// ---------------------------------------------------------------------------

// R rounds, unrolled (the key schedule folds into constants)
template <int R>
__device__ __forceinline__ uint4 philox4x32_r(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    // one 32x32 -> 64-bit multiply gives both halves of each product
    const uint64_t pA = static_cast<uint64_t>(kMulA) * c.x;
    const uint64_t pB = static_cast<uint64_t>(kMulB) * c.z;
    c = make_uint4(static_cast<uint32_t>(pB >> 32) ^ c.y ^ (k0 + r * kWeylA), static_cast<uint32_t>(pB),
                   static_cast<uint32_t>(pA >> 32) ^ c.w ^ (k1 + r * kWeylB), static_cast<uint32_t>(pA));
  }
  return c;
}

__device__ __forceinline__ uint4 philox4x32(uint4 c, uint32_t k0, uint32_t k1, int rounds) {
  if (rounds == 10) return philox4x32_r<10>(c, k0, k1);  // the usual round count, unrolled
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
  for (int r = 0; r < rounds; ++r) {
    if (r > 0) {
      k0 += kWeylA;
      k1 += kWeylB;
    }
    const uint64_t pA = static_cast<uint64_t>(kMulA) * c.x;
    const uint64_t pB = static_cast<uint64_t>(kMulB) * c.z;
    c = make_uint4(static_cast<uint32_t>(pB >> 32) ^ c.y ^ k0, static_cast<uint32_t>(pB),
                   static_cast<uint32_t>(pA >> 32) ^ c.w ^ k1, static_cast<uint32_t>(pA));
  }
  return c;
}

// C independent counters through `rounds` rounds side by side (the usual
// 10 unrolled, so that the chains interleave).
template <int C>
__device__ __forceinline__ void philox4x32_n(uint4 (&c)[C], uint32_t k0, uint32_t k1, int rounds) {
  if (rounds == 10) {
#pragma unroll
    for (int q = 0; q < C; ++q) c[q] = philox4x32_r<10>(c[q], k0, k1);
    return;
  }
#pragma unroll
  for (int q = 0; q < C; ++q) c[q] = philox4x32(c[q], k0, k1, rounds);
}

// ---------------------------------------------------------------------------
// stochastic rounding
// ---------------------------------------------------------------------------
// An element's magnitude goes up to the next grid point iff the top 16 bits of
// its discarded part plus its 16-bit random number carry past 2^16; the
// result saturates to the largest finite value (infinity too) and keeps its
// sign.  bf16, f16 and fp8 e4m3 take the decision in the conversion
// instruction with stochastic rounding (cvt.rs, sm_100 family), which reads
// one 32-bit word of random bits per two 16-bit or four fp8 results:
//   bf16x2 / f16x2: the low result with rbits[15:0], the high with
//     rbits[31:16] (f16 compares their low 13 bits with its 13 discarded bits);
//   e4m3x4: byte 0 with rbits[15:0], byte 1 with rbits[15:0] bit-reversed,
//     byte 2 with rbits[31:16], byte 3 with rbits[31:16] bit-reversed.
__device__ __forceinline__ uint32_t sr_bf16x2(float lo, float hi, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.satfinite.bf16x2.f32 %0, %1, %2, %3;" : "=r"(d) : "f"(hi), "f"(lo), "r"(rbits));
  return d;
}
__device__ __forceinline__ uint32_t sr_f16x2(float lo, float hi, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.satfinite.f16x2.f32 %0, %1, %2, %3;" : "=r"(d) : "f"(hi), "f"(lo), "r"(rbits));
  return d;
}
// four values, v0 in byte 0
__device__ __forceinline__ uint32_t sr_e4m3x4(float v0, float v1, float v2, float v3, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.satfinite.e4m3x4.f32 %0, {%1, %2, %3, %4}, %5;" : "=r"(d) : "f"(v3), "f"(v2), "f"(v1), "f"(v0), "r"(rbits));
  return d;
}
// two 16-bit state values, `lo` in the low half
template <int F>
__device__ __forceinline__ uint32_t sr_pack2(float lo, float hi, uint32_t rbits) {
  static_assert(F == RSM_BF16 || F == RSM_F16, "16-bit state");
  if constexpr (F == RSM_BF16) return sr_bf16x2(lo, hi, rbits);
  else return sr_f16x2(lo, hi, rbits);
}

// int8 on the integer grid, in fp32: |y| - trunc|y| and its scaling by 2^16
// are exact (|y| < 2^23), and so is the floor that keeps the top 16 bits.
__device__ __forceinline__ float sr_i8(float y, uint32_t r16) {
  const float a = fabsf(y);
  const float lo = truncf(a);
  const float d16 = floorf((a - lo) * 65536.0f);
  const float r = __uint_as_float(0x4B000000u | r16) - 8388608.0f;  // r16 as fp32, exactly
  const float q = fminf(lo + (d16 + r >= 65536.0f ? 1.0f : 0.0f), 127.0f);
  return copysignf(q, y);
}

// The random numbers of four one-byte elements from their word: lo16,
// lo16 reversed, hi16, hi16 reversed (the e4m3x4 assignment).
__device__ __forceinline__ void sr_r16x4(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t rv = __brev(w);
  r[0] = w & 0xFFFFu;
  r[1] = rv >> 16;
  r[2] = w >> 16;
  r[3] = rv & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// vectors of state elements: a thread moves one vector per tile row, 16 bytes
// for 4- and 2-byte formats and 8 bytes (8 codes) for one-byte formats
// ---------------------------------------------------------------------------

template <int F>
struct Vec {
  static constexpr int N = Fmt<F>::bytes == 1 ? 8 : 16 / Fmt<F>::bytes;  // elements
  static constexpr int BYTES = N * Fmt<F>::bytes;
  static constexpr int WORDS = BYTES / 4;
  using Raw = typename std::conditional<BYTES == 16, uint4, uint2>::type;
};

template <int F>
__device__ __forceinline__ void raw_words(const typename Vec<F>::Raw& r, uint32_t* w) {
  if constexpr (Vec<F>::BYTES == 16) {
    w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
  } else {
    w[0] = r.x; w[1] = r.y;
  }
}

template <int F>
__device__ __forceinline__ typename Vec<F>::Raw words_raw(const uint32_t* w) {
  if constexpr (Vec<F>::BYTES == 16) return make_uint4(w[0], w[1], w[2], w[3]);
  else return make_uint2(w[0], w[1]);
}

// raw words -> fp32 values (one-byte formats: codes only; the caller scales)
template <int F, int NW>
__device__ __forceinline__ void unpack_words(const uint32_t* w, float* v) {
  if constexpr (F == RSM_F32) {
#pragma unroll
    for (int q = 0; q < NW; ++q) v[q] = __uint_as_float(w[q]);
  } else if constexpr (F == RSM_BF16) {
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      v[2 * q] = bf16lo(w[q]);
      v[2 * q + 1] = bf16hi(w[q]);
    }
  } else if constexpr (F == RSM_F16) {
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const float2 f = f16x2_to_f32(w[q]);
      v[2 * q] = f.x;
      v[2 * q + 1] = f.y;
    }
  } else if constexpr (F == RSM_I8) {
    // int8 -> fp32 exactly on the integer pipes: flip the sign bit so that each
    // byte holds code + 128, place it in the mantissa of 2^23 (0x4B0000xx) and
    // subtract 2^23 + 128 (two values per packed add).
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const uint32_t u = w[q] ^ 0x80808080u;
#pragma unroll
      for (int b = 0; b < 4; b += 2) {
        const float2 d = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u + b)),
                                                __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541u + b))),
                                    bias);
        v[4 * q + b] = d.x;
        v[4 * q + b + 1] = d.y;
      }
    }
  } else {  // FP8 e4m3
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const float2 a = e4m3x2_to_f32(w[q] & 0xFFFFu);
      const float2 b = e4m3x2_to_f32(w[q] >> 16);
      v[4 * q + 0] = a.x;
      v[4 * q + 1] = a.y;
      v[4 * q + 2] = b.x;
      v[4 * q + 3] = b.y;
    }
  }
}

// fp32 values (already scaled into code units for one-byte formats) -> raw
// words, round to nearest even (saturating for one-byte formats)
template <int F, int NW>
__device__ __forceinline__ void pack_words_rne(const float* v, uint32_t* w) {
  if constexpr (F == RSM_F32) {
#pragma unroll
    for (int q = 0; q < NW; ++q) w[q] = __float_as_uint(v[q]);
  } else if constexpr (F == RSM_BF16) {
#pragma unroll
    for (int q = 0; q < NW; ++q) w[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
  } else if constexpr (F == RSM_F16) {
#pragma unroll
    for (int q = 0; q < NW; ++q) w[q] = pack_f16x2(v[2 * q], v[2 * q + 1]);
  } else if constexpr (F == RSM_I8) {
    // round to nearest even by adding 1.5 * 2^23: the sum's low byte is the
    // two's-complement code.  No clamp is needed: |v| <= amax, so
    // |v * fl(127/amax)| < 127.5 and the code lies in [-127, 127].
    const float2 magic = make_float2(12582912.0f, 12582912.0f);
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const float2 r01 = __fadd2_rn(make_float2(v[4 * q], v[4 * q + 1]), magic);
      const float2 r23 = __fadd2_rn(make_float2(v[4 * q + 2], v[4 * q + 3]), magic);
      w[q] = __byte_perm(__byte_perm(__float_as_uint(r01.x), __float_as_uint(r01.y), 0x0040u),
                         __byte_perm(__float_as_uint(r23.x), __float_as_uint(r23.y), 0x0040u), 0x5410u);
    }
  } else {
#pragma unroll
    for (int q = 0; q < NW; ++q)
      w[q] = f32x2_to_e4m3x2(v[4 * q], v[4 * q + 1]) | (f32x2_to_e4m3x2(v[4 * q + 2], v[4 * q + 3]) << 16);
  }
}

// one vector <-> float2 pairs (the accumulators of the packed fp32x2 FMA path):
// element 2u is .x, element 2u+1 is .y
template <int F>
__device__ __forceinline__ void unpack_vec(const typename Vec<F>::Raw raw, float2* v) {
  uint32_t w[Vec<F>::WORDS];
  raw_words<F>(raw, w);
  float t[Vec<F>::N];
  unpack_words<F, Vec<F>::WORDS>(w, t);
#pragma unroll
  for (int u = 0; u < Vec<F>::N / 2; ++u) v[u] = make_float2(t[2 * u], t[2 * u + 1]);
}

template <int F>
__device__ __forceinline__ typename Vec<F>::Raw pack_vec_rne(const float2* v) {
  float t[Vec<F>::N];
#pragma unroll
  for (int u = 0; u < Vec<F>::N / 2; ++u) {
    t[2 * u] = v[u].x;
    t[2 * u + 1] = v[u].y;
  }
  uint32_t w[Vec<F>::WORDS];
  pack_words_rne<F, Vec<F>::WORDS>(t, w);
  return words_raw<F>(w);
}

}  // namespace rsm
