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

// ---------------------------------------------------------------------------
// stochastic rounding of an fp32 value to a target grid
// ---------------------------------------------------------------------------
// The grid: spacing 2^(max(floor(log2|y|), emin) - mant) (integer grid: 1).
// Returns the rounded value as fp32 (exactly on the grid), saturated to maxfin.
template <int MANT, int EMIN, bool INTEGER>
__device__ __forceinline__ float sr_round(float y, uint32_t word, float maxfin) {
  const uint32_t bits = __float_as_uint(y);
  const uint32_t sign = bits & 0x80000000u;
  const uint32_t ab = bits ^ sign;
  {
    // Common case: a normal input whose grid spacing leaves 0 < d < 24 low
    // bits.  Adding the complement of the d-bit random number r carries into
    // the next grid point exactly when r < the discarded bits (the rule
    // below), so the sum truncated to the grid is the rounded value.
    const int eb = static_cast<int>(ab >> 23);
    const int d = INTEGER ? 150 - eb : 23 - MANT;
    if (eb >= (INTEGER ? 127 : EMIN + 127) && eb < 255 && d > 0 && d < 24) {
      const uint32_t r = (ab + ((~word) >> (32 - d))) & ~((1u << d) - 1u);
      return __uint_as_float(min(r, __float_as_uint(maxfin)) | sign);
    }
  }
  if (ab == 0u) return y;
  if (ab >= 0x7F800000u) return ab == 0x7F800000u ? __uint_as_float(__float_as_uint(maxfin) | sign) : y;
  const int eb = static_cast<int>(ab >> 23);
  const int E = eb ? eb - 127 : -126;                              // a = M * 2^(E-23)
  const uint32_t M = (ab & 0x7FFFFFu) | (eb ? 0x800000u : 0u);
  const int ulp_exp = INTEGER ? 0 : (E > EMIN ? E : EMIN) - MANT;  // grid spacing 2^ulp_exp
  const int d = ulp_exp - (E - 23);                                // bits of M below the spacing
  float r;
  if (d <= 0) {
    r = __uint_as_float(ab);  // already on the grid
  } else if (d < 24) {
    const uint32_t low = ab & ((1u << d) - 1u);
    const uint32_t lo_bits = ab - low;
    const bool up = (word >> (32 - d)) < low;
    r = __uint_as_float(up ? lo_bits + (1u << d) : lo_bits);
  } else {  // |y| below one spacing: neighbours are 0 and the spacing itself
    bool up;
    if (d <= 32)
      up = (word >> (32 - d)) < M;
    else if (d < 56)
      up = (static_cast<uint64_t>(word) << (d - 32)) < M;
    else
      up = (word == 0u);
    const float spacing = ulp_exp >= -126 ? __uint_as_float(static_cast<uint32_t>(ulp_exp + 127) << 23)
                                          : __uint_as_float(1u << (ulp_exp + 149));
    r = up ? spacing : 0.0f;
  }
  r = fminf(r, maxfin);
  return __uint_as_float(__float_as_uint(r) | sign);
}

__device__ __forceinline__ float sr_bf16(float y, uint32_t w) {
  return sr_round<7, -126, false>(y, w, __uint_as_float(0x7F7F0000u));
}
__device__ __forceinline__ float sr_f16(float y, uint32_t w) { return sr_round<10, -14, false>(y, w, 65504.0f); }
__device__ __forceinline__ float sr_e4m3(float y, uint32_t w) { return sr_round<3, -6, false>(y, w, 448.0f); }
__device__ __forceinline__ float sr_i8(float y, uint32_t w) { return sr_round<0, 0, true>(y, w, 127.0f); }

// stochastic rounding to the grid of state format F (fp32: identity)
template <int F>
__device__ __forceinline__ float sr_fmt(float y, uint32_t w) {
  if constexpr (F == RSM_BF16) return sr_bf16(y, w);
  else if constexpr (F == RSM_F16) return sr_f16(y, w);
  else if constexpr (F == RSM_I8) return sr_i8(y, w);
  else if constexpr (F == RSM_FP8_E4M3) return sr_e4m3(y, w);
  else return y;
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
