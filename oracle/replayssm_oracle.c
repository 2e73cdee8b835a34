/*
 * replayssm_oracle.c -- plain CPU oracle for ReplaySSM prefix materialization.
 *
 * TEST INFRASTRUCTURE ONLY (see replayssm_oracle.h).  Slow on purpose: one
 * nested loop per definition, in the order the definition is written, with
 * no blocking, fusion or reordering.  Built with -O2 -ffp-contract=off and
 * no fast-math so that every fp32 step below rounds on its own.
 *
 * Precision.  The recurrence is evaluated in fp64.  The pages fix only the
 * storage formats, so every decision that turns a real number into stored
 * bits (the fp32 value a state element is rounded to, a row's amax and scale,
 * a quantized code, a stochastic-rounding choice) is taken in fp32, the
 * kernel's precision, from the fp64 result rounded once to fp32.  A stored
 * one-byte state decodes to the real number code * scale, which fp64 holds
 * exactly, so the decode adds no rounding of its own.
 *
 * Sources (all restated, none copied):
 *  - flashinfer.mamba.replayssm_materialize API page: signature, Parameters
 *    (pointer/stride tables, slot tables, ring_start/replay_prefix_len,
 *    active_request_indices, pad_slot_id, rand_seed/philox_rounds) and Notes.
 *  - FlashInfer PR #4815 "Replayssm prefix materialize", Description: a
 *    historical state plus a ring of inputs; apply a caller-chosen prefix.
 *  - Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
 *    (SC'11), section 5.2 (Philox): the 4x32 round function and key schedule.
 *  - IEEE 754 binary16 / bfloat16 (upper half of binary32) / OCP FP8 E4M3
 *    ("fn": no infinities, S.1111.111 is NaN, max 448) element formats.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - the caches are indexed by the SOURCE slot (the ring belongs to the
 *    source state); slot layouts are x [R,H,D], B [R,G,N], dt [R,H],
 *    state [H,D,N], scale [H,D], each contiguous inside its slot;
 *  - head h uses B group h / heads_per_group;
 *  - dt in the cache is the final fp32 step size, A the final (negative) value;
 *  - one-byte state is symmetric, one fp32 scale per (head, dim-row):
 *    scale = amax/qmax and codes = round(v / scale), the plain quotient, both
 *    fp32 operations, with qmax 127 (int8) or 448 (fp8 e4m3fn); a row whose
 *    qmax/amax is not finite (amax == 0, or so small that the scale cannot
 *    be inverted in fp32) is stored as zero codes with scale 0;
 *  - stochastic rounding: Philox-4x32 with philox_rounds rounds,
 *    key = (lo32(seed), hi32(seed)); element e = (h*dim + i)*dstate + j gets
 *    a 16-bit random number r16, and its magnitude goes up to the next grid
 *    point iff floor((|y| - lo)/ulp * 2^16) + r16 >= 2^16 (the top 16 bits of
 *    the discarded part plus r16 carry), then saturates to the largest finite
 *    value.  The bits are assigned as the sm_100-family conversion with
 *    stochastic rounding (PTX cvt.rs) consumes one 32-bit word:
 *      16-bit state: counter (e>>3, dst_slot, layer, 0), word w = out[(e>>1)&3],
 *        half c = low (e even) or high (e odd) 16 bits of w; bf16 r16 = c,
 *        f16 r16 = (c << 3) mod 2^16 (13 random bits for 13 discarded bits);
 *      one-byte state: counter (e>>4, dst_slot, layer, 0), w = out[(e>>2)&3],
 *        c = low (e&3 < 2) or high half of w, r16 = c for e&3 even and c with
 *        its 16 bits reversed for e&3 odd (two elements per half).
 */
#include "replayssm_oracle.h"

#include <float.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static char g_err[256];

static int fail(const char *msg, long long v) {
  snprintf(g_err, sizeof g_err, "%s (%lld)", msg, v);
  return -1;
}

const char *oracle_last_error(void) { return g_err; }
int oracle_args_size(void) { return (int)sizeof(oracle_args); }

/* ------------------------------------------------------------------------ */
/* Element formats, from their definitions.                                  */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static uint32_t bits_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

double oracle_decode(int fmt, uint32_t bits) {
  switch (fmt) {
    case ORACLE_F32:
      return f32_from_bits(bits);
    case ORACLE_BF16: /* bfloat16 is the upper half of a binary32 */
      return f32_from_bits((bits & 0xFFFFu) << 16);
    case ORACLE_F16: {
      int s = (bits >> 15) & 1, e = (bits >> 10) & 31, m = bits & 1023;
      double v;
      if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m/1024 * 2^-14 */
      else if (e == 31)
        v = m ? NAN : INFINITY;
      else
        v = ldexp((double)(1024 + m), e - 25); /* (1+m/1024) * 2^(e-15) */
      return s ? -v : v;
    }
    case ORACLE_FP8_E4M3: {
      int s = (bits >> 7) & 1, e = (bits >> 3) & 15, m = bits & 7;
      double v;
      if (e == 15 && m == 7)
        v = NAN; /* the only NaN pattern; the format has no infinities */
      else if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
      else
        v = ldexp((double)(8 + m), e - 10); /* (1+m/8) * 2^(e-7) */
      return s ? -v : v;
    }
    case ORACLE_I8:
      return (double)(int8_t)(bits & 0xFF);
  }
  return NAN;
}

/* Grid description: a value on the grid is k * ulp(|v|) with
 * ulp(a) = 2^(max(floor(log2 a), emin) - mant); int8 is the integer grid. */
typedef struct {
  int mant, emin, integer, inf_on_overflow;
  double maxfin;
} grid_t;

static int grid_of(int fmt, grid_t *g) {
  switch (fmt) {
    case ORACLE_BF16:
      *g = (grid_t){7, -126, 0, 1, ldexp(255.0, 120)}; /* (2 - 2^-7) * 2^127 */
      return 0;
    case ORACLE_F16:
      *g = (grid_t){10, -14, 0, 1, 65504.0};
      return 0;
    case ORACLE_FP8_E4M3:
      *g = (grid_t){3, -6, 0, 0, 448.0};
      return 0;
    case ORACLE_I8:
      *g = (grid_t){0, 0, 1, 0, 127.0};
      return 0;
  }
  return -1;
}

static double grid_ulp(const grid_t *g, double a) {
  if (g->integer) return 1.0;
  int e;
  frexp(a, &e); /* a = f * 2^e with f in [0.5, 1): floor(log2 a) = e - 1 */
  int E = e - 1;
  if (E < g->emin) E = g->emin;
  return ldexp(1.0, E - g->mant);
}

double oracle_round(int fmt, double y, int stochastic, uint32_t r16) {
  grid_t g;
  if (grid_of(fmt, &g) != 0) return NAN;
  if (isnan(y)) return y;
  double a = fabs(y);
  if (a == 0.0) return y;
  double ulp = grid_ulp(&g, a);
  double lo = floor(a / ulp) * ulp; /* exact: ulp is a power of two */
  double hi = lo + ulp;
  double r;
  if (!stochastic) {
    double dlo = a - lo, dhi = hi - a;
    if (dlo < dhi)
      r = lo;
    else if (dhi < dlo)
      r = hi;
    else /* tie: keep the neighbour whose last grid digit is even */
      r = (fmod(lo / ulp, 2.0) == 0.0) ? lo : hi;
  } else {
    /* up with probability floor((a-lo)/ulp * 2^16) / 2^16: the top 16 bits of
     * the discarded part (exact in fp64: a power-of-two scaling and a floor)
     * plus the random number carry past 2^16 */
    const double d16 = floor((a - lo) / ulp * 65536.0);
    r = (d16 + (double)(r16 & 0xFFFFu) >= 65536.0) ? hi : lo;
  }
  if (r > g.maxfin) r = (g.inf_on_overflow && !stochastic) ? INFINITY : g.maxfin;
  return copysign(r, y);
}

uint32_t oracle_encode(int fmt, double v) {
  int s = signbit(v) ? 1 : 0;
  double a = fabs(v);
  switch (fmt) {
    case ORACLE_F32:
      return bits_from_f32((float)v);
    case ORACLE_BF16:
      /* v is on the bfloat16 grid, hence exact in binary32: keep the top half */
      return bits_from_f32((float)v) >> 16;
    case ORACLE_F16: {
      uint32_t sb = (uint32_t)s << 15;
      if (isnan(v)) return sb | 0x7E00u;
      if (isinf(v)) return sb | 0x7C00u;
      if (a < ldexp(1.0, -14)) return sb | (uint32_t)(a / ldexp(1.0, -24));
      int e;
      frexp(a, &e);
      int E = e - 1;
      uint32_t m = (uint32_t)(a / ldexp(1.0, E - 10)) - 1024u;
      return sb | ((uint32_t)(E + 15) << 10) | m;
    }
    case ORACLE_FP8_E4M3: {
      uint32_t sb = (uint32_t)s << 7;
      if (isnan(v)) return sb | 0x7Fu;
      if (a < ldexp(1.0, -6)) return sb | (uint32_t)(a / ldexp(1.0, -9));
      int e;
      frexp(a, &e);
      int E = e - 1;
      uint32_t m = (uint32_t)(a / ldexp(1.0, E - 3)) - 8u;
      return sb | ((uint32_t)(E + 7) << 3) | m;
    }
    case ORACLE_I8:
      return (uint32_t)(uint8_t)(int8_t)v;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Philox-4x32 (Salmon et al., SC'11, section 5.2).                          */
/* ------------------------------------------------------------------------ */

void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds,
                       uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u; /* round multipliers */
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u; /* Weyl key increments */
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < rounds; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * c0;
    uint64_t p1 = (uint64_t)M1 * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

static uint32_t reverse16(uint32_t c) {
  uint32_t r = 0;
  for (int i = 0; i < 16; ++i)
    if (c & (1u << i)) r |= 1u << (15 - i);
  return r;
}

/* The 16-bit random number of element e of (layer, dst slot) in format fmt
 * (the assignment stated at the top of this file). */
static uint32_t sr_bits(const oracle_args *a, int fmt, int layer, int32_t dst, int64_t e) {
  int64_t seed = *a->rand_seed;
  uint32_t key[2] = {(uint32_t)((uint64_t)seed & 0xFFFFFFFFu),
                     (uint32_t)((uint64_t)seed >> 32)};
  uint32_t out[4];
  if (fmt == ORACLE_I8 || fmt == ORACLE_FP8_E4M3) {
    uint32_t ctr[4] = {(uint32_t)(e >> 4), (uint32_t)dst, (uint32_t)layer, 0u};
    oracle_philox4x32(ctr, key, a->philox_rounds, out);
    uint32_t w = out[(e >> 2) & 3];
    uint32_t c = (e & 3) < 2 ? (w & 0xFFFFu) : (w >> 16);
    return (e & 1) ? reverse16(c) : c;
  }
  uint32_t ctr[4] = {(uint32_t)(e >> 3), (uint32_t)dst, (uint32_t)layer, 0u};
  oracle_philox4x32(ctr, key, a->philox_rounds, out);
  uint32_t w = out[(e >> 1) & 3];
  uint32_t c = (e & 1) ? (w >> 16) : (w & 0xFFFFu);
  return fmt == ORACLE_F16 ? ((c << 3) & 0xFFFFu) : c;
}

/* ------------------------------------------------------------------------ */
/* Storage access.                                                           */
/* ------------------------------------------------------------------------ */

static int elem_size(int fmt) {
  switch (fmt) {
    case ORACLE_F32: return 4;
    case ORACLE_BF16:
    case ORACLE_F16: return 2;
    case ORACLE_I8:
    case ORACLE_FP8_E4M3: return 1;
  }
  return 0;
}

static uint32_t load_bits(const void *base, int64_t idx, int fmt) {
  const unsigned char *p = (const unsigned char *)base + idx * elem_size(fmt);
  switch (elem_size(fmt)) {
    case 4: { uint32_t u; memcpy(&u, p, 4); return u; }
    case 2: { uint16_t u; memcpy(&u, p, 2); return u; }
    case 1: return p[0];
  }
  return 0;
}

static void store_bits(void *base, int64_t idx, int fmt, uint32_t bits) {
  unsigned char *p = (unsigned char *)base + idx * elem_size(fmt);
  switch (elem_size(fmt)) {
    case 4: memcpy(p, &bits, 4); break;
    case 2: { uint16_t u = (uint16_t)bits; memcpy(p, &u, 2); break; }
    case 1: p[0] = (unsigned char)bits; break;
  }
}

static int is_quantized(int fmt) { return fmt == ORACLE_I8 || fmt == ORACLE_FP8_E4M3; }

static float load_f32(const void *base, int64_t idx) {
  float f;
  memcpy(&f, (const unsigned char *)base + idx * 4, 4);
  return f;
}

/* ------------------------------------------------------------------------ */
/* The operation.                                                            */
/* ------------------------------------------------------------------------ */

static int check_args(const oracle_args *a) {
  if (!a) return fail("null args", 0);
  if (!a->state_ptrs || !a->state_slot_strides || !a->x_cache_ptrs ||
      !a->x_cache_slot_strides || !a->B_cache_ptrs || !a->B_cache_slot_strides ||
      !a->dt_cache_ptrs || !a->dt_cache_slot_strides || !a->A_ptrs ||
      !a->src_slots || !a->dst_slots || !a->ring_start || !a->replay_prefix_len ||
      !a->active_request_indices)
    return fail("null table", 0);
  if (a->num_layers <= 0) return fail("num_layers", a->num_layers);
  if (a->batch <= 0) return fail("batch", a->batch);
  if (a->dim <= 0 || a->dstate <= 0) return fail("dim/dstate", a->dim);
  if (a->num_heads <= 0 || a->num_heads > 0x7FFFFFFF) return fail("num_heads", a->num_heads);
  if (a->heads_per_group <= 0 || a->num_heads % a->heads_per_group != 0)
    return fail("heads_per_group", a->heads_per_group);
  if (a->max_window < 1) return fail("max_window", a->max_window);
  if (a->ring_buffer_len < 1) return fail("ring_buffer_len", a->ring_buffer_len);
  if (elem_size(a->state_dtype) == 0) return fail("state_dtype", a->state_dtype);
  if (a->input_dtype != ORACLE_BF16 && a->input_dtype != ORACLE_F32)
    return fail("input_dtype", a->input_dtype);
  if (a->matrixA_dtype != ORACLE_F32 && a->matrixA_dtype != ORACLE_BF16 &&
      a->matrixA_dtype != ORACLE_F16)
    return fail("matrixA_dtype", a->matrixA_dtype);
  if (is_quantized(a->state_dtype) && (!a->state_scale_ptrs || !a->state_scale_slot_strides))
    return fail("quantized state needs scale tables", 0);
  if (a->philox_rounds < 0) return fail("philox_rounds", a->philox_rounds);
  if (a->philox_rounds > 0 && !a->rand_seed) return fail("philox_rounds needs rand_seed", 0);
  return 0;
}

/* n = position of the first -1; validates what the selected entries refer to. */
static int active_count(const oracle_args *a, int32_t *n_out) {
  int32_t n = 0;
  while (n < a->batch && a->active_request_indices[n] != -1) ++n;
  for (int32_t i = 0; i < n; ++i) {
    int32_t b = a->active_request_indices[i];
    if (b < 0 || b >= a->batch) return fail("active index out of range", b);
    for (int32_t q = 0; q < i; ++q)
      if (a->active_request_indices[q] == b) return fail("active index repeated", b);
    if (a->ring_start[b] < 0 || a->ring_start[b] >= a->ring_buffer_len)
      return fail("ring_start out of range", a->ring_start[b]);
    if (a->replay_prefix_len[b] < 0 || a->replay_prefix_len[b] > a->max_window)
      return fail("replay_prefix_len out of range", a->replay_prefix_len[b]);
  }
  *n_out = n;
  return 0;
}

/* Destination slots must be distinct and must not alias a slot that another
 * (layer, request) reads.  A destination equal to its own source slot is the
 * in-place case (the prefix committed into the source slot): each head tile is
 * read completely before it is written, so it is well defined. */
static int check_aliasing(const oracle_args *a, int32_t n) {
  for (int32_t l = 0; l < a->num_layers; ++l) {
    for (int32_t i = 0; i < n; ++i) {
      int32_t b = a->active_request_indices[i];
      int32_t s = a->src_slots[(int64_t)l * a->batch + b];
      int32_t d = a->dst_slots[(int64_t)l * a->batch + b];
      if (s == a->pad_slot_id || d == a->pad_slot_id) continue;
      if (s < 0 || d < 0) return fail("negative slot that is not pad_slot_id", s < 0 ? s : d);
      if (a->num_slots > 0 && (s >= a->num_slots || d >= a->num_slots))
        return fail("slot past the end of the pool", s >= a->num_slots ? s : d);
      for (int32_t q = 0; q < n; ++q) {
        int32_t b2 = a->active_request_indices[q];
        int32_t s2 = a->src_slots[(int64_t)l * a->batch + b2];
        int32_t d2 = a->dst_slots[(int64_t)l * a->batch + b2];
        if (s2 == a->pad_slot_id || d2 == a->pad_slot_id) continue;
        if (d == s2 && q != i) return fail("destination slot is also a source slot", d);
        if (q != i && d == d2) return fail("destination slot repeated", d);
      }
    }
  }
  return 0;
}

static double load_input(const void *base, int64_t idx, int fmt) {
  return oracle_decode(fmt, load_bits(base, idx, fmt));
}

/* Writes one head's [dim, dstate] fp64 state S to the destination tile;
 * (layer, dst) are the Philox counter's layer and slot words. */
static void write_head(const oracle_args *a, int layer, int32_t dst, int64_t h,
                       const double *S, void *dst_state, float *dst_scale) {
  const int fmt = a->state_dtype;
  const int D = a->dim, N = a->dstate;
  const int sr = a->philox_rounds > 0;
  for (int i = 0; i < D; ++i) {
    const int64_t row = (h * D + i) * (int64_t)N;
    if (fmt == ORACLE_F32) {
      for (int j = 0; j < N; ++j)
        store_bits(dst_state, row + j, fmt, bits_from_f32((float)S[i * N + j]));
    } else if (fmt == ORACLE_BF16 || fmt == ORACLE_F16) {
      for (int j = 0; j < N; ++j) {
        float y = (float)S[i * N + j];
        uint32_t w = sr ? sr_bits(a, fmt, layer, dst, row + j) : 0u;
        store_bits(dst_state, row + j, fmt, oracle_encode(fmt, oracle_round(fmt, y, sr, w)));
      }
    } else { /* one-byte state: symmetric, one scale per (head, dim-row) */
      const float qmax = (fmt == ORACLE_I8) ? 127.0f : 448.0f;
      float amax = 0.0f;
      for (int j = 0; j < N; ++j) {
        float v = (float)S[i * N + j];
        amax = fmaxf(amax, fabsf(v));
      }
      float scale = amax / qmax;
      if (!(qmax / amax <= FLT_MAX)) { /* amax == 0 or so small that qmax/amax overflows */
        for (int j = 0; j < N; ++j) store_bits(dst_state, row + j, fmt, 0u);
        dst_scale[h * D + i] = 0.0f;
        continue;
      }
      for (int j = 0; j < N; ++j) {
        float v = (float)S[i * N + j];
        float y = v / scale; /* the code in units of the scale, one fp32 division */
        uint32_t w = sr ? sr_bits(a, fmt, layer, dst, row + j) : 0u;
        store_bits(dst_state, row + j, fmt, oracle_encode(fmt, oracle_round(fmt, y, sr, w)));
      }
      dst_scale[h * D + i] = scale;
    }
  }
}

int oracle_materialize(const oracle_args *a) {
  int rc = check_args(a);
  if (rc) return rc;
  int32_t n = 0;
  if ((rc = active_count(a, &n))) return rc;
  if ((rc = check_aliasing(a, n))) return rc;

  const int fmt = a->state_dtype, esz = elem_size(fmt);
  const int D = a->dim, N = a->dstate, R = a->ring_buffer_len;
  const int64_t H = a->num_heads, G = H / a->heads_per_group;
  const int64_t tile = (int64_t)D * N;
  double *S = (double *)malloc(sizeof(double) * tile);
  if (!S) return fail("out of host memory", tile);

  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = a->active_request_indices[i];
    const int32_t k = a->replay_prefix_len[b];
    const int32_t rs = a->ring_start[b];
    for (int32_t l = 0; l < a->num_layers; ++l) {
      const int32_t src = a->src_slots[(int64_t)l * a->batch + b];
      const int32_t dst = a->dst_slots[(int64_t)l * a->batch + b];
      /* the Philox counter's slot and layer words (reading 11) */
      const int32_t ctr_slot = a->sr_counter_slots ? a->sr_counter_slots[(int64_t)l * a->batch + b] : dst;
      const int ctr_layer = a->sr_counter_layers ? a->sr_counter_layers[l] : l;
      if (src == a->pad_slot_id || dst == a->pad_slot_id) continue;

      unsigned char *state = (unsigned char *)(intptr_t)a->state_ptrs[l];
      const int64_t sstride = a->state_slot_strides[l];
      const unsigned char *src_state = state + (int64_t)src * sstride * esz;
      unsigned char *dst_state = state + (int64_t)dst * sstride * esz;
      float *src_scale = NULL, *dst_scale = NULL;
      if (is_quantized(fmt)) {
        float *scale = (float *)(intptr_t)a->state_scale_ptrs[l];
        const int64_t cstride = a->state_scale_slot_strides[l];
        src_scale = scale + (int64_t)src * cstride;
        dst_scale = scale + (int64_t)dst * cstride;
      }

      if (k == 0) { /* exact state and scale copy */
        memmove(dst_state, src_state, (size_t)(H * tile * esz));
        if (is_quantized(fmt)) memmove(dst_scale, src_scale, (size_t)(H * D) * sizeof(float));
        continue;
      }

      /* the ring of the source slot */
      const unsigned char *x = (const unsigned char *)(intptr_t)a->x_cache_ptrs[l] +
                               (int64_t)src * a->x_cache_slot_strides[l] * elem_size(a->input_dtype);
      const unsigned char *Bc = (const unsigned char *)(intptr_t)a->B_cache_ptrs[l] +
                                (int64_t)src * a->B_cache_slot_strides[l] * elem_size(a->input_dtype);
      const float *dtc = (const float *)(intptr_t)a->dt_cache_ptrs[l] +
                         (int64_t)src * a->dt_cache_slot_strides[l];
      const void *Ap = (const void *)(intptr_t)a->A_ptrs[l];

      for (int64_t h = 0; h < H; ++h) {
        const int64_t g = h / a->heads_per_group;
        const double Ah = load_input(Ap, h, a->matrixA_dtype);
        /* decode the source tile */
        for (int ii = 0; ii < D; ++ii) {
          const int64_t row = (h * D + ii) * (int64_t)N;
          for (int j = 0; j < N; ++j) {
            uint32_t bits = load_bits(src_state, row + j, fmt);
            if (is_quantized(fmt)) {
              /* code * scale, exact in fp64 (8 significant bits times 24) */
              S[ii * N + j] = oracle_decode(fmt, bits) * (double)src_scale[h * D + ii];
            } else {
              S[ii * N + j] = oracle_decode(fmt, bits);
            }
          }
        }
        /* apply the prefix, token by token */
        for (int32_t t = 0; t < k; ++t) {
          const int64_t p = (rs + t) % R;
          const double dt = (double)load_f32(dtc, p * H + h);
          const double decay = exp(dt * Ah);
          for (int ii = 0; ii < D; ++ii) {
            const double dtx = dt * load_input(x, (p * H + h) * D + ii, a->input_dtype);
            for (int j = 0; j < N; ++j) {
              const double Bj = load_input(Bc, (p * G + g) * N + j, a->input_dtype);
              S[ii * N + j] = S[ii * N + j] * decay + dtx * Bj;
            }
          }
        }
        write_head(a, ctr_layer, ctr_slot, h, S, dst_state, dst_scale);
      }
    }
  }
  free(S);
  return 0;
}
