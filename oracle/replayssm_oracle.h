/*
 * replayssm_oracle.h -- plain CPU oracle for ReplaySSM prefix materialization.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct checker that
 * the CUDA library is compared against.  Only the test suite, the package's
 * smoke entry and the benchmark's CPU-baseline leg may load it; the product
 * path never does.  It shares no code, header or table with the CUDA library.
 *
 * Operation (flashinfer.mamba.replayssm_materialize API page, signature,
 * Parameters and Notes): for every request selected by the -1-terminated
 * active list and every layer, read the source state slot, apply
 * replay_prefix_len[b] ring entries starting at ring_start[b] (mod
 * ring_buffer_len) through  state = state*exp(dt*A[h]) + dt*x[p] (x) B[p],
 * and write the destination slot.  Prefix 0 is an exact state+scale copy;
 * a pad slot on either side skips the (layer, request).
 *
 * All table entries are HOST addresses (int64) and strides are in elements,
 * exactly as the pages define them for device memory.
 */
#ifndef REPLAYSSM_ORACLE_H
#define REPLAYSSM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORACLE_F32 = 0,
  ORACLE_BF16 = 1,
  ORACLE_F16 = 2,
  ORACLE_I8 = 3,
  ORACLE_FP8_E4M3 = 4
};

typedef struct oracle_args {
  const int64_t *state_ptrs, *state_slot_strides;
  const int64_t *x_cache_ptrs, *x_cache_slot_strides;
  const int64_t *B_cache_ptrs, *B_cache_slot_strides;
  const int64_t *dt_cache_ptrs, *dt_cache_slot_strides;
  const int64_t *A_ptrs;
  const int64_t *state_scale_ptrs, *state_scale_slot_strides;
  const int32_t *src_slots, *dst_slots;          /* [L, batch] row-major */
  const int32_t *ring_start, *replay_prefix_len; /* [batch] */
  const int32_t *active_request_indices;         /* [batch], -1 padded */
  const int64_t *rand_seed;                      /* one value, or NULL */
  int32_t num_layers, batch;
  int32_t state_dtype, input_dtype, matrixA_dtype;
  int32_t dim, dstate;
  int64_t num_heads;
  int32_t heads_per_group, max_window, ring_buffer_len, pad_slot_id;
  int32_t philox_rounds;
  /* Optional, NULL when unused: the slot and layer words of the Philox
   * counter are taken from these tables ([L, batch] and [L]) instead of the
   * destination slot and the layer index of this call.  A one-request copy of
   * a larger call then draws the random words that call draws. */
  const int32_t *sr_counter_slots;
  const int32_t *sr_counter_layers;
  /* Slots in every layer's pool; a selected (layer, request) whose slot is
   * at or past it is refused.  0 = not checked. */
  int32_t num_slots;
} oracle_args;

/* 0 on success; <0 when an argument or a metadata value is out of contract
 * (the oracle checks everything; it is a checker, not a product). */
int oracle_materialize(const oracle_args *a);
const char *oracle_last_error(void);

/* Pieces exposed so that tests can pin them one by one. */
void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds,
                       uint32_t out[4]);
/* Round y to the grid of `fmt` (ORACLE_BF16/F16/I8/FP8_E4M3): round to nearest
 * even when stochastic == 0, else stochastic rounding driven by the element's
 * 16-bit random number r16 (the magnitude goes up iff the top 16 bits of its
 * discarded part plus r16 carry past 2^16). */
double oracle_round(int fmt, double y, int stochastic, uint32_t r16);
/* Storage <-> value for one element of each state format. */
double oracle_decode(int fmt, uint32_t bits);
uint32_t oracle_encode(int fmt, double value_on_grid);
int oracle_args_size(void);

#ifdef __cplusplus
}
#endif
#endif
