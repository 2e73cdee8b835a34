/*
 * replayssm.h -- C ABI of libreplayssm.so: ReplaySSM prefix materialization on
 * GB300 (sm_103a).
 *
 * rsm_materialize() mirrors flashinfer.mamba.replayssm_materialize (API page:
 * signature, Parameters, Notes).  The page's torch.compile dependency anchors
 * (dependency_inputs / dependency_outputs) are torch plumbing and are not part
 * of a C call.  rsm_gdn_commit() (declared further down) mirrors
 * flashinfer.gdn_decode.gated_delta_rule_replayssm_commit.
 *
 * What it computes.  For every request b selected by the -1-terminated
 * active_request_indices and every layer l, read the source state slot
 * src_slots[l, b], apply replay_prefix_len[b] ring entries starting at ring
 * row ring_start[b] (modulo ring_buffer_len) through
 *     state[h, i, j] = state[h, i, j] * exp(dt[p, h] * A[h]) + dt[p, h] * x[p, h, i] * B[p, g(h), j]
 * and write the result to dst_slots[l, b].  The ring and the source slot are
 * only read.  Prefix 0 is an exact copy of the state (and of the scales of a
 * one-byte state).  A (layer, request) whose source or destination slot equals
 * pad_slot_id is skipped and its destination is not touched.  The work runs in
 * one launch over all layers; with an empty active list (first entry -1) the
 * launch does one load and exits.
 *
 * Memory layout (per layer; every stride below is in ELEMENTS of the table's
 * own element type and steps from one slot to the next):
 *   state  slot = [num_heads, dim, dstate], contiguous, state_dtype
 *   scale  slot = [num_heads, dim] fp32 (one-byte state only): value = code * scale
 *   x      slot = [ring_buffer_len, num_heads, dim]   input_dtype
 *   B      slot = [ring_buffer_len, num_heads/heads_per_group, dstate]   input_dtype
 *   dt     slot = [ring_buffer_len, num_heads] fp32, the final step size
 *   A           = [num_heads] matrixA_dtype (fp32), the final negative value
 * The caches of a (layer, request) are the ones of its SOURCE slot.  Head h
 * uses B group h / heads_per_group.
 *
 * Ownership.  The caller owns every buffer.  All table and metadata pointers
 * are DEVICE pointers.  The library allocates nothing, reads no device memory
 * on the host and does not synchronize: the call enqueues one kernel on
 * `stream` (a cudaStream_t, NULL = the legacy default stream) and returns.
 *
 * Errors.  Host-checkable arguments are validated before anything is
 * launched; on error nothing is enqueued, the return value is negative and
 * rsm_last_error() (thread-local) describes it.  Device-resident metadata is
 * not read on the host: out-of-contract values there are undefined behaviour
 * as on the API page, except that the kernel skips any (layer, request) whose
 * active index, ring_start or replay_prefix_len is out of range, or whose slot
 * is negative (and not pad_slot_id), instead of touching memory for it, and
 * ORs an RSM_STATUS_* bit into *device_status when that optional word is
 * given.  Slots past the end of a pool are caught the same way only when the
 * caller states the pool size in num_slots; with num_slots = 0 a slot at or
 * past the end of the pool is undefined behaviour (the kernel would read and
 * write outside the caller's buffers).
 *
 * Aliasing.  Destination slots must be distinct and must not be a source slot
 * that another (layer, request) of the same call reads; otherwise the result
 * is undefined.  dst_slots[l, b] == src_slots[l, b] is allowed: the prefix is
 * then committed into the source slot in place (each head tile is read whole
 * before it is written).
 */
#ifndef REPLAYSSM_H
#define REPLAYSSM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RSM_ABI_VERSION 4

#if defined(__GNUC__)
#define RSM_API __attribute__((visibility("default")))
#else
#define RSM_API
#endif

/* return codes */
#define RSM_OK 0
#define RSM_EINVAL (-1)  /* an argument fails a host-side check */
#define RSM_ENOTSUP (-2) /* valid, but no compiled kernel for this (dtype, dim, dstate) */
#define RSM_ECUDA (-3)   /* the CUDA runtime refused the launch */

/* bits the kernel ORs into *device_status (when device_status != NULL) */
#define RSM_STATUS_BAD_ACTIVE_INDEX 1u /* an active entry outside [0, batch) */
#define RSM_STATUS_BAD_RING_START 2u   /* ring_start outside [0, ring_buffer_len) */
#define RSM_STATUS_BAD_PREFIX_LEN 4u   /* replay_prefix_len outside [0, max_window] */
#define RSM_STATUS_BAD_SLOT 8u         /* a negative slot that is not pad_slot_id, or one >= num_slots */
#define RSM_STATUS_WAIT_TIMEOUT 16u    /* an internal pipeline wait gave up (never expected) */

typedef enum rsm_dtype {
  RSM_F32 = 0,
  RSM_BF16 = 1,
  RSM_F16 = 2,
  RSM_I8 = 3,       /* one-byte state: symmetric int8 codes, |code| <= 127 */
  RSM_FP8_E4M3 = 4  /* one-byte state: OCP FP8 E4M3 "fn" codes, |value| <= 448 */
} rsm_dtype;

typedef struct rsm_materialize_args {
  /* per-layer tables, each [num_layers], device int64 */
  const int64_t *state_ptrs, *state_slot_strides;
  const int64_t *x_cache_ptrs, *x_cache_slot_strides;
  const int64_t *B_cache_ptrs, *B_cache_slot_strides;
  const int64_t *dt_cache_ptrs, *dt_cache_slot_strides;
  const int64_t *A_ptrs;
  /* one-byte state only; otherwise may be NULL or hold zero entries */
  const int64_t *state_scale_ptrs, *state_scale_slot_strides;
  /* slot tables [num_layers, batch] row-major, device int32 */
  const int32_t *src_slots, *dst_slots;
  /* per-request metadata [batch], device int32 */
  const int32_t *ring_start, *replay_prefix_len;
  /* [batch] device int32: selected request indices, each once, then -1s */
  const int32_t *active_request_indices;
  /* one device int64 seed, required when philox_rounds > 0 */
  const int64_t *rand_seed;
  /* optional device uint32 word that receives RSM_STATUS_* bits; may be NULL */
  uint32_t *device_status;

  int32_t num_layers; /* L, rows of the slot tables */
  int32_t batch;      /* B, columns of the slot tables, length of the [B] tensors */
  int32_t state_dtype, input_dtype, matrixA_dtype; /* rsm_dtype values */
  int32_t dim, dstate;
  int64_t num_heads;        /* 1 .. INT32_MAX */
  int32_t heads_per_group;  /* divides num_heads */
  int32_t max_window;       /* 1 .. 64: largest replay_prefix_len the call may see */
  int32_t ring_buffer_len;  /* >= 1 */
  int32_t pad_slot_id;      /* slot sentinel to skip (the API page's default is -1) */
  int32_t philox_rounds;    /* 0 = round to nearest even; > 0 = Philox stochastic rounding */
  /* slots in every layer's state pool (and in its scale and cache pools): a
   * (layer, request) whose source or destination slot is >= num_slots is
   * skipped and flagged RSM_STATUS_BAD_SLOT.  0 = the pool size is not stated
   * and only negative slots are caught.  Not on the API page, whose tensors
   * carry their sizes; a C call has only pointers. */
  int32_t num_slots;
} rsm_materialize_args;

/*
 * Enqueue the materialization described by *args on `stream`.
 * Returns RSM_OK when the kernel was enqueued (or there was nothing to
 * enqueue), RSM_EINVAL / RSM_ENOTSUP / RSM_ECUDA otherwise.
 *
 * Supported: state_dtype F32, BF16, F16 with (dim, dstate) in {(16,16),
 * (64,64), (64,128)}; I8 and FP8_E4M3 with (64,128) only (the API page's rule
 * for one-byte state); input_dtype BF16 (the API page's requirement) or F32;
 * matrixA_dtype F32.
 *
 * Rounding of the written state: fp32 as is; bf16/fp16 round to nearest even;
 * one-byte state rewrites each (head, dim-row) with scale = amax/qmax and
 * codes = round(value / scale) (qmax 127 or 448, saturating), a row whose
 * qmax/amax is not finite becoming zero codes with scale 0.  The kernel forms
 * the quotient as value * (qmax/amax), so a code can sit one step from the
 * rounded quotient when the quotient lies within an fp32 ulp of a rounding
 * boundary.  With
 * philox_rounds > 0 every non-fp32 format rounds stochastically instead:
 * element e = (h*dim + i)*dstate + j gets a 16-bit random number r16 and its
 * magnitude goes up to the next grid point iff the top 16 bits of the part
 * the rounding discards, plus r16, carry past 2^16 (then saturates to the
 * largest finite value).  r16 comes from Philox-4x32 (philox_rounds rounds,
 * key = (lo32, hi32) of *rand_seed): for 16-bit state, counter (e>>3,
 * dst_slot, layer, 0), the low (e even) or high (e odd) half of word (e>>1)&3
 * (f16 uses its low 13 bits, as the top 13 of r16); for one-byte state,
 * counter (e>>4, dst_slot, layer, 0), the low (e&3 < 2) or high half of word
 * (e>>2)&3, bit-reversed for odd e.  This is the assignment of the sm_100
 * family's conversion with stochastic rounding (cvt.rs).
 */
RSM_API int rsm_materialize(const rsm_materialize_args *args, void *stream);

/* Message of the last failing call on this thread ("" if none). */
RSM_API const char *rsm_last_error(void);

/* sizeof(rsm_materialize_args), so that bindings can check their layout. */
RSM_API int rsm_args_size(void);

/* RSM_ABI_VERSION of the built library. */
RSM_API int rsm_abi_version(void);

/*
 * The launch rsm_materialize would make for *args on the current device,
 * without launching: grid CTAs, threads per CTA, dynamic shared memory bytes
 * and pipeline stages.  Same validation and return codes as rsm_materialize.
 */
RSM_API int rsm_launch_config(const rsm_materialize_args *args, int *grid, int *block,
                      int *smem_bytes, int *stages);

/*
 * Name of the kernel rsm_materialize would launch for *args:
 * "materialize_kernel" (fp32 and 16-bit state on the CUDA cores),
 * "materialize_q8tc_kernel" (int8 and fp8 state with bf16 inputs and an even
 * heads_per_group: items of two heads, the prefix as a tensor-core rank-k
 * update), "materialize_q8_kernel" (the other int8 and fp8 calls) or
 * "materialize_tc_kernel" (16-bit state with bf16 inputs at dim 64 x dstate
 * 128 and max_window >= 16: every replayed prefix applied as a tensor-core
 * rank-k update).  "" when
 * *args fails validation (the reason is in rsm_last_error()).  Needs no GPU;
 * the string is static.
 */
RSM_API const char *rsm_kernel_name(const rsm_materialize_args *args);

/*
 * ---------------------------------------------------------------------------
 * Gated-delta-rule commit (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit,
 * API page: signature, Parameters, Notes).
 *
 * What it computes.  For every request b whose slot s = state_indices[b] is
 * live (s > null_block_id) and whose accepted length n = accept_lens[b] is not
 * zero, and for every layer l and value head hv, the accepted tokens
 * t = 0 .. n-1 of the slot's windows are applied in order to the checkpoint
 * S = checkpoint_state[l, s, hv] (128 value rows x 128 key columns, fp32,
 * K-last), in place:
 *     k^ = k_t / sqrt(|k_t|^2 + 1e-6)   (use_qk_l2norm; otherwise k^ = k_t)
 *     S  = exp(g_t) * S
 *     S  = S + beta_t * (v_t - S k^) k^T
 * with k_t = rawk_cache[l, s, hv / (num_v_heads / num_k_heads), t, :] and
 * v_t = rawv_cache[l, s, hv, t, :].  With tracking, the state right after
 * token track_steps[b] (zero-based) is also written to
 * checkpoint_state[l, track_state_indices[b], hv] when that slot is live and
 * the step lies inside the accepted prefix; otherwise the track slot is left
 * unchanged.  The windows are only read; nothing is shifted or cleared.
 *
 * Memory layout (contiguous, every base 16-byte aligned, as the page requires):
 *   checkpoint_state [layers, slots, num_v_heads, 128, 128] fp32
 *   rawv_cache       [layers, slots, num_v_heads, window, 128] bf16
 *   rawk_cache       [layers, slots, num_k_heads, window, 128] bf16 (before normalisation)
 *   g_cache          [layers, slots, num_v_heads, window] fp32 log-decay
 *   beta_cache       [layers, slots, num_v_heads, window] fp32 (sigmoid already applied)
 *   state_indices, accept_lens, track_state_indices, track_steps: [batch] int32
 *
 * Ownership, errors and the status word are as for rsm_materialize: device
 * pointers, caller-owned, one kernel enqueued on `stream`, no allocation, no
 * host read of device memory, no synchronization.  The kernel skips a request
 * whose slot is >= slots (RSM_STATUS_BAD_SLOT) or whose accepted length is
 * outside [0, window] (RSM_STATUS_BAD_PREFIX_LEN); a track slot >= slots is
 * ignored and flagged likewise.  Live state slots must be unique and live
 * track slots distinct and disjoint from them (caller contract, not checked).
 */
typedef struct rsm_gdn_commit_args {
  float *checkpoint_state;
  const uint16_t *rawv_cache, *rawk_cache; /* bf16 bit patterns */
  const float *g_cache, *beta_cache;
  const int32_t *state_indices, *accept_lens;
  const int32_t *track_state_indices, *track_steps; /* both NULL, or both given */
  uint32_t *device_status;                         /* optional, RSM_STATUS_* bits */
  int32_t layers, slots;
  int32_t num_v_heads, num_k_heads; /* num_k_heads divides num_v_heads */
  int32_t window;                   /* T: 1 .. 64 */
  int32_t batch;                    /* >= 0; 0 enqueues nothing */
  int32_t use_qk_l2norm;            /* nonzero: normalise k with epsilon 1e-6 */
  int32_t null_block_id;            /* >= -1; slots <= it are ignored */
  int32_t backend;                  /* RSM_GDN_BACKEND_*; see below */
} rsm_gdn_commit_args;

/* Backends (GDN page, Parameters: backend).  AUTO and SIMT run the fp32 kernel
 * (contractions on the CUDA cores).  TCGEN05 runs the contractions on the
 * tensor cores with TF32 operands (10 explicit mantissa bits, so results
 * differ from the fp32 kernel's in the fourth significant digit); as on the
 * page it requires use_qk_l2norm, no tracking (track arrays NULL) and a window
 * of 4 to 8 tokens, and is refused otherwise (RSM_EINVAL). */
#define RSM_GDN_BACKEND_AUTO 0
#define RSM_GDN_BACKEND_SIMT 1
#define RSM_GDN_BACKEND_TCGEN05 2

/* Enqueue the commit described by *args on `stream`; same return codes as
 * rsm_materialize.  Host checks: non-NULL tensors, positive sizes, divisibility
 * of the heads, window range, null_block_id >= -1, track arrays both or
 * neither, and 16-byte alignment of every tensor base (RSM_EINVAL). */
RSM_API int rsm_gdn_commit(const rsm_gdn_commit_args *args, void *stream);

/* sizeof(rsm_gdn_commit_args). */
RSM_API int rsm_gdn_args_size(void);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H */
