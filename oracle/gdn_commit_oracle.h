/* gdn_commit_oracle.h -- plain CPU oracle for
 * flashinfer.gdn_decode.gated_delta_rule_replayssm_commit (API page).
 * TEST INFRASTRUCTURE ONLY. */
#pragma once
#include <stdint.h>

typedef struct {
  float* state;                       /* [layers, slots, hv, 128, 128] fp32, K-last; updated in place */
  const uint16_t* rawv;               /* bf16 [layers, slots, hv, t, 128] */
  const uint16_t* rawk;               /* bf16 [layers, slots, h, t, 128], before normalisation */
  const float* g;                     /* [layers, slots, hv, t] log-decay */
  const float* beta;                  /* [layers, slots, hv, t] sigmoid-beta */
  const int32_t* state_indices;       /* [batch] */
  const int32_t* accept_lens;         /* [batch], in [0, t] */
  const int32_t* track_state_indices; /* [batch] or NULL */
  const int32_t* track_steps;         /* [batch] or NULL (with track_state_indices) */
  int32_t layers, slots, hv, h, t, batch;
  int32_t use_qk_l2norm, null_block_id;
} oracle_gdn_args;

/* 0 on success; -1 on a contract violation (message in oracle_gdn_last_error). */
int oracle_gdn_commit(const oracle_gdn_args* a);
const char* oracle_gdn_last_error(void);
