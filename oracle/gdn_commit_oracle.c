/*
 * gdn_commit_oracle.c -- plain CPU oracle for committing an accepted ReplaySSM
 * prefix into gated-delta-rule checkpoints
 * (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit, API page:
 * signature, Parameters, Notes).
 *
 * TEST INFRASTRUCTURE ONLY: the slow, obviously correct checker that the
 * CUDA kernel is compared against.  It shares no code with the CUDA library.
 *
 * What it computes.  For every request b whose slot s = state_indices[b] is
 * live (s > null_block_id) and for every layer l and value head hv, the
 * accepted tokens t = 0 .. accept_lens[b]-1 of the slot's windows are applied
 * in order to the fp32 checkpoint S = checkpoint_state[l, s, hv] (K-last:
 * S[i][j], i over the 128 value dims, j over the 128 key dims), in place:
 *
 *   k^  = k_t / sqrt(|k_t|^2 + 1e-6)   (use_qk_l2norm; else k^ = k_t)
 *   S   = exp(g_t) * S                 (g: log-decay)
 *   u   = beta_t * (v_t - S k^)        (beta: sigmoid-beta, already applied)
 *   S   = S + u k^T
 *
 * with k_t = rawk[l, s, hv / (HV/H), t, :] and v_t = rawv[l, s, hv, t, :].
 * If a track slot is given (track_state_indices[b] > null_block_id) and
 * 0 <= track_steps[b] < accept_lens[b], the state right after token
 * track_steps[b] is also written to checkpoint_state[l, track slot, hv].
 *
 * Readings of what the page leaves open (the page names the method and its
 * inputs but prints no recurrence):
 *  - the recurrence is the gated delta rule in the order above (decay, then
 *    the delta correction against the decayed state);
 *  - value heads map to key heads in contiguous groups: h = hv / (HV/H);
 *  - window position t holds accepted token t (the cache is not shifted);
 *  - the epsilon of the K normalisation sits inside the square root (pinned
 *    by a key of squared norm 2^-20, where the other placements of the
 *    epsilon give results 30% or more apart);
 *  - evaluation in fp64, each stored value rounded once to fp32.
 */
#include "gdn_commit_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define DK 128
#define DV 128

static const char* g_gdn_err = "";

const char* oracle_gdn_last_error(void) { return g_gdn_err; }

static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static int live(int32_t slot, int32_t null_block_id) { return slot > null_block_id; }

/* Live state slots unique and in range; live track slots in range, mutually
 * distinct and disjoint from every live state slot (API page, Parameters). */
static int check_contract(const oracle_gdn_args* a) {
  for (int32_t b = 0; b < a->batch; ++b) {
    const int32_t s = a->state_indices[b];
    if (!live(s, a->null_block_id)) continue;
    if (s >= a->slots) { g_gdn_err = "state slot out of range"; return -1; }
    if (a->accept_lens[b] < 0 || a->accept_lens[b] > a->t) { g_gdn_err = "accept_len out of [0, T]"; return -1; }
    for (int32_t c = b + 1; c < a->batch; ++c)
      if (a->state_indices[c] == s) { g_gdn_err = "duplicate live state slot"; return -1; }
  }
  if (a->track_state_indices == NULL) return 0;
  for (int32_t b = 0; b < a->batch; ++b) {
    const int32_t ts = a->track_state_indices[b];
    if (!live(ts, a->null_block_id)) continue;
    if (ts >= a->slots) { g_gdn_err = "track slot out of range"; return -1; }
    for (int32_t c = 0; c < a->batch; ++c) {
      if (c != b && a->track_state_indices[c] == ts) { g_gdn_err = "duplicate live track slot"; return -1; }
      if (a->state_indices[c] == ts) { g_gdn_err = "track slot aliases a state slot"; return -1; }
    }
  }
  return 0;
}

int oracle_gdn_commit(const oracle_gdn_args* a) {
  g_gdn_err = "";
  if (!a || !a->state || !a->rawv || !a->rawk || !a->g || !a->beta || !a->state_indices || !a->accept_lens) {
    g_gdn_err = "null argument";
    return -1;
  }
  if (a->layers <= 0 || a->slots <= 0 || a->hv <= 0 || a->h <= 0 || a->t <= 0 || a->batch < 0 ||
      a->hv % a->h != 0 || a->null_block_id < -1) {
    g_gdn_err = "bad sizes";
    return -1;
  }
  if ((a->track_state_indices == NULL) != (a->track_steps == NULL)) {
    g_gdn_err = "track_state_indices and track_steps come together";
    return -1;
  }
  if (check_contract(a)) return -1;

  const int64_t L = a->layers, SL = a->slots, HV = a->hv, H = a->h, T = a->t;
  const int64_t per_h = HV / H;
  double* S = (double*)malloc(sizeof(double) * DV * DK);
  double kh[DK], v[DV];
  if (!S) { g_gdn_err = "out of memory"; return -1; }

  for (int32_t b = 0; b < a->batch; ++b) {
    const int64_t s = a->state_indices[b];
    const int32_t n = a->accept_lens[b];
    if (!live((int32_t)s, a->null_block_id) || n == 0) continue;
    int64_t ts = -1, step = -1;
    if (a->track_state_indices && live(a->track_state_indices[b], a->null_block_id)) {
      ts = a->track_state_indices[b];
      step = a->track_steps[b];
    }
    for (int64_t l = 0; l < L; ++l) {
      for (int64_t hv = 0; hv < HV; ++hv) {
        const int64_t hk = hv / per_h;
        float* st = a->state + ((l * SL + s) * HV + hv) * DV * DK;
        for (int i = 0; i < DV * DK; ++i) S[i] = (double)st[i];
        for (int32_t t = 0; t < n; ++t) {
          const uint16_t* kr = a->rawk + (((l * SL + s) * H + hk) * T + t) * DK;
          const uint16_t* vr = a->rawv + (((l * SL + s) * HV + hv) * T + t) * DV;
          const int64_t gi = ((l * SL + s) * HV + hv) * T + t;
          double nrm = 0.0;
          for (int j = 0; j < DK; ++j) {
            kh[j] = bf16_to_f64(kr[j]);
            nrm += kh[j] * kh[j];
          }
          if (a->use_qk_l2norm) {
            const double r = 1.0 / sqrt(nrm + 1e-6);
            for (int j = 0; j < DK; ++j) kh[j] *= r;
          }
          for (int i = 0; i < DV; ++i) v[i] = bf16_to_f64(vr[i]);
          const double alpha = exp((double)a->g[gi]);
          const double beta = (double)a->beta[gi];
          for (int i = 0; i < DV; ++i) {
            double* row = S + i * DK;
            double d = 0.0;
            for (int j = 0; j < DK; ++j) {
              row[j] *= alpha;
              d += row[j] * kh[j];
            }
            const double u = beta * (v[i] - d);
            for (int j = 0; j < DK; ++j) row[j] += u * kh[j];
          }
          if (ts >= 0 && t == step) {
            float* tr = a->state + ((l * SL + ts) * HV + hv) * DV * DK;
            for (int i = 0; i < DV * DK; ++i) tr[i] = (float)S[i];
          }
        }
        for (int i = 0; i < DV * DK; ++i) st[i] = (float)S[i];
      }
    }
  }
  free(S);
  return 0;
}
