"""Pins of the gated-delta-rule commit oracle
(flashinfer.gdn_decode.gated_delta_rule_replayssm_commit, API page) against
what the mathematics and the page fix, not against a retyped formula:

- one token is fully determined by two projections: along k^ the new state
  gives alpha*S k^ + beta*(v - alpha*S k^) (the delta rule's correction), and
  on any w orthogonal to k^ it gives alpha*S w (pure decay);
- beta = 0 is pure decay by exp(sum g);
- j tokens then k more equal j+k tokens;
- the track copy equals a call that stops at the tracked step; steps outside
  the accepted prefix and zero lengths write nothing (API page, track_steps,
  accept_lens);
- slots <= null_block_id are ignored (API page, state_indices);
- value head hv reads key head hv / (HV/H);
- normalised K is invariant to scaling the raw K.
"""
import numpy as np
import pytest

import oracle
from mamba_replayssm_state_gb300 import gdn_workloads as gw

DK = DV = 128


def one_head_world(T=1, n=1, seed=0, l2norm=True):
    shape = gw.GdnShape("one", L=1, B=1, HV=1, H=1, T=T, slots=2, accept=("fixed", n), use_qk_l2norm=l2norm)
    return gw.gdn_host_world(shape, seed=seed)


def bf16(v):
    return gw.bf16_bits_from_f32(np.asarray(v, np.float32))


def f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run(w):
    r = w.copy()
    oracle.gdn_commit(r)
    return r


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_single_token_projections(seed):
    w = one_head_world(seed=seed)
    s = int(w.state_indices[0])
    S0 = w.state[0, s, 0].astype(np.float64)
    k = f(w.rawk[0, s, 0, 0])
    kh = k / np.linalg.norm(k)
    v = f(w.rawv[0, s, 0, 0])
    alpha = np.exp(np.float64(w.g[0, s, 0, 0]))
    beta = np.float64(w.beta[0, s, 0, 0])
    S1 = run(w).state[0, s, 0].astype(np.float64)
    along = alpha * (S0 @ kh)
    np.testing.assert_allclose(S1 @ kh, along + beta * (v - along), rtol=2e-6, atol=2e-6)
    rng = np.random.default_rng(seed)
    for _ in range(3):
        x = rng.standard_normal(DK)
        x -= (x @ kh) * kh
        np.testing.assert_allclose(S1 @ x, alpha * (S0 @ x), rtol=2e-6, atol=2e-5)


def test_single_token_unnormalised_k():
    """Without normalisation k is used raw: S1 k = alpha S0 k + beta (v - alpha S0 k) |k|^2."""
    w = one_head_world(seed=4, l2norm=False)
    s = int(w.state_indices[0])
    k = np.zeros(DK, np.float32)
    k[[3, 77]] = [2.0, -1.0]                       # |k|^2 = 5, exact in bf16
    w.rawk[0, s, 0, 0] = bf16(k)
    S0 = w.state[0, s, 0].astype(np.float64)
    v = f(w.rawv[0, s, 0, 0])
    alpha = np.exp(np.float64(w.g[0, s, 0, 0]))
    beta = np.float64(w.beta[0, s, 0, 0])
    S1 = run(w).state[0, s, 0].astype(np.float64)
    k = k.astype(np.float64)
    along = alpha * (S0 @ k)
    np.testing.assert_allclose(S1 @ k, along + beta * (v - along) * 5.0, rtol=2e-6, atol=2e-5)


def test_beta_zero_is_pure_decay():
    w = one_head_world(T=6, n=5, seed=5)
    w.beta[:] = 0.0
    s = int(w.state_indices[0])
    S1 = run(w).state[0, s, 0].astype(np.float64)
    decay = np.exp(np.sum(w.g[0, s, 0, :5].astype(np.float64)))
    np.testing.assert_allclose(S1, decay * w.state[0, s, 0].astype(np.float64), rtol=2e-6, atol=1e-30)


def test_composition_j_then_k():
    j, k = 3, 4
    w = one_head_world(T=8, n=j + k, seed=6)
    s = int(w.state_indices[0])
    whole = run(w).state[0, s, 0]
    first = w.copy()
    first.accept_lens[:] = j
    first = run(first)
    second = first.copy()
    for arr in (second.rawv, second.rawk, second.g, second.beta):
        arr[0, s, :, :k] = arr[0, s, :, j:j + k].copy()
    second.accept_lens[:] = k
    second = run(second)
    np.testing.assert_allclose(second.state[0, s, 0], whole, rtol=1e-6, atol=1e-6)


def tracked_world(seed=7):
    shape = gw.GdnShape("trk", L=2, B=3, HV=4, H=2, T=8, track=True, accept=("fixed", 6))
    w = gw.gdn_host_world(shape, seed=seed)
    w.track_steps[:] = [2, 6, -1]   # inside, just outside, outside
    return w


def test_track_copy_equals_the_state_at_that_step():
    w = tracked_world()
    out = run(w)
    stop = w.copy()
    stop.accept_lens[0] = 3          # zero-based step 2 -> three tokens
    stop.track_state_indices = stop.track_steps = None
    stop = run(stop)
    s0, t0 = int(w.state_indices[0]), int(w.track_state_indices[0])
    assert np.array_equal(out.state[:, t0], stop.state[:, s0])
    for b in (1, 2):                 # steps outside the prefix: track slots untouched
        tb = int(w.track_state_indices[b])
        assert np.array_equal(out.state[:, tb], w.state[:, tb])


def test_zero_length_is_a_no_op_including_track():
    w = tracked_world(seed=8)
    w.accept_lens[:] = 0
    w.track_steps[:] = 0
    assert np.array_equal(run(w).state, w.state)


def test_null_slots_are_ignored_and_other_slots_untouched():
    shape = gw.GdnShape("nul", L=2, B=4, HV=2, H=1, T=4, slots=12, null_block_id=3, accept=("fixed", 4))
    w = gw.gdn_host_world(shape, seed=9)
    w.state_indices[:] = [3, 7, 1, 9]           # 3 and 1 are <= null_block_id
    out = run(w)
    changed = {s for s in range(12) if not np.array_equal(out.state[:, s], w.state[:, s])}
    assert changed == {7, 9}


def test_value_heads_read_their_key_head():
    shape = gw.GdnShape("gqa", L=1, B=1, HV=6, H=3, T=2, accept=("fixed", 2))
    w = gw.gdn_host_world(shape, seed=10)
    s = int(w.state_indices[0])
    base = run(w)
    pert = w.copy()
    pert.rawk[0, s, 1] = bf16(np.ones((2, DK)))
    out = run(pert)
    changed = [hv for hv in range(6) if not np.array_equal(out.state[0, s, hv], base.state[0, s, hv])]
    assert changed == [2, 3]


def test_normalised_k_is_scale_invariant():
    shape = gw.GdnShape("scl", L=1, B=2, HV=2, H=2, T=4, accept=("fixed", 4))
    w = gw.gdn_host_world(shape, seed=11)
    scaled = w.copy()
    scaled.rawk[:] = bf16(4.0 * f(w.rawk))      # a power of two: exact in bf16
    np.testing.assert_allclose(run(scaled).state, run(w).state, rtol=1e-6, atol=1e-6)


def test_windows_come_from_the_requests_own_slot():
    shape = gw.GdnShape("own", L=1, B=1, HV=2, H=1, T=4, slots=6, accept=("fixed", 4))
    w = gw.gdn_host_world(shape, seed=12)
    s = int(w.state_indices[0])
    other = (s + 1) % 3
    pert = w.copy()
    pert.rawv[0, other] = 0
    pert.rawk[0, other] = 0
    pert.g[0, other] = 0.0
    assert np.array_equal(run(pert).state[:, s], run(w).state[:, s])


@pytest.mark.parametrize("bad", ["dup_state", "track_alias", "len"])
def test_contract_violations_are_refused(bad):
    w = tracked_world(seed=13)
    if bad == "dup_state":
        w.state_indices[1] = w.state_indices[0]
    elif bad == "track_alias":
        w.track_state_indices[1] = w.state_indices[2]
    else:
        w.accept_lens[0] = w.shape.T + 1
    with pytest.raises(ValueError):
        oracle.gdn_commit(w)


@pytest.mark.parametrize("which", ["rawv", "g", "beta"])
def test_value_head_inputs_reach_only_their_head(which):
    shape = gw.GdnShape("vh", L=1, B=1, HV=4, H=2, T=2, accept=("fixed", 2))
    w = gw.gdn_host_world(shape, seed=14)
    s = int(w.state_indices[0])
    pert = w.copy()
    arr = getattr(pert, which)
    if which == "rawv":
        arr[0, s, 1] = bf16(np.full((2, DV), 3.0))
    else:
        arr[0, s, 1] = arr[0, s, 1] * 0.5
    out, base = run(pert), run(w)
    changed = [hv for hv in range(4) if not np.array_equal(out.state[0, s, hv], base.state[0, s, hv])]
    assert changed == [1]


def test_epsilon_sits_inside_the_square_root():
    """GDN page, Parameters, use_qk_l2norm: K is normalised with epsilon 1e-6.
    The reading fixed here is k^ = k / sqrt(|k|^2 + 1e-6).  With S0 = 0 and
    g = 0, one token leaves S1 = beta v k^T, so column c of S1 over beta v is
    k^'s entry c.  With |k|^2 = 2^-20 (about the epsilon) the placements differ
    by a factor near sqrt(2): inside the root 2^-10 / sqrt(2^-20 + 1e-6) = 0.716,
    added to the norm 2^-10 / (2^-10 + 1e-6) = 0.999, left out 1."""
    w = one_head_world(seed=15)
    s = int(w.state_indices[0])
    w.state[0, s, 0] = 0.0
    w.g[0, s, 0, 0] = 0.0
    k = np.zeros(DK, np.float32)
    k[5] = 2.0 ** -10                           # exact in bf16; |k|^2 = 2^-20
    w.rawk[0, s, 0, 0] = bf16(k)
    v = f(w.rawv[0, s, 0, 0])
    beta = np.float64(w.beta[0, s, 0, 0])
    S1 = run(w).state[0, s, 0].astype(np.float64)
    inside = 2.0 ** -10 / np.sqrt(2.0 ** -20 + 1e-6)
    np.testing.assert_allclose(S1[:, 5], beta * v * inside, rtol=1e-6, atol=1e-30)
    assert not np.any(np.delete(S1, 5, axis=1))
    # the other placements are far outside that tolerance
    for other in (2.0 ** -10 / (2.0 ** -10 + 1e-6), 1.0):
        assert abs(other / inside - 1.0) > 0.3
