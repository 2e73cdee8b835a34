"""Gated-delta-rule commit: the CUDA kernel against the CPU oracle, element by
element, through the C ABI (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit,
API page).  Tolerance for the fp32 state: |gpu - ref| <= 1e-5 + 1e-5 |ref|;
slots the oracle leaves untouched must be bit-exact."""
import numpy as np
import pytest

import oracle
import mamba_replayssm_state_gb300 as rsm
from mamba_replayssm_state_gb300 import gdn_workloads as gw

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = 1e-5


def run_cuda(hw, status_expected=0):
    dw = gw.gdn_device_world_from_host(hw)
    rsm.gated_delta_rule_replayssm_commit(**dw.call_kwargs())
    torch.cuda.synchronize()
    assert int(dw.status.item()) == status_expected
    return dw.state.cpu().numpy()


def run_oracle(hw):
    ref = hw.copy()
    oracle.gdn_commit(ref)
    return ref.state


def compare(got, ref, before):
    untouched = np.all(ref == before, axis=(-1, -2))
    assert np.array_equal(got[untouched], before[untouched]), "a slot the oracle leaves alone was written"
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = TOL + TOL * np.abs(ref.astype(np.float64))
    worst = np.max(err - bound)
    assert worst <= 0, f"max error {err.max():.3e} exceeds the tolerance"
    return int((~untouched).sum())


def check(hw):
    got = run_cuda(hw)
    ref = run_oracle(hw)
    return compare(got, ref, hw.state)


def test_tiny_with_tracking():
    hw = gw.gdn_host_world(gw.GDN_SHAPES["gdn_tiny"], seed=0)
    hw.accept_lens[:] = [8, 0, 3, 5]
    hw.track_steps[:] = [4, 0, 2, 9]      # inside, (zero length), last token, outside
    assert check(hw) >= 3 * 2 * 4


@pytest.mark.parametrize("T,HV,H", [(1, 4, 4), (5, 8, 2), (8, 16, 4), (64, 4, 1)])
def test_windows_and_head_groups(T, HV, H):
    shape = gw.GdnShape("w", L=2, B=5, HV=HV, H=H, T=T, track=True)
    hw = gw.gdn_host_world(shape, seed=T * 100 + HV)
    hw.accept_lens[0] = T                  # the longest prefix
    hw.track_steps[0] = T - 1
    check(hw)


def test_every_accepted_length():
    shape = gw.GdnShape("len", L=1, B=9, HV=4, H=2, T=8, track=True)
    hw = gw.gdn_host_world(shape, seed=3)
    hw.accept_lens[:] = np.arange(9)
    hw.track_steps[:] = np.arange(9) - 1
    check(hw)


def test_raw_k():
    shape = gw.GdnShape("raw", L=2, B=4, HV=4, H=2, T=8, use_qk_l2norm=False, track=True)
    check(gw.gdn_host_world(shape, seed=4))


def test_null_slots_and_null_block_id():
    shape = gw.GdnShape("nul", L=2, B=6, HV=4, H=2, T=6, slots=16, null_block_id=2, track=True)
    hw = gw.gdn_host_world(shape, seed=5)
    hw.state_indices[:] = [2, 5, 0, 7, 3, 1]        # 2, 0, 1 are ignored
    hw.track_state_indices[:] = [9, 1, 10, 12, 2, 14]  # 1 and 2 are not live track slots
    hw.accept_lens[:] = 6
    hw.track_steps[:] = 3
    check(hw)


@pytest.mark.parametrize("bad,bit", [("slot", 8), ("len", 4), ("track", 8)])
def test_out_of_range_metadata_is_skipped_and_flagged(bad, bit):
    shape = gw.GdnShape("bad", L=2, B=4, HV=4, H=2, T=8, track=True, accept=("fixed", 5))
    hw = gw.gdn_host_world(shape, seed=6)
    hw.track_steps[:] = 2
    ref_in = hw.copy()
    if bad == "slot":
        hw.state_indices[1] = shape.pool + 3
        ref_in.accept_lens[1] = 0
    elif bad == "len":
        hw.accept_lens[1] = shape.T + 1
        ref_in.accept_lens[1] = 0
    else:
        hw.track_state_indices[1] = shape.pool + 3
        ref_in.track_state_indices[1] = -1
    got = run_cuda(hw, status_expected=bit)
    compare(got, run_oracle(ref_in), hw.state)


def test_repeated_calls_are_identical():
    hw = gw.gdn_host_world(gw.GDN_SHAPES["gdn_tiny"], seed=7)
    assert np.array_equal(run_cuda(hw), run_cuda(hw))


def test_full_size_sampled():
    """The benchmark's full-size call, checked on sampled (request, layer)
    pairs: each one's inputs are copied out and the oracle recomputes them."""
    shape = gw.GDN_SHAPES["gdn36_hv32_t8"]
    dw = gw.gdn_device_world_random(shape, seed=0)
    before = {}
    rng = np.random.default_rng(1)
    live = [b for b in range(shape.B) if int(dw.accept_lens[b]) > 0]
    picks = [(int(b), int(rng.integers(shape.L))) for b in rng.choice(live, size=4, replace=False)]
    for b, l in picks:
        s = int(dw.state_indices[b])
        ts = int(dw.track_state_indices[b])
        sub = gw.GdnShape("sub", L=1, B=1, HV=shape.HV, H=shape.H, T=shape.T, slots=2, track=True)
        before[(b, l)] = gw.GdnWorld(
            sub,
            np.stack([dw.state[l, s].cpu().numpy(), dw.state[l, ts].cpu().numpy()])[None].copy(),
            dw.rawv[l, s].view(torch.int16).cpu().numpy().view(np.uint16)[None, None].repeat(2, 1).copy(),
            dw.rawk[l, s].view(torch.int16).cpu().numpy().view(np.uint16)[None, None].repeat(2, 1).copy(),
            dw.g[l, s].cpu().numpy()[None, None].repeat(2, 1).copy(),
            dw.beta[l, s].cpu().numpy()[None, None].repeat(2, 1).copy(),
            np.array([0], np.int32), np.array([int(dw.accept_lens[b])], np.int32),
            np.array([1], np.int32), np.array([int(dw.track_steps[b])], np.int32))
    rsm.gated_delta_rule_replayssm_commit(**dw.call_kwargs())
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    for (b, l), w in before.items():
        s, ts = int(dw.state_indices[b]), int(dw.track_state_indices[b])
        ref = run_oracle(w)
        got = np.stack([dw.state[l, s].cpu().numpy(), dw.state[l, ts].cpu().numpy()])[None]
        compare(got, ref, w.state)


# ----------------------------------------------------------------------------
# the tcgen05 backend (TF32 contractions): normalised K, windows 4..8, no tracking
# ----------------------------------------------------------------------------

def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _tf32_bound(hw):
    """First-order bound on |tcgen05 result - exact result| for every element
    the call writes (the derivation is in the design notes): TF32 operands
    carry a relative error below delta = 2^-10, fp32 accumulation 2^-16 of
    the summed magnitudes; W = S0 k^ is off by (2 delta + 2^-16) sum|S0 k^|,
    the triangular solve propagates that through |L|, and the rank-n update
    adds 2 delta sum|c u k^| of its own."""
    delta, acc = 2.0 ** -10, 2.0 ** -16
    sh = hw.shape
    bound = np.zeros(hw.state.shape, np.float64)
    per_kh = sh.HV // sh.H
    for b in range(sh.B):
        s, n = int(hw.state_indices[b]), int(hw.accept_lens[b])
        if s <= sh.null_block_id or n == 0:
            continue
        for l in range(sh.L):
            for hv in range(sh.HV):
                k = _bf16_to_f64(hw.rawk[l, s, hv // per_kh, :n])                  # [n, DK]
                kh = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
                v = _bf16_to_f64(hw.rawv[l, s, hv, :n])                             # [n, DV]
                gam = np.cumprod(np.exp(hw.g[l, s, hv, :n].astype(np.float64)))
                beta = hw.beta[l, s, hv, :n].astype(np.float64)
                S0 = hw.state[l, s, hv].astype(np.float64)                          # [DV, DK]
                W = S0 @ kh.T                                                       # [DV, n]
                L = np.zeros((n, n))
                for t in range(n):
                    for q in range(t):
                        L[q, t] = beta[q] * gam[t] / gam[q] * (kh[q] @ kh[t])
                u = np.zeros((gw.DV, n))
                for t in range(n):
                    u[:, t] = v[t] - gam[t] * W[:, t] - u[:, :t] @ L[:t, t]
                c = beta * gam[-1] / gam
                dW = (2 * delta + acc) * (np.abs(S0) @ np.abs(kh).T)                # [DV, n]
                du = np.zeros((gw.DV, n))
                for t in range(n):
                    du[:, t] = gam[t] * dW[:, t] + du[:, :t] @ np.abs(L[:t, t])
                bound[l, s, hv] = (2 * delta * (np.abs(c * u) @ np.abs(kh))
                                   + (np.abs(c) * du) @ np.abs(kh))
    return bound


def _check_tc(hw):
    dw = gw.gdn_device_world_from_host(hw)
    kw = dw.call_kwargs()
    kw.update(track_state_indices=None, track_steps=None, backend="tcgen05")
    rsm.gated_delta_rule_replayssm_commit(**kw)
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    got = dw.state.cpu().numpy()
    ref = run_oracle(hw)
    before = hw.state
    untouched = np.all(ref == before, axis=(-1, -2))
    assert np.array_equal(got[untouched], before[untouched]), "a slot the oracle leaves alone was written"
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = 1.25 * _tf32_bound(hw) + 2.0 ** -22 * np.abs(ref.astype(np.float64)) + 1e-7
    assert np.all(err <= bound), f"max error {err.max():.3e}, worst excess {(err - bound).max():.3e}"
    return int((~untouched).sum()), float(err[~untouched].max()) if (~untouched).any() else 0.0


@pytest.mark.parametrize("T,HV,H", [(4, 4, 2), (6, 8, 2), (8, 8, 4), (8, 16, 16)])
def test_gdn_tcgen05_backend_within_the_tf32_bound(T, HV, H):
    shape = gw.GdnShape("tc", L=2, B=5, HV=HV, H=H, T=T, track=False)
    hw = gw.gdn_host_world(shape, seed=700 + T * 10 + HV)
    hw.accept_lens[0] = T                      # the longest prefix
    written, worst = _check_tc(hw)
    assert written >= 2 * HV


def test_gdn_tcgen05_backend_every_accepted_length_and_null_slots():
    shape = gw.GdnShape("tclen", L=2, B=9, HV=4, H=2, T=8, slots=24, null_block_id=1, track=False)
    hw = gw.gdn_host_world(shape, seed=71)
    hw.accept_lens[:] = np.arange(9)
    hw.state_indices[4] = 1                    # a null slot (<= null_block_id): left alone
    _check_tc(hw)


def test_gdn_tcgen05_backend_many_items_per_cta():
    """Several value heads per CTA, so that the arena wraps and both operand
    and accumulator buffers are reused many times."""
    shape = gw.GdnShape("tcmany", L=3, B=24, HV=16, H=4, T=8, track=False)
    hw = gw.gdn_host_world(shape, seed=72)
    written, _ = _check_tc(hw)
    assert written > 500
