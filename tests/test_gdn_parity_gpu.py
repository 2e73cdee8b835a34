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
