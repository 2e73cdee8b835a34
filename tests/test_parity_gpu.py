"""CUDA path against the CPU oracle, element by element, through the C ABI.

Small worlds are compared in full (every slot of every layer); the full-size
headline call is checked on sampled (layer, request) outputs, each recomputed
by the oracle from its own copy of the inputs, plus properties that hold at
any size.  Tolerances are in tests/parity.py.
"""
import zlib

import numpy as np
import pytest

import oracle
import mamba_replayssm_state_gb300 as rsm
from mamba_replayssm_state_gb300 import workloads as wl

from parity import compare_slot, compare_worlds, written_dsts

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def run_cuda(hw, status_expected=0):
    """Runs the CUDA path on a copy of host world `hw`; returns the host copy of the result."""
    dw = wl.device_world_from_host(hw)
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    got.scale = [None if t is None else wl._to_np(t) for t in dw.scale]
    status = int(dw.status.item())
    assert status == status_expected, f"device status {status:#x}"
    return got


def run_oracle(hw):
    ref = hw.copy()
    oracle.materialize(ref)
    return ref


def check(hw, exact=False):
    got = run_cuda(hw)
    ref = run_oracle(hw)
    return compare_worlds(got, ref, hw, exact=exact)


# ----------------------------------------------------------------------------
# the named workloads, reduced so that the oracle takes seconds
# ----------------------------------------------------------------------------

def test_tiny_all_active():
    hw = wl.host_world(wl.SHAPES["tiny_fp32"], seed=0)
    assert check(hw) >= 4


def test_tiny_three_active_then_terminator():
    hw = wl.host_world(wl.SHAPES["tiny_fp32"], seed=1)
    hw.active[3] = -1
    assert check(hw) >= 3


def test_tiny_entries_after_terminator_ignored():
    hw = wl.host_world(wl.SHAPES["tiny_fp32"], seed=2)
    b = hw.active.copy()
    hw.active[:] = [b[0], -1, b[2], b[3]]
    check(hw)


def test_empty_active_list_writes_nothing():
    hw = wl.host_world(wl.SHAPES["tiny_fp32"], seed=3)
    hw.active[:] = -1
    got = run_cuda(hw)
    for l in range(hw.L):
        assert got.state[l].tobytes() == hw.state[l].tobytes()


REDUCED = [
    ("mamba2_2p7b_fp32", dict(L=3, Bt=8, n_active=6)),
    ("hybrid48_bf16", dict(L=2, Bt=6, n_active=5)),
    ("hybrid48_int8", dict(L=2, Bt=4, n_active=3)),
    ("hybrid48_fp8_sr", dict(L=2, Bt=4, n_active=3)),
    ("ring_sweep_fp16", dict(L=2, Bt=6, n_active=6, prefix=("fixed", 16))),
]


@pytest.mark.parametrize("name,over", REDUCED, ids=[r[0] for r in REDUCED])
def test_named_workload_reduced(name, over):
    hw = wl.host_world(wl.SHAPES[name].replace(**over), seed=11)
    assert check(hw) >= 1


@pytest.mark.parametrize("k", [0, 1, 4, 16, 64])
def test_ring_sweep_prefix_lengths(k):
    shape = wl.SHAPES["ring_sweep_fp16"].replace(L=2, Bt=5, n_active=5, prefix=("fixed", k), pad_frac=0.2)
    hw = wl.host_world(shape, seed=100 + k)
    check(hw)


# ----------------------------------------------------------------------------
# every compiled instance
# ----------------------------------------------------------------------------

WIDE = [(sd, idt, d, n) for sd in ("f32", "bf16", "f16") for idt in ("bf16", "f32")
        for d, n in ((16, 16), (64, 64), (64, 128))]
BYTE = [(sd, idt, 64, 128) for sd in ("i8", "fp8_e4m3") for idt in ("bf16", "f32")]


@pytest.mark.parametrize("sd,idt,D,N", WIDE + BYTE, ids=lambda v: str(v))
def test_every_instance(sd, idt, D, N):
    shape = wl.Shape("inst", L=2, Bt=5, H=6, hpg=3, D=D, N=N, R=8, W=8, state_dtype=sd, input_dtype=idt,
                     n_active=4, ring_start=(0, 8), prefix=("uniform", 0, 8))
    hw = wl.host_world(shape, seed=zlib.crc32(repr((sd, idt, D, N)).encode()) % 1000)
    check(hw)


@pytest.mark.parametrize("sd,idt,D,N", WIDE + BYTE, ids=lambda v: str(v))
def test_every_instance_long_window(sd, idt, D, N):
    """A 40-token window: prefixes of up to 40 ring rows span up to three
    pipeline stages of 16 tokens, the last one ragged, with ring wrap."""
    shape = wl.Shape("instw", L=2, Bt=6, H=6, hpg=3, D=D, N=N, R=48, W=40, state_dtype=sd, input_dtype=idt,
                     n_active=5, ring_start=(0, 48), prefix=("uniform", 0, 40))
    hw = wl.host_world(shape, seed=zlib.crc32(repr(("w", sd, idt, D, N)).encode()) % 1000)
    hw.replay_prefix_len[int(hw.active[0])] = 40
    hw.replay_prefix_len[int(hw.active[1])] = 17
    check(hw)


@pytest.mark.parametrize("sd", ["bf16", "f16", "i8"])
def test_stochastic_rounding_long_window(sd):
    shape = wl.Shape("srw", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=64, W=64, state_dtype=sd, n_active=4,
                     ring_start=(0, 64), prefix=("uniform", 17, 64), philox_rounds=10, rand_seed=0xABCDEF)
    hw = wl.host_world(shape, seed=8)
    check(hw)


@pytest.mark.parametrize("sd", ["bf16", "f16", "i8", "fp8_e4m3"])
def test_stochastic_rounding_every_format(sd):
    shape = wl.Shape("sr", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype=sd, n_active=4,
                     philox_rounds=10, rand_seed=0x1234_5678_9ABC)
    hw = wl.host_world(shape, seed=7)
    check(hw)


@pytest.mark.parametrize("sd,W", [("bf16", 8), ("f16", 8), ("bf16", 16), ("f16", 16), ("i8", 8), ("fp8_e4m3", 8)])
def test_stochastic_rounding_matches_the_oracle_bit_for_bit(sd, W):
    """A replay that both sides compute exactly (A = 0, dt = 1/16, one token of
    bf16 inputs: S_1 = S_0 + x B^T / 16 with one fp32 rounding) isolates the
    rounding decisions.  16-bit state is bit-exact, on the CUDA cores (window 8)
    and on the tensor-core path (window 16); one-byte scales are bit-exact and
    codes may differ only where the kernel's product v * (qmax / amax) and the
    oracle's quotient v / scale straddle a decision (expected: almost never)."""
    L = 3
    shape = wl.Shape("srbits", L=L, Bt=2, H=4, hpg=2, D=64, N=128, R=W, W=W, state_dtype=sd, input_dtype="bf16",
                     n_active=2, pool=8, philox_rounds=10, rand_seed=0x0123_4567_89AB_CDEF)
    meta = dict(src_slots=np.stack([np.arange(L), np.full(L, 3)], 1).astype(np.int32),
                dst_slots=np.stack([7 - np.arange(L), np.full(L, 4)], 1).astype(np.int32),
                ring_start=np.array([1, W - 1], np.int32), replay_prefix_len=np.array([1, 1], np.int32),
                active=np.array([0, 1], np.int32), pool=8)
    hw = wl.host_world(shape, seed=404, metadata=meta)
    for l in range(L):
        hw.A[l][:] = 0.0
        hw.dt[l][:] = 0.0625
    got, ref = run_cuda(hw), run_oracle(hw)
    for (l, d), _ in written_dsts(hw).items():
        g, r = got.state[l][d], ref.state[l][d]
        if sd in ("bf16", "f16"):
            assert g.tobytes() == r.tobytes(), f"layer {l} slot {d}: {(g != r).mean():.2e} of the elements differ"
        else:
            assert got.scale[l][d].tobytes() == ref.scale[l][d].tobytes(), f"layer {l} slot {d}: scales"
            assert (g != r).mean() <= 1e-3, f"layer {l} slot {d}: {(g != r).mean():.2e} of the codes differ"


def test_stochastic_rounding_is_unbiased_over_seeds():
    """Over 48 seeds the bf16 outputs average to the unrounded result: the
    summed error, over 4096 elements and all seeds, is within 5 standard
    deviations of zero (each element's variance frac*(1-frac)*spacing^2)."""
    shape = wl.Shape("srstat", L=1, Bt=4, H=4, hpg=2, D=16, N=16, R=8, W=8, state_dtype="bf16", n_active=4,
                     prefix=("fixed", 4), philox_rounds=10, rand_seed=1)
    hw = wl.host_world(shape, seed=5)
    as_f32 = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32)
    # the unrounded result: the same call with the bf16 source decoded into an fp32 state
    hw32 = hw.copy()
    hw32.shape = shape.replace(state_dtype="f32", philox_rounds=0)
    hw32.state = [as_f32(a) for a in hw.state]
    oracle.materialize(hw32)
    dsts = [int(hw.dst_slots[0, b]) for b in hw.active if b >= 0]
    ref = np.stack([hw32.state[0][d] for d in dsts]).astype(np.float64)
    mag = np.abs(ref)
    spacing = np.exp2(np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 7)
    frac = mag / spacing - np.floor(mag / spacing)
    var = frac * (1 - frac) * spacing ** 2
    seeds = 48
    err = np.zeros_like(ref)
    for s in range(seeds):
        w = hw.copy()
        w.rand_seed = 1000 + s
        got = run_cuda(w)
        err += np.stack([as_f32(got.state[0][d]) for d in dsts]).astype(np.float64) - ref
    z = err.sum() / np.sqrt(seeds * var.sum())
    assert abs(z) < 5.0, z


@pytest.mark.parametrize("sd", ["bf16", "f16", "i8", "fp8_e4m3"])
@pytest.mark.parametrize("rounds", [0, 10])
def test_requantization_is_bit_exact_when_state_is_unchanged(sd, rounds):
    """dt = 0 makes the replay an identity in any precision, so the rewrite of the
    source state (RNE or stochastic: same words, same decisions) is bit-exact for
    16-bit state and for one-byte scales; one-byte codes are within one step, the
    one-code tolerance of one-byte state (tests/parity.py says why they may differ)."""
    shape = wl.Shape("dt0", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype=sd, n_active=4,
                     prefix=("uniform", 1, 8), philox_rounds=rounds, rand_seed=0x5EED)
    hw = wl.host_world(shape, seed=9)
    for a in hw.dt:
        a[:] = 0.0
    check(hw, exact=True)


@pytest.mark.parametrize("sd", ["i8", "fp8_e4m3"])
@pytest.mark.parametrize("rounds", [0, 10])
def test_one_byte_rows_without_a_finite_scale_become_zero(sd, rounds):
    """A row that replays to exact zeros (zero codes, zero x) and a row that
    replays to fp32 subnormals (zero codes, x ~ 1e-38): qmax/amax is not finite
    for both, so both are written as zero codes (+0 for fp8) with scale 0, on
    either rounding path; the other rows of the tile are ordinary."""
    shape = wl.Shape("zrow", L=1, Bt=4, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype=sd, n_active=4,
                     prefix=("fixed", 5), philox_rounds=rounds, rand_seed=0x5EED)
    hw = wl.host_world(shape, seed=61)
    b = int(hw.active[0])
    src, dst = int(hw.src_slots[0, b]), int(hw.dst_slots[0, b])
    h, zero_row, tiny_row = 1, 5, 9
    hw.state[0][src, h, zero_row, :] = 0
    hw.state[0][src, h, tiny_row, :] = 0
    hw.x[0][src, :, h, zero_row] = 0
    hw.x[0][src, :, h, tiny_row] = wl.bf16_bits_from_f32(np.full(shape.R, 1e-38, np.float32))
    got, ref = run_cuda(hw), run_oracle(hw)
    for w in (got, ref):
        for r in (zero_row, tiny_row):
            assert not w.state[0][dst, h, r].any(), f"row {r}: codes not zero"
            assert w.scale[0][dst, h, r] == 0.0, f"row {r}: scale not zero"
        assert w.state[0][dst, h, 0].any()
    compare_worlds(got, ref, hw)


# ----------------------------------------------------------------------------
# edge cases
# ----------------------------------------------------------------------------

def _offset_copy(a: np.ndarray, offset_elems: int) -> np.ndarray:
    """Same contents, stored `offset_elems` elements past an aligned base."""
    buf = np.zeros(a.size + offset_elems, dtype=a.dtype)
    v = buf[offset_elems:].reshape(a.shape)
    v[...] = a
    return v


def test_misaligned_state_and_ring_take_the_byte_path():
    shape = wl.Shape("mis", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype="bf16", n_active=4)
    hw = wl.host_world(shape, seed=21)
    hw.state[0] = _offset_copy(hw.state[0], 1)   # 2-byte offset: source and destination tiles misaligned
    hw.x[1] = _offset_copy(hw.x[1], 1)           # ring rows misaligned in layer 1
    # device copies keep the offset: build the device world by hand
    dw = wl.device_world_from_host(hw)
    for l, arr in ((0, hw.state[0]),):
        buf = torch.zeros(arr.size + 1, dtype=torch.int16, device="cuda")
        view = buf[1:].view(arr.shape)
        view.copy_(torch.from_numpy(arr.view(np.int16).copy()))
        dw.state[l] = view
    buf = torch.zeros(hw.x[1].size + 1, dtype=torch.int16, device="cuda")
    xv = buf[1:].view(hw.x[1].shape)
    xv.copy_(torch.from_numpy(hw.x[1].view(np.int16).copy()))
    dw.x[1] = xv
    dw.tables = wl._tables(dw.state, dw.scale, dw.x, dw.B, dw.dt, dw.A, "cuda")
    assert dw.state[0].data_ptr() % 16 == 2
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    compare_worlds(got, run_oracle(hw), hw)


def test_misaligned_ring_long_window():
    """Byte-copy path over several stages: misaligned B rows, prefixes up to 48."""
    shape = wl.Shape("misw", L=1, Bt=4, H=4, hpg=2, D=64, N=128, R=64, W=48, state_dtype="f16", n_active=4,
                     ring_start=(0, 64), prefix=("uniform", 10, 48))
    hw = wl.host_world(shape, seed=23)
    hw.B[0] = _offset_copy(hw.B[0], 1)
    dw = wl.device_world_from_host(hw)
    buf = torch.zeros(hw.B[0].size + 1, dtype=torch.int16, device="cuda")
    bv = buf[1:].view(hw.B[0].shape)
    bv.copy_(torch.from_numpy(hw.B[0].view(np.int16).copy()))
    dw.B[0] = bv
    dw.tables = wl._tables(dw.state, dw.scale, dw.x, dw.B, dw.dt, dw.A, "cuda")
    assert dw.B[0].data_ptr() % 16 == 2
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    compare_worlds(got, run_oracle(hw), hw)


def test_misaligned_scales():
    shape = wl.Shape("mis8", L=1, Bt=3, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype="i8", n_active=3)
    hw = wl.host_world(shape, seed=22)
    dw = wl.device_world_from_host(hw)
    sc = hw.scale[0]
    buf = torch.zeros(sc.size + 1, dtype=torch.float32, device="cuda")
    v = buf[1:].view(sc.shape)
    v.copy_(torch.from_numpy(sc))
    dw.scale[0] = v
    dw.tables = wl._tables(dw.state, dw.scale, dw.x, dw.B, dw.dt, dw.A, "cuda")
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t) for t in dw.state]
    got.scale = [wl._to_np(t) for t in dw.scale]
    compare_worlds(got, run_oracle(hw), hw)


def test_pad_slot_id_zero():
    """With pad_slot_id = 0, slot 0 is the sentinel and -1 is not."""
    shape = wl.SHAPES["tiny_fp32"].replace(pad_slot_id=0, special="")
    hw = wl.host_world(shape, seed=31)
    hw.src_slots[0, int(hw.active[0])] = 0
    assert (0, int(hw.dst_slots[0, int(hw.active[0])])) not in written_dsts(hw)
    check(hw)


@pytest.mark.parametrize("bad,bit", [("prefix", 4), ("ring_start", 2), ("active", 1), ("slot", 8)])
def test_out_of_range_metadata_is_skipped_and_flagged(bad, bit):
    shape = wl.Shape("bad", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype="bf16", n_active=4)
    hw = wl.host_world(shape, seed=41)
    victim = int(hw.active[1])
    if bad == "prefix":
        hw.replay_prefix_len[victim] = shape.W + 1
    elif bad == "ring_start":
        hw.ring_start[victim] = shape.R
    elif bad == "active":
        hw.active[1] = shape.Bt + 5
    else:
        hw.src_slots[0, victim] = -7
    got = run_cuda(hw, status_expected=bit)
    # reference: the oracle without the offending entry
    ref_in = hw.copy()
    if bad == "slot":
        ref_in.dst_slots[0, victim] = ref_in.pad_slot_id
        ref_in.src_slots[0, victim] = 0
    else:
        keep = [a for i, a in enumerate(hw.active) if i != 1]
        ref_in.active[:] = keep + [-1]
        if bad != "active":
            ref_in.replay_prefix_len[victim] = 0
            ref_in.ring_start[victim] = 0
    compare_worlds(got, run_oracle(ref_in), ref_in)


@pytest.mark.parametrize("side", ["dst", "src"])
@pytest.mark.parametrize("window", [8, 64], ids=["cuda_cores", "tensor_cores"])
def test_slot_past_the_stated_pool_is_skipped_and_flagged(side, window):
    """With num_slots stated, a slot at or past it is skipped and flagged
    (RSM_STATUS_BAD_SLOT) instead of addressed.  The call states a pool one slot
    shorter than the allocation and uses that last, unused slot, so that nothing
    outside the buffers could be touched even if the check were missing."""
    shape = wl.Shape("pastpool", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=window, W=window, state_dtype="bf16",
                     n_active=4, pool=10, ring_start=(0, window), prefix=("uniform", 1, window))
    hw = wl.host_world(shape, seed=43)
    last = hw.state[0].shape[0] - 1
    used = list(hw.dst_slots[0])
    if last in used:  # free the last slot: hand its request the destination slot nobody uses
        spare = next(d for d in range(hw.state[0].shape[0] // 2, last) if d not in used)
        hw.dst_slots[0, used.index(last)] = spare
    victim = int(hw.active[1])
    if side == "dst":
        hw.dst_slots[0, victim] = last
    else:
        hw.src_slots[0, victim] = last
    dw = wl.device_world_from_host(hw)
    kw = dw.call_kwargs()
    kw["num_slots"] = last
    rsm.replayssm_materialize(**kw)
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 8
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    ref_in = hw.copy()
    ref_in.dst_slots[0, victim] = ref_in.pad_slot_id
    compare_worlds(got, run_oracle(ref_in), ref_in)
    assert bool((wl._to_np(dw.state[0][last]).view(np.uint8) == 0xFF).all())


@pytest.mark.parametrize("sd", ["f32", "bf16", "fp8_e4m3"])
def test_in_place_commit(sd):
    """dst_slots == src_slots: the prefix is committed into the source slots."""
    shape = wl.Shape("inplace", L=2, Bt=5, H=6, hpg=3, D=64, N=128, R=8, W=8, state_dtype=sd,
                     input_dtype="f32" if sd == "f32" else "bf16", n_active=4, philox_rounds=3 if sd == "fp8_e4m3" else 0,
                     rand_seed=5)
    hw = wl.host_world(shape, seed=71)
    hw.dst_slots[:] = hw.src_slots
    assert check(hw) >= 4


def test_repeated_calls_are_identical():
    shape = wl.Shape("rep", L=2, Bt=4, H=8, hpg=4, D=64, N=128, R=8, W=8, state_dtype="fp8_e4m3", n_active=4,
                     philox_rounds=7, rand_seed=99)
    hw = wl.host_world(shape, seed=51)
    a = run_cuda(hw)
    b = run_cuda(hw)
    for l in range(hw.L):
        assert a.state[l].tobytes() == b.state[l].tobytes()
        assert a.scale[l].tobytes() == b.scale[l].tobytes()


def test_prepared_call_replays_from_a_cuda_graph():
    """The call enqueues one kernel and nothing else (no allocation, no copy,
    no host sync), so a prepared call can be captured in a CUDA graph: the
    capture writes nothing, and a replay writes what the oracle writes."""
    shape = wl.Shape("graph", L=2, Bt=5, H=6, hpg=3, D=64, N=128, R=8, W=8, state_dtype="bf16", n_active=4,
                     prefix=("uniform", 0, 8))
    hw = wl.host_world(shape, seed=123)
    warm = wl.device_world_from_host(hw)  # the host-side launch plan is set up outside the capture
    rsm.prepare(**warm.call_kwargs())()
    torch.cuda.synchronize()
    dw = wl.device_world_from_host(hw)
    call = rsm.prepare(**dw.call_kwargs())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    for l in range(hw.L):
        assert wl._to_np(dw.state[l]).tobytes() == hw.state[l].tobytes(), "capture must not run the kernel"
    g.replay()
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    compare_worlds(got, run_oracle(hw), hw)


# ----------------------------------------------------------------------------
# full size: the 48-layer x 256-head x 64x128 bf16 call that the benchmark times
# ----------------------------------------------------------------------------

def _unwritten_destinations_untouched(dw, shape, n):
    """On the device: every destination-half slot of every layer that no
    selected (layer, request) writes is still the 0xFF sentinel."""
    active = dw.active.cpu().numpy()[:n]
    src, dst = dw.src_slots.cpu().numpy(), dw.dst_slots.cpu().numpy()
    pad, half = shape.pad_slot_id, dw.pool // 2
    checked = 0
    for l in range(shape.L):
        written = {int(dst[l, b]) for b in active if src[l, b] != pad and dst[l, b] != pad}
        idle = [d for d in range(half, dw.pool) if d not in written]
        if idle:
            idx = torch.tensor(idle, device=dw.state[l].device)
            assert bool((dw.state[l].index_select(0, idx).view(torch.uint8) == 0xFF).all()), f"layer {l}"
            checked += len(idle)
    return checked


@pytest.mark.slow
@pytest.mark.parametrize("variant", ["bench", "pads_and_terminator"])
def test_headline_full_size_sampled(variant):
    """The 48-layer x 256-head x 64x128 bf16 call at full size: as the
    benchmark times it (all 256 requests active), and with 200 active requests
    before the -1s and 10% of the (layer, request) entries padded.  Sampled
    (layer, request) outputs are recomputed by the oracle one by one; every
    prefix-0 request is a byte copy; every destination slot that nothing
    writes keeps its sentinel."""
    shape = wl.SHAPES["hybrid48_bf16"]
    if variant == "pads_and_terminator":
        shape = shape.replace(n_active=200, pad_frac=0.10)
    dw = wl.device_world_random(shape, seed=0)
    cfg = rsm.launch_config(**dw.call_kwargs())
    assert cfg["grid"] > 0
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    n = shape.n_active
    active = dw.active.cpu().numpy()
    assert (active[n:] == -1).all() and (active[:n] >= 0).all()
    live = active[:n]
    prefix = dw.replay_prefix_len.cpu().numpy()
    src = dw.src_slots.cpu().numpy()
    dst = dw.dst_slots.cpu().numpy()
    pad = shape.pad_slot_id
    rng = np.random.default_rng(5)
    # property at full size: every prefix-0 request is a bit-exact copy in every unpadded layer
    zero = [int(b) for b in live if prefix[b] == 0]
    for b in zero[:8]:
        for l in range(shape.L):
            if src[l, b] != pad and dst[l, b] != pad:
                assert torch.equal(dw.state[l][dst[l, b]], dw.state[l][src[l, b]])
    idle = _unwritten_destinations_untouched(dw, shape, n)
    if variant == "pads_and_terminator":
        assert idle >= shape.L * (shape.Bt - n)
    # sampled outputs, each recomputed by the oracle from its own inputs
    want = 12 if variant == "bench" else 32
    picks, tries = [], 0
    while len(picks) < want and tries < 10 * want:
        l, b = int(rng.integers(shape.L)), int(live[int(rng.integers(n))])
        tries += 1
        if src[l, b] != pad and dst[l, b] != pad and (l, b) not in picks:
            picks.append((l, b))
    picks.append((shape.L - 1, int(live[-1])))
    checked = 0
    for l, b in picks:
        if src[l, b] == pad or dst[l, b] == pad:
            continue
        sub = wl.host_subworld(dw, l, b)
        oracle.materialize(sub)
        got = wl._to_np(dw.state[l][dst[l, b]])
        ref = sub.state[0][1]
        if prefix[b] == 0:
            assert got.tobytes() == ref.tobytes()
        else:
            compare_slot(got, ref, "bf16", where=f"layer {l} request {b}")
        checked += 1
    assert checked >= want
    del dw
    torch.cuda.empty_cache()


FULL = [
    ("hybrid48_int8", {}),
    ("hybrid48_int8", {"state_dtype": "fp8_e4m3"}),
    ("mamba2_2p7b_fp32", {}),
    ("ring_sweep_fp16", {"prefix": ("fixed", 16)}),
    ("ring_sweep_fp16", {"prefix": ("fixed", 64)}),
    ("hybrid48_fp8_sr", {}),
]


@pytest.mark.slow
@pytest.mark.parametrize("name,over", FULL, ids=["int8", "fp8_rne", "mamba2_fp32", "ring_k16", "ring_k64", "fp8_sr"])
def test_named_workload_full_size_sampled(name, over):
    """The benchmark's other workloads at full size and in its launch
    configuration (one-byte state, fp32 state with ring wrap, the 64-token
    window on the tensor cores), checked on sampled (layer, request) outputs
    that the oracle recomputes one by one (with stochastic rounding, from the
    Philox words of the call's own destination slot and layer), and on the
    bytes of pads."""
    shape = wl.SHAPES[name].replace(**over)
    dw = wl.device_world_random(shape, seed=3)
    rsm.prepare(**dw.call_kwargs())()   # the prepared call the bench times
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    n = shape.n_active
    live = dw.active.cpu().numpy()[:n]
    prefix = dw.replay_prefix_len.cpu().numpy()
    src = dw.src_slots.cpu().numpy()
    dst = dw.dst_slots.cpu().numpy()
    pad = shape.pad_slot_id
    sd = shape.state_dtype
    rng = np.random.default_rng(7)
    picks = [(int(rng.integers(shape.L)), int(live[int(rng.integers(n))])) for _ in range(6)]
    picks.append((shape.L - 1, int(live[-1])))
    checked = 0
    for l, b in picks:
        if src[l, b] == pad or dst[l, b] == pad:
            continue
        sub = wl.host_subworld(dw, l, b)
        oracle.materialize(sub)
        got = wl._to_np(dw.state[l][dst[l, b]])
        ref = sub.state[0][1]
        gs = None if dw.scale[l] is None else wl._to_np(dw.scale[l][dst[l, b]])
        rs = None if sub.scale[0] is None else sub.scale[0][1]
        if prefix[b] == 0:
            assert got.tobytes() == ref.tobytes()
            assert gs is None or gs.tobytes() == rs.tobytes()
        else:
            compare_slot(got, ref, sd, gs, rs, where=f"{name} layer {l} request {b}")
        checked += 1
    assert checked >= 4
    # a destination whose (layer, request) is padded on the source side stays as it was (0xFF)
    for l in range(shape.L):
        for b in live[:16]:
            if src[l, b] == pad and dst[l, b] != pad:
                assert bool((dw.state[l][dst[l, b]].view(torch.uint8) == 0xFF).all())
    del dw
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------
# long windows: the tensor-core path (16-bit state, bf16 inputs, 64 x 128,
# windows of 16 or more; every replayed prefix goes through the MMA)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("sd", ["bf16", "f16"])
@pytest.mark.parametrize("k", [6, 7, 9, 10, 15, 17, 31, 33, 63])
def test_tensor_core_prefix_lengths(sd, k):
    shape = wl.Shape("tc", L=2, Bt=4, H=8, hpg=4, D=64, N=128, R=64, W=64, state_dtype=sd, n_active=4,
                     ring_start=(0, 64), prefix=("fixed", k))
    hw = wl.host_world(shape, seed=300 + k)
    check(hw)


@pytest.mark.parametrize("sd", ["bf16", "f16"])
def test_tensor_core_mixed_prefixes_many_units_per_cta(sd):
    """Prefixes U[0,64] over ~3 (request, layer, head-run) units per CTA:
    copies, CUDA-core items and tensor-core items follow one another inside a
    CTA, the tensor-core items alternate between the two consumer groups, and
    B^T is reused across groups within a B group."""
    shape = wl.Shape("tcmix", L=2, Bt=64, H=32, hpg=8, D=64, N=128, R=64, W=64, state_dtype=sd, n_active=60,
                     ring_start=(0, 64), prefix=("uniform", 0, 64), pad_frac=0.05)
    hw = wl.host_world(shape, seed=91)
    for i in (3, 17):  # two exact copies among them
        hw.replay_prefix_len[int(hw.active[i])] = 0
    k = np.asarray(hw.replay_prefix_len)[np.asarray(hw.active)[:60]]
    assert (k == 0).any() and ((k > 0) & (k < 7)).any() and (k >= 7).any()
    assert check(hw) >= 100


def test_tensor_core_misaligned_destination():
    """Destination tiles 2 bytes off a 16-byte boundary: the staged tile is
    written with byte stores."""
    shape = wl.Shape("tcmis", L=1, Bt=3, H=4, hpg=2, D=64, N=128, R=64, W=64, state_dtype="f16", n_active=3,
                     ring_start=(0, 64), prefix=("uniform", 10, 64))
    hw = wl.host_world(shape, seed=24)
    hw.state[0] = _offset_copy(hw.state[0], 1)
    dw = wl.device_world_from_host(hw)
    buf = torch.zeros(hw.state[0].size + 1, dtype=torch.float16, device="cuda")
    view = buf[1:].view(hw.state[0].shape)
    view.copy_(torch.from_numpy(hw.state[0]))
    dw.state[0] = view
    dw.tables = wl._tables(dw.state, dw.scale, dw.x, dw.B, dw.dt, dw.A, "cuda")
    assert dw.state[0].data_ptr() % 16 == 2
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    compare_worlds(got, run_oracle(hw), hw)


@pytest.mark.parametrize("bad,bit", [("prefix", 4), ("ring_start", 2), ("active", 1), ("slot", 8)])
def test_tensor_core_out_of_range_metadata_is_skipped_and_flagged(bad, bit):
    shape = wl.Shape("tcbad", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=64, W=64, state_dtype="bf16", n_active=4,
                     ring_start=(0, 64), prefix=("uniform", 12, 64))
    hw = wl.host_world(shape, seed=42)
    victim = int(hw.active[1])
    if bad == "prefix":
        hw.replay_prefix_len[victim] = shape.W + 1
    elif bad == "ring_start":
        hw.ring_start[victim] = shape.R
    elif bad == "active":
        hw.active[1] = shape.Bt + 5
    else:
        hw.src_slots[0, victim] = -7
    got = run_cuda(hw, status_expected=bit)
    ref_in = hw.copy()
    if bad == "slot":
        ref_in.dst_slots[0, victim] = ref_in.pad_slot_id
        ref_in.src_slots[0, victim] = 0
    else:
        keep = [a for i, a in enumerate(hw.active) if i != 1]
        ref_in.active[:] = keep + [-1]
        if bad != "active":
            ref_in.replay_prefix_len[victim] = 0
            ref_in.ring_start[victim] = 0
    compare_worlds(got, run_oracle(ref_in), ref_in)


def _bf16_bits_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tc_f16_error_report(hw, got, ref):
    """fp16 state on the tensor cores: per written slot, |gpu - oracle| against
    one fp16 ulp plus 2^-13 (sum_t dt_t |x_t[i]| |B_t[j]| + |S0[i][j]|).

    With C = w x split into bf16 hi + lo (16 significant bits a term, the
    decay weights and P in fp32, fp32 accumulation) the error before the final
    rounding stays below 2^-14.4 of that sum, so the result is within one ulp
    plus the sum's term; C rounded to a single bf16 operand (2^-9 a term)
    leaves several ulps on long prefixes.  Returns (max |err|, max err/allow,
    fraction of elements that differ from the oracle)."""
    H, hpg = hw.H, hw.hpg
    worst, ratio, diff, n = 0.0, 0.0, 0, 0
    for (l, d), (b, k) in written_dsts(hw).items():
        if k == 0:
            continue
        src = int(hw.src_slots[l, b])
        pos = (int(hw.ring_start[b]) + np.arange(k)) % hw.R
        x = np.abs(_bf16_bits_to_f64(hw.x[l][src][pos]))                      # (k, H, D)
        B = np.abs(_bf16_bits_to_f64(hw.B[l][src][pos]))[:, np.arange(H) // hpg]  # (k, H, N)
        dt = hw.dt[l][src][pos].astype(np.float64)                            # (k, H)
        s0 = np.abs(hw.state[l][src].astype(np.float64))                      # (H, D, N)
        terms = np.einsum("th,thi,thj->hij", dt, x, B)
        g = got.state[l][d].astype(np.float64)
        r = ref.state[l][d].astype(np.float64)
        ulp = np.maximum(np.spacing(np.abs(g).astype(np.float16)), np.spacing(np.abs(r).astype(np.float16)))
        allow = ulp.astype(np.float64) + 2.0 ** -13 * (terms + s0)
        err = np.abs(g - r)
        worst = max(worst, float(err.max()))
        ratio = max(ratio, float((err / allow).max()))
        diff += int((g != r).sum())
        n += g.size
    return worst, ratio, diff / max(n, 1)


@pytest.mark.parametrize("k", [16, 33, 64])
def test_tensor_core_fp16_state_error_bound(k):
    """fp16 state: every element within one fp16 ulp of the oracle plus
    2^-13 of the replayed terms' magnitudes (tc_f16_error_report)."""
    shape = wl.Shape("tcprec", L=2, Bt=4, H=32, hpg=16, D=64, N=128, R=64, W=64, state_dtype="f16",
                     n_active=4, ring_start=(0, 64), prefix=("fixed", k))
    hw = wl.host_world(shape, seed=700 + k)
    got, ref = run_cuda(hw), run_oracle(hw)
    worst, ratio, frac = tc_f16_error_report(hw, got, ref)
    print(f"fp16 tensor cores, k={k}: max |err| {worst:.3e}, max err/allow {ratio:.3f}, {frac:.2%} differ")
    assert ratio <= 1.0
    compare_worlds(got, ref, hw)


@pytest.mark.parametrize("sd,hpg", [("f16", 1), ("bf16", 1), ("f16", 2)])
def test_tensor_core_launch_plan_and_single_head_groups(sd, hpg):
    """Groups of one head: every item carries its B rows, so two 64-token
    items need 82 KB of arena.  fp16 state (with its 16 KB hi + lo operand)
    then plans one CTA per SM with the whole shared memory, bf16 state two;
    groups of two heads fit two CTAs per SM in both formats.  Results match
    the oracle in every plan."""
    shape = wl.Shape("tcplan", L=2, Bt=4, H=8, hpg=hpg, D=64, N=128, R=64, W=64, state_dtype=sd, n_active=4,
                     ring_start=(0, 64), prefix=("uniform", 40, 64))
    hw = wl.host_world(shape, seed=37 + hpg)
    kw = wl.device_world_from_host(hw).call_kwargs()
    assert rsm.kernel_name(**kw) == "materialize_tc_kernel"
    cfg = rsm.launch_config(**kw)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one_cta = sd == "f16" and hpg == 1
    assert cfg["grid"] == (sms if one_cta else 2 * sms), cfg
    check(hw)


@pytest.mark.parametrize("sd", ["bf16", "f16"])
def test_tensor_core_in_place_commit(sd):
    shape = wl.Shape("tcinplace", L=2, Bt=5, H=6, hpg=3, D=64, N=128, R=64, W=64, state_dtype=sd, n_active=4,
                     ring_start=(0, 64), prefix=("uniform", 0, 64))
    hw = wl.host_world(shape, seed=73)
    hw.dst_slots[:] = hw.src_slots
    assert check(hw) >= 4


def test_tensor_core_empty_active_list_writes_nothing():
    shape = wl.Shape("tcempty", L=2, Bt=4, H=4, hpg=2, D=64, N=128, R=64, W=64, state_dtype="bf16", n_active=0,
                     ring_start=(0, 64), prefix=("uniform", 10, 64))
    hw = wl.host_world(shape, seed=74)
    hw.active[:] = -1
    got = run_cuda(hw)
    for l in range(hw.L):
        assert got.state[l].tobytes() == hw.state[l].tobytes()


# ----------------------------------------------------------------------------
# one-byte state on the tensor cores (int8 / fp8 state, bf16 inputs, an even
# number of heads per B group: items of two heads, the replay as MMAs)
# ----------------------------------------------------------------------------

def _q8tc_world(shape, seed):
    hw = wl.host_world(shape, seed=seed)
    assert rsm.kernel_name(**wl.device_world_from_host(hw).call_kwargs()) == "materialize_q8tc_kernel"
    return hw


@pytest.mark.parametrize("sd", ["i8", "fp8_e4m3"])
@pytest.mark.parametrize("k", [1, 5, 8, 15, 16, 17, 33, 64])
def test_one_byte_tensor_core_prefix_lengths(sd, k):
    """Whole MMAs (16, 64), ragged last ones and a single token, with ring wrap."""
    shape = wl.Shape("q8tc", L=2, Bt=4, H=8, hpg=4, D=64, N=128, R=64, W=64, state_dtype=sd, n_active=4,
                     ring_start=(0, 64), prefix=("fixed", k))
    check(_q8tc_world(shape, seed=500 + k))


@pytest.mark.parametrize("sd", ["i8", "fp8_e4m3"])
@pytest.mark.parametrize("rounds", [0, 10])
def test_one_byte_tensor_core_mixed_prefixes_many_units_per_cta(sd, rounds):
    """Prefixes U[0,8] over several (request, layer, head-run) units per CTA:
    copies and replays follow one another, items alternate between the two
    accumulators, and the B operand is reused along each B group."""
    shape = wl.Shape("q8tcmix", L=2, Bt=48, H=32, hpg=8, D=64, N=128, R=8, W=8, state_dtype=sd, n_active=44,
                     prefix=("uniform", 0, 8), pad_frac=0.05, philox_rounds=rounds, rand_seed=0xC0FFEE)
    hw = _q8tc_world(shape, seed=92)
    for i in (2, 11):  # two exact copies among them
        hw.replay_prefix_len[int(hw.active[i])] = 0
    assert check(hw) >= 60


@pytest.mark.parametrize("sd", ["i8", "fp8_e4m3"])
def test_one_byte_tensor_core_misaligned_state(sd):
    """Codes one byte off a 16-byte boundary: the loader copies the tiles
    byte-wise and the epilogue writes them with byte stores."""
    shape = wl.Shape("q8tcmis", L=1, Bt=3, H=4, hpg=2, D=64, N=128, R=8, W=8, state_dtype=sd, n_active=3)
    hw = _q8tc_world(shape, seed=25)
    dw = wl.device_world_from_host(hw)
    buf = torch.zeros(hw.state[0].size + 1, dtype=torch.uint8, device="cuda")
    view = buf[1:].view(hw.state[0].shape)
    view.copy_(torch.from_numpy(hw.state[0].view(np.uint8)))
    dw.state[0] = view
    dw.tables = wl._tables(dw.state, dw.scale, dw.x, dw.B, dw.dt, dw.A, "cuda")
    assert dw.state[0].data_ptr() % 16 == 1
    rsm.replayssm_materialize(**dw.call_kwargs())
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(dw.state, hw.state)]
    got.scale = [wl._to_np(t) for t in dw.scale]
    compare_worlds(got, run_oracle(hw), hw)


@pytest.mark.parametrize("sd", ["i8", "fp8_e4m3"])
def test_one_byte_tensor_core_in_place_commit(sd):
    shape = wl.Shape("q8tcinplace", L=2, Bt=5, H=6, hpg=2, D=64, N=128, R=8, W=8, state_dtype=sd, n_active=4,
                     philox_rounds=10 if sd == "fp8_e4m3" else 0, rand_seed=5)
    hw = _q8tc_world(shape, seed=72)
    hw.dst_slots[:] = hw.src_slots
    assert check(hw) >= 4


@pytest.mark.parametrize("sd", ["i8", "fp8_e4m3"])
@pytest.mark.parametrize("idt,hpg", [("f32", 2), ("bf16", 3)])
@pytest.mark.parametrize("rounds", [0, 10])
def test_one_byte_cuda_core_kernel(sd, idt, hpg, rounds):
    """fp32 inputs, or B groups of an odd number of heads, keep one-byte state on
    the CUDA-core kernel, with both rounding modes."""
    shape = wl.Shape("q8cc", L=2, Bt=5, H=6, hpg=hpg, D=64, N=128, R=8, W=8, state_dtype=sd, input_dtype=idt,
                     n_active=4, prefix=("uniform", 0, 8), philox_rounds=rounds, rand_seed=0xBEEF)
    hw = wl.host_world(shape, seed=93)
    assert rsm.kernel_name(**wl.device_world_from_host(hw).call_kwargs()) == "materialize_q8_kernel"
    check(hw)
