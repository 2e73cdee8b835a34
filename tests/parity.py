"""Element-by-element comparison of a CUDA result against the oracle's.

Tolerances (the |gpu - ref| <= tol + tol*|ref| form):
  f32 state        tol = 1e-5
  bf16 / f16 state tol = 2e-2
  int8 / fp8 codes within one code step (ordered code distance <= 1); scales
                   within the fp32 tolerance
Slots that are not written (pads, entries after the first -1, untouched pool
slots) and prefix-0 copies must be bit-identical.

One-byte codes: the oracle rounds the plain quotient v / scale, the kernel the
product v * (qmax / amax); the two differ by an fp32 ulp at most, which moves a
code by one step only when the quotient sits next to a rounding boundary.  So
where the state itself is exact (compare_worlds(exact=True): the replay is an
identity and v is the decoded source), a code may differ by one step only
where the quotient lies within two fp32 ulps of a boundary of round-to-nearest
(a half-integer for int8, a midpoint of the fp8 grid); with stochastic
rounding, where the boundary is drawn at random, at most 0.1% of codes may
differ.
"""
import numpy as np

TOL = {"f32": 1e-5, "bf16": 2e-2, "f16": 2e-2}


def _as_float(arr, sd):
    if sd == "f32":
        return arr.astype(np.float64)
    if sd == "f16":
        return arr.astype(np.float64)
    if sd == "bf16":
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(sd)


def _ordered_code(arr, sd):
    if sd == "i8":
        return arr.astype(np.int64)
    c = arr.astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _fp8_grid():
    import torch
    v = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    return np.unique(v)


def _decode_codes(arr, sd):
    if sd == "i8":
        return arr.astype(np.float32)
    import torch
    return torch.from_numpy(arr.copy()).view(torch.float8_e4m3fn).float().numpy()


def _near_rne_boundary(y, sd):
    """|y| within two fp32 ulps of a round-to-nearest boundary of the format."""
    a = np.abs(y.astype(np.float64))
    if sd == "i8":
        bnd = np.floor(a) + 0.5
    else:
        grid = _fp8_grid()
        hi = np.clip(np.searchsorted(grid, a), 1, len(grid) - 1)
        bnd = (grid[hi - 1] + grid[hi]) / 2
    return np.abs(a - bnd) <= 2.0 ** -22 * np.maximum(a, 2.0 ** -126)


def written_dsts(world):
    """{(layer, dst_slot): (request, k)} for every (layer, request) the call writes."""
    out = {}
    for i in range(world.Bt):
        b = int(world.active[i])
        if b == -1:
            break
        for l in range(world.L):
            s, d = int(world.src_slots[l, b]), int(world.dst_slots[l, b])
            if s == world.pad_slot_id or d == world.pad_slot_id:
                continue
            out[(l, d)] = (b, int(world.replay_prefix_len[b]))
    return out


def compare_slot(got_state, ref_state, sd, got_scale=None, ref_scale=None, where=""):
    """One written destination slot: tolerance for state (and scales)."""
    if sd in ("f32", "bf16", "f16"):
        g, r = _as_float(got_state, sd), _as_float(ref_state, sd)
        tol = TOL[sd]
        err = np.abs(g - r)
        bound = tol + tol * np.abs(r)
        bad = ~(err <= bound)
        assert not bad.any(), (f"{where}: {bad.sum()} elements out of tolerance, max err {np.nanmax(err):.3e}, "
                               f"first at {np.argwhere(bad)[0].tolist()}")
    else:
        dg, dr = _ordered_code(got_state, sd), _ordered_code(ref_state, sd)
        dist = np.abs(dg - dr)
        assert dist.max() <= 1, f"{where}: code distance {dist.max()} at {np.argwhere(dist > 1)[0].tolist()}"
        err = np.abs(got_scale.astype(np.float64) - ref_scale.astype(np.float64))
        assert np.all(err <= 1e-5 + 1e-5 * np.abs(ref_scale)), f"{where}: scale error {err.max():.3e}"


def compare_worlds(got, ref, before, exact=False):
    """got: world after the CUDA call (host copies); ref: after the oracle;
    before: the inputs.  Every slot of every layer is checked."""
    sd = ref.state_dtype
    written = written_dsts(before)
    n_written = 0
    for l in range(ref.L):
        pool = ref.state[l].shape[0]
        for slot in range(pool):
            g, r = got.state[l][slot], ref.state[l][slot]
            gs = got.scale[l][slot] if got.scale[l] is not None else None
            rs = ref.scale[l][slot] if ref.scale[l] is not None else None
            key = (l, slot)
            if key in written and written[key][1] > 0 and not exact:
                compare_slot(g, r, sd, gs, rs, where=f"layer {l} slot {slot}")
                n_written += 1
            elif key in written and written[key][1] > 0 and sd in ("i8", "fp8_e4m3"):
                assert gs.tobytes() == rs.tobytes(), f"layer {l} slot {slot}: scale bytes differ"
                dist = np.abs(_ordered_code(g, sd) - _ordered_code(r, sd))
                assert dist.max() <= 1, f"layer {l} slot {slot}: code distance {dist.max()}"
                if before.philox_rounds > 0:
                    assert (dist > 0).mean() <= 1e-3, f"layer {l} slot {slot}: {(dist > 0).mean():.2e} differ"
                elif dist.any():
                    src = int(before.src_slots[l, written[key][0]])
                    v = (_decode_codes(before.state[l][src], sd) * before.scale[l][src][..., None]).astype(np.float32)
                    with np.errstate(divide="ignore", invalid="ignore"):
                        y = (v / rs[..., None]).astype(np.float32)
                    off = dist > 0
                    assert _near_rne_boundary(y[off], sd).all(), \
                        f"layer {l} slot {slot}: a code differs away from a rounding boundary"
                n_written += 1
            else:
                assert g.tobytes() == r.tobytes(), f"layer {l} slot {slot}: bytes differ (copy/untouched)"
                if gs is not None:
                    assert gs.tobytes() == rs.tobytes(), f"layer {l} slot {slot}: scale bytes differ"
                if key in written:
                    n_written += 1
    return n_written
