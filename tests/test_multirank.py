"""The N > 1 path on CPU: two gloo ranks each materialize their own shard of a
batch (no data-path collective), and the union of their outputs equals the
single-process result.  Also checks the measurement reductions the benchmark
uses across ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as td  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from mamba_replayssm_state_gb300 import dist  # noqa: E402
from mamba_replayssm_state_gb300 import workloads as wl  # noqa: E402

SHAPE = wl.Shape("dp", L=2, Bt=7, H=4, hpg=2, D=16, N=16, R=8, W=8, state_dtype="f32", input_dtype="f32",
                 n_active=6, ring_start=(0, 8), prefix=("uniform", 0, 8))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def slice_requests(hw, start, end):
    """The world of requests [start, end) as a rank holds it: local batch
    indices, same pools."""
    w = hw.copy()
    w.shape = hw.shape.replace(Bt=end - start)
    w.src_slots = hw.src_slots[:, start:end].copy()
    w.dst_slots = hw.dst_slots[:, start:end].copy()
    w.ring_start = hw.ring_start[start:end].copy()
    w.replay_prefix_len = hw.replay_prefix_len[start:end].copy()
    w.active = dist.shard_active(hw.active, start, end)
    return w


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import oracle
    try:
        assert dist.init("gloo")
        hw = wl.host_world(SHAPE, seed=3)
        start, end = dist.shard(SHAPE.Bt, rank, world)
        mine = slice_requests(hw, start, end)
        oracle.materialize(mine)
        # every rank works alone; only the results travel, for the check
        written = {l: {int(d): mine.state[l][int(d)].tobytes() for d in mine.dst_slots[l]
                       if d != SHAPE.pad_slot_id} for l in range(SHAPE.L)}
        gathered = [None] * world
        td.all_gather_object(gathered, written)
        worst = dist.max_over_ranks(float(rank + 1))
        dist.barrier()
        q.put((rank, gathered, worst, (start, end)))
    finally:
        if td.is_initialized():
            td.destroy_process_group()


def test_two_ranks_equal_one_process():
    import oracle
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    ranges = [r[3] for r in results]
    assert ranges == [(0, 3), (3, 7)]
    assert all(r[2] == 2.0 for r in results)

    full = wl.host_world(SHAPE, seed=3)
    ref = full.copy()
    oracle.materialize(ref)
    gathered = results[0][1]
    checked = 0
    for l in range(SHAPE.L):
        for rank_written in gathered:
            for slot, data in rank_written[l].items():
                n = int(np.argmax(full.active == -1)) if (full.active == -1).any() else SHAPE.Bt
                active = set(int(b) for b in full.active[:n])
                b = int(np.where(full.dst_slots[l] == slot)[0][0])
                if b in active and full.src_slots[l, b] != SHAPE.pad_slot_id:
                    assert data == ref.state[l][slot].tobytes(), (l, slot)
                    checked += 1
    assert checked == sum(1 for b in full.active if b >= 0) * SHAPE.L


def test_shard_covers_batch_exactly():
    for batch in (1, 7, 256):
        for world in (1, 2, 3, 8):
            if world > batch:
                continue
            spans = [dist.shard(batch, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == batch
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


def test_shard_active_keeps_order_and_terminator():
    active = np.array([5, 0, 3, -1, 2, 6], np.int32)   # 2 and 6 sit after the -1: ignored
    np.testing.assert_array_equal(dist.shard_active(active, 0, 3), [0, -1, -1])
    np.testing.assert_array_equal(dist.shard_active(active, 3, 6), [2, 0, -1])


# ----------------------------------------------------------------------------
# tensor-parallel head shards and pipeline-parallel layer shards
# ----------------------------------------------------------------------------

MP_SHAPES = {
    "bf16": wl.Shape("mp16", L=4, Bt=5, H=8, hpg=2, D=16, N=16, R=8, W=8, state_dtype="bf16", n_active=4,
                     ring_start=(0, 8), prefix=("uniform", 0, 8), pad_frac=0.1),
    "i8": wl.Shape("mp8", L=4, Bt=3, H=8, hpg=2, D=64, N=128, R=8, W=8, state_dtype="i8", n_active=3,
                   ring_start=(0, 8), prefix=("uniform", 1, 8)),
}


def slice_heads(hw, h0, h1):
    """The world as a tensor-parallel rank holds it: heads [h0, h1) of every
    layer (state, scales, x, dt and A) and their B groups."""
    g0, g1 = h0 // hw.hpg, h1 // hw.hpg
    w = hw.copy()
    w.shape = hw.shape.replace(H=h1 - h0)
    w.state = [np.ascontiguousarray(a[:, h0:h1]) for a in hw.state]
    w.scale = [None if a is None else np.ascontiguousarray(a[:, h0:h1]) for a in hw.scale]
    w.x = [np.ascontiguousarray(a[:, :, h0:h1]) for a in hw.x]
    w.B = [np.ascontiguousarray(a[:, :, g0:g1]) for a in hw.B]
    w.dt = [np.ascontiguousarray(a[:, :, h0:h1]) for a in hw.dt]
    w.A = [np.ascontiguousarray(a[h0:h1]) for a in hw.A]
    return w


def slice_layers(hw, l0, l1):
    """The world as a pipeline-parallel rank holds it: layers [l0, l1)."""
    w = hw.copy()
    w.shape = hw.shape.replace(L=l1 - l0)
    for name in ("state", "scale", "x", "B", "dt", "A"):
        setattr(w, name, getattr(w, name)[l0:l1])
    w.src_slots = hw.src_slots[l0:l1].copy()
    w.dst_slots = hw.dst_slots[l0:l1].copy()
    return w


def _mp_worker(rank, world, port, mode, fmt, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import oracle
    try:
        assert dist.init("gloo")
        shape = MP_SHAPES[fmt]
        hw = wl.host_world(shape, seed=21)
        if mode == "heads":
            lo, hi = dist.head_shard(shape.H, shape.hpg, rank, world)
            mine = slice_heads(hw, lo, hi)
        else:
            lo, hi = dist.layer_shard(shape.L, rank, world)
            mine = slice_layers(hw, lo, hi)
        oracle.materialize(mine)   # each rank alone, on its own shard
        part = {"range": (lo, hi), "state": mine.state, "scale": mine.scale}
        gathered = [None] * world
        td.all_gather_object(gathered, part)   # only for the check
        q.put((rank, gathered))
    finally:
        if td.is_initialized():
            td.destroy_process_group()


@pytest.mark.parametrize("fmt", ["bf16", "i8"])
@pytest.mark.parametrize("mode", ["heads", "layers"])
def test_head_and_layer_shards_equal_one_process(mode, fmt):
    """Two gloo ranks, each owning half of every layer's heads (whole B groups)
    or half of the layers, materialize their shards alone; put back together,
    every slot of every layer equals the single-process result byte for byte
    (round to nearest: no stochastic draws involved).  Unmeasured on GPUs: this
    pool runs one GPU per call."""
    import oracle
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_mp_worker, args=(r, world, port, mode, fmt, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    parts = sorted(results)[0][1]
    shape = MP_SHAPES[fmt]
    ref = wl.host_world(shape, seed=21)
    oracle.materialize(ref)
    for l in range(shape.L):
        if mode == "heads":
            state = np.concatenate([pt["state"][l] for pt in parts], axis=1)
            scale = None if ref.scale[l] is None else np.concatenate([pt["scale"][l] for pt in parts], axis=1)
        else:
            owner = next(pt for pt in parts if pt["range"][0] <= l < pt["range"][1])
            state = owner["state"][l - owner["range"][0]]
            scale = owner["scale"][l - owner["range"][0]]
        assert state.tobytes() == ref.state[l].tobytes(), (mode, l)
        if scale is not None:
            assert scale.tobytes() == ref.scale[l].tobytes(), (mode, l)


def test_head_shard_keeps_b_groups_whole():
    assert [dist.head_shard(256, 32, r, 8) for r in (0, 7)] == [(0, 32), (224, 256)]
    assert dist.head_shard(80, 80, 0, 1) == (0, 80)
    with pytest.raises(ValueError, match="cut a B group"):
        dist.head_shard(256, 32, 0, 16)      # 16 heads per rank, groups of 32
    with pytest.raises(ValueError, match="evenly"):
        dist.head_shard(80, 80, 0, 3)
    with pytest.raises(ValueError, match="cut a B group"):
        dist.head_shard(80, 80, 1, 2)        # one group: no head split at all


def test_layer_shard_kwargs_slices_per_layer_tables_only():
    import torch
    L, B = 6, 3
    kw = {key: torch.arange(L * B).view(L, B) if key in ("src_slots", "dst_slots") else torch.arange(L)
          for key in dist.PER_LAYER_KEYS}
    kw.update(ring_start=torch.arange(B), active_request_indices=torch.arange(B), num_heads=4)
    kw["state_scale_ptrs"] = None
    out = dist.layer_shard_kwargs(kw, 2, 5)
    assert out["state_ptrs"].tolist() == [2, 3, 4] and out["state_scale_ptrs"] is None
    assert out["src_slots"].shape == (3, B) and out["src_slots"][0].tolist() == [6, 7, 8]
    assert out["ring_start"] is kw["ring_start"] and out["num_heads"] == 4
