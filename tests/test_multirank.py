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
