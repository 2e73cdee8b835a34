"""Multi-GPU plumbing for the data-parallel case.

Every (request, layer, head) item is independent and no step of the
materialization exchanges data, so N GPUs run N independent shards and each
launches its own kernel on its own part of the slot pools:
  - request shards (data parallel): a contiguous block of the global batch;
  - head shards (tensor parallel): a contiguous block of every layer's heads,
    made of whole B groups (a rank holds only its own groups' B cache);
  - layer shards (pipeline parallel): a contiguous block of the layers.
The only cross-rank traffic is measurement (barriers and a max over ranks of
the elapsed time), never the data path.  Stochastic rounding draws its Philox
words from each call's own (layer, head) numbering, so a sharded run rounds
differently from an unsharded one (each is a valid draw); round-to-nearest
results are identical.
"""
from __future__ import annotations

import os


def env() -> tuple[int, int, int]:
    """(rank, local_rank, world_size) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def init(backend: str) -> bool:
    """Initialises the default process group when running under torchrun."""
    import torch.distributed as td
    _, _, world = env()
    if world > 1 and not td.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        td.init_process_group(backend=backend, init_method="env://")
    return td.is_available() and td.is_initialized()


def barrier() -> None:
    import torch.distributed as td
    if td.is_available() and td.is_initialized():
        td.barrier()


def max_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def shard(batch: int, rank: int, world: int) -> tuple[int, int]:
    """[start, end) of the requests rank `rank` owns out of a global batch."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    return batch * rank // world, batch * (rank + 1) // world


def shard_active(active, start: int, end: int):
    """The global active list restricted to requests in [start, end), re-indexed
    to the shard's local batch and -1 padded to its length."""
    import numpy as np
    active = np.asarray(active)
    n = int(np.argmax(active == -1)) if (active == -1).any() else len(active)
    mine = [int(b) - start for b in active[:n] if start <= b < end]
    out = np.full(end - start, -1, np.int32)
    out[:len(mine)] = mine
    return out


def head_shard(num_heads: int, heads_per_group: int, rank: int, world: int) -> tuple[int, int]:
    """[h0, h1) of the heads a tensor-parallel rank owns: an even split of
    every layer's heads in which every B group (heads_per_group consecutive
    heads reading one B cache row) stays on one rank.  Raises ValueError when
    the split would cut a group."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    if num_heads % world:
        raise ValueError(f"{num_heads} heads do not split evenly over {world} ranks")
    per = num_heads // world
    if per % heads_per_group:
        raise ValueError(f"{per} heads per rank would cut a B group of {heads_per_group} heads")
    return rank * per, (rank + 1) * per


def layer_shard(num_layers: int, rank: int, world: int) -> tuple[int, int]:
    """[l0, l1) of the layers a pipeline-parallel rank owns (contiguous)."""
    return shard(num_layers, rank, world)


# replayssm_materialize arguments with one entry (or row) per layer
PER_LAYER_KEYS = ("state_ptrs", "state_slot_strides", "x_cache_ptrs", "x_cache_slot_strides", "B_cache_ptrs",
                  "B_cache_slot_strides", "dt_cache_ptrs", "dt_cache_slot_strides", "A_ptrs", "state_scale_ptrs",
                  "state_scale_slot_strides", "src_slots", "dst_slots")


def layer_shard_kwargs(kwargs: dict, l0: int, l1: int) -> dict:
    """replayssm_materialize keyword arguments restricted to layers [l0, l1):
    the per-layer pointer and stride tables and the rows of the slot tables
    (views, no copies).  Everything per request stays as it is."""
    out = dict(kwargs)
    for key in PER_LAYER_KEYS:
        if out.get(key) is not None:
            out[key] = out[key][l0:l1]
    return out
