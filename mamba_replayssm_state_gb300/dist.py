"""Multi-GPU plumbing for the data-parallel case.

Every (request, layer, head) item is independent and no step of the
materialization exchanges data, so N GPUs run N independent shards: each rank
owns a contiguous block of the global batch (its own state pool and rings)
and launches its own kernel.  The only cross-rank traffic is measurement
(barriers and a max over ranks of the elapsed time), never the data path.
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
