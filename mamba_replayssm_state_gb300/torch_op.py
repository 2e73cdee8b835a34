"""torch.library custom op for torch.compile graphs.

`torch.ops.replayssm.materialize` wraps `replayssm_materialize` (API page:
flashinfer.mamba.replayssm_materialize, Parameters `dependency_inputs` and
`dependency_outputs`).  The kernel reads and writes through pointer tables,
which a tracing compiler cannot follow, so the caller names the backing
storage: `dependency_inputs` (read) and `dependency_outputs` (written, declared
mutated).  The op returns nothing; its fake implementation does nothing, so a
compiled graph only orders the op after the producers of the inputs and before
the readers of the outputs.

Dtypes travel as the integer codes of include/replayssm.h (RSM_F32 = 0,
RSM_BF16, RSM_F16, RSM_I8, RSM_FP8_E4M3).
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import _dtype_code, replayssm_materialize

__all__ = ["materialize", "OP"]


@torch.library.custom_op("replayssm::materialize", mutates_args=("dependency_outputs",))
def _materialize(state_ptrs: torch.Tensor, state_slot_strides: torch.Tensor, x_cache_ptrs: torch.Tensor,
                 x_cache_slot_strides: torch.Tensor, B_cache_ptrs: torch.Tensor, B_cache_slot_strides: torch.Tensor,
                 dt_cache_ptrs: torch.Tensor, dt_cache_slot_strides: torch.Tensor, A_ptrs: torch.Tensor,
                 state_scale_ptrs: Optional[torch.Tensor], state_scale_slot_strides: Optional[torch.Tensor],
                 src_slots: torch.Tensor, dst_slots: torch.Tensor, ring_start: torch.Tensor,
                 replay_prefix_len: torch.Tensor, active_request_indices: torch.Tensor,
                 rand_seed: Optional[torch.Tensor], dependency_inputs: List[torch.Tensor],
                 dependency_outputs: List[torch.Tensor], state_dtype: int, input_dtype: int, matrixA_dtype: int,
                 dim: int, dstate: int, num_heads: int, heads_per_group: int, max_window: int,
                 ring_buffer_len: int, pad_slot_id: int, philox_rounds: int, num_slots: int = 0) -> None:
    replayssm_materialize(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs,
                          B_cache_slot_strides, dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs,
                          state_scale_slot_strides, src_slots, dst_slots, ring_start, replay_prefix_len,
                          active_request_indices, state_dtype=state_dtype, input_dtype=input_dtype,
                          matrixA_dtype=matrixA_dtype, dim=dim, dstate=dstate, num_heads=num_heads,
                          heads_per_group=heads_per_group, max_window=max_window,
                          ring_buffer_len=ring_buffer_len, pad_slot_id=pad_slot_id, rand_seed=rand_seed,
                          philox_rounds=philox_rounds, num_slots=num_slots)


@_materialize.register_fake
def _materialize_fake(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs,
                      B_cache_slot_strides, dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs,
                      state_scale_slot_strides, src_slots, dst_slots, ring_start, replay_prefix_len,
                      active_request_indices, rand_seed, dependency_inputs, dependency_outputs, state_dtype,
                      input_dtype, matrixA_dtype, dim, dstate, num_heads, heads_per_group, max_window,
                      ring_buffer_len, pad_slot_id, philox_rounds, num_slots=0) -> None:
    return None


OP = torch.ops.replayssm.materialize


def materialize(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs,
                B_cache_slot_strides, dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs,
                state_scale_slot_strides, src_slots, dst_slots, ring_start, replay_prefix_len,
                active_request_indices, *, state_dtype, input_dtype, matrixA_dtype, dim, dstate, num_heads,
                heads_per_group, max_window, ring_buffer_len, pad_slot_id=-1, rand_seed=None, philox_rounds=0,
                dependency_inputs=None, dependency_outputs=None, num_slots=0) -> None:
    """replayssm_materialize's arguments (dtypes as torch dtypes, names or
    codes), through the custom op so that torch.compile can trace it."""
    OP(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs, B_cache_slot_strides,
       dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs, state_scale_slot_strides, src_slots,
       dst_slots, ring_start, replay_prefix_len, active_request_indices, rand_seed, list(dependency_inputs or []),
       list(dependency_outputs or []), _dtype_code(state_dtype), _dtype_code(input_dtype),
       _dtype_code(matrixA_dtype), int(dim), int(dstate), int(num_heads), int(heads_per_group), int(max_window),
       int(ring_buffer_len), int(pad_slot_id), int(philox_rounds), int(num_slots or 0))
