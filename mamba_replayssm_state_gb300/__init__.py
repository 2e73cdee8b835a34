"""GB300-native ReplaySSM prefix materialization.

`replayssm_materialize(...)` takes the arguments of
flashinfer.mamba.replayssm_materialize (API page: signature and Parameters)
as CUDA tensors, marshals them into the C ABI of libreplayssm.so
(include/replayssm.h) and enqueues the sm_103a kernel on the current CUDA
stream.  Every step of the computation runs in that kernel; this module only
passes pointers.  There is no fallback: if the library is missing or cannot
load, calls raise.

The torch.compile dependency anchors of the API page (dependency_inputs /
dependency_outputs) are accepted and ignored: they carry no data.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["replayssm_materialize", "gated_delta_rule_replayssm_commit", "prepare", "launch_config", "kernel_name",
           "pointer_table", "stride_table", "library_path", "load_library", "ReplaySSMError", "STATUS_BITS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libreplayssm.so")

RSM_F32, RSM_BF16, RSM_F16, RSM_I8, RSM_FP8_E4M3 = 0, 1, 2, 3, 4
STATUS_BITS = {"bad_active_index": 1, "bad_ring_start": 2, "bad_prefix_len": 4, "bad_slot": 8,
               "wait_timeout": 16}


class ReplaySSMError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"rsm_materialize failed ({code}): {message}")
        self.code = code


_P = ctypes.c_void_p


class RsmArgs(ctypes.Structure):
    """Mirror of rsm_materialize_args (include/replayssm.h)."""
    _fields_ = [
        ("state_ptrs", _P), ("state_slot_strides", _P),
        ("x_cache_ptrs", _P), ("x_cache_slot_strides", _P),
        ("B_cache_ptrs", _P), ("B_cache_slot_strides", _P),
        ("dt_cache_ptrs", _P), ("dt_cache_slot_strides", _P),
        ("A_ptrs", _P),
        ("state_scale_ptrs", _P), ("state_scale_slot_strides", _P),
        ("src_slots", _P), ("dst_slots", _P),
        ("ring_start", _P), ("replay_prefix_len", _P),
        ("active_request_indices", _P),
        ("rand_seed", _P),
        ("device_status", _P),
        ("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32), ("input_dtype", ctypes.c_int32),
        ("matrixA_dtype", ctypes.c_int32),
        ("dim", ctypes.c_int32), ("dstate", ctypes.c_int32),
        ("num_heads", ctypes.c_int64),
        ("heads_per_group", ctypes.c_int32), ("max_window", ctypes.c_int32),
        ("ring_buffer_len", ctypes.c_int32), ("pad_slot_id", ctypes.c_int32),
        ("philox_rounds", ctypes.c_int32),
        ("num_slots", ctypes.c_int32),
    ]


EXPORTS = ("rsm_materialize", "rsm_last_error", "rsm_args_size", "rsm_abi_version", "rsm_launch_config",
           "rsm_kernel_name", "rsm_gdn_commit", "rsm_gdn_args_size")

_lib = None


def library_path() -> str:
    return _LIB_PATH


class GdnArgs(ctypes.Structure):
    """Mirror of rsm_gdn_commit_args (include/replayssm.h)."""
    _fields_ = [
        ("checkpoint_state", _P), ("rawv_cache", _P), ("rawk_cache", _P), ("g_cache", _P), ("beta_cache", _P),
        ("state_indices", _P), ("accept_lens", _P), ("track_state_indices", _P), ("track_steps", _P),
        ("device_status", _P),
        ("layers", ctypes.c_int32), ("slots", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
        ("num_k_heads", ctypes.c_int32), ("window", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("use_qk_l2norm", ctypes.c_int32), ("null_block_id", ctypes.c_int32), ("backend", ctypes.c_int32),
    ]


GDN_BACKENDS = {"auto": 0, "simt": 1, "tcgen05": 2}  # RSM_GDN_BACKEND_* (include/replayssm.h)


def load_library(build_if_missing: bool = True):
    """Loads libreplayssm.so (building it in-tree first when it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        if not build_if_missing:
            raise OSError(f"libreplayssm.so is not built ({_LIB_PATH})")
        from . import _build
        _build.build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.rsm_materialize.argtypes = [ctypes.POINTER(RsmArgs), ctypes.c_void_p]
    lib.rsm_materialize.restype = ctypes.c_int
    lib.rsm_last_error.restype = ctypes.c_char_p
    lib.rsm_args_size.restype = ctypes.c_int
    lib.rsm_abi_version.restype = ctypes.c_int
    lib.rsm_launch_config.argtypes = [ctypes.POINTER(RsmArgs)] + [ctypes.POINTER(ctypes.c_int)] * 4
    lib.rsm_launch_config.restype = ctypes.c_int
    lib.rsm_kernel_name.argtypes = [ctypes.POINTER(RsmArgs)]
    lib.rsm_kernel_name.restype = ctypes.c_char_p
    if lib.rsm_args_size() != ctypes.sizeof(RsmArgs):
        raise OSError("rsm_materialize_args layout mismatch between libreplayssm.so and the binding")
    lib.rsm_gdn_commit.argtypes = [ctypes.POINTER(GdnArgs), ctypes.c_void_p]
    lib.rsm_gdn_commit.restype = ctypes.c_int
    lib.rsm_gdn_args_size.restype = ctypes.c_int
    if lib.rsm_gdn_args_size() != ctypes.sizeof(GdnArgs):
        raise OSError("rsm_gdn_commit_args layout mismatch between libreplayssm.so and the binding")
    _lib = lib
    return lib


def _dtype_code(dt) -> int:
    if isinstance(dt, int):
        return dt
    if isinstance(dt, str):
        return {"f32": RSM_F32, "float32": RSM_F32, "bf16": RSM_BF16, "bfloat16": RSM_BF16, "f16": RSM_F16,
                "float16": RSM_F16, "i8": RSM_I8, "int8": RSM_I8, "fp8_e4m3": RSM_FP8_E4M3,
                "float8_e4m3fn": RSM_FP8_E4M3}[dt]
    import torch
    table = {torch.float32: RSM_F32, torch.bfloat16: RSM_BF16, torch.float16: RSM_F16, torch.int8: RSM_I8}
    if hasattr(torch, "float8_e4m3fn"):
        table[torch.float8_e4m3fn] = RSM_FP8_E4M3
    if dt not in table:
        raise ValueError(f"unsupported dtype {dt}")
    return table[dt]


def _ptr(t, name, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _build_args(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs,
                B_cache_slot_strides, dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs,
                state_scale_slot_strides, src_slots, dst_slots, ring_start, replay_prefix_len,
                active_request_indices, *, state_dtype, input_dtype, matrixA_dtype, dim, dstate, num_heads,
                heads_per_group, max_window, ring_buffer_len, pad_slot_id=-1, rand_seed=None, philox_rounds=0,
                device_status=None, num_slots=0):
    import torch
    i64, i32 = torch.int64, torch.int32
    a = RsmArgs()
    a.state_ptrs = _ptr(state_ptrs, "state_ptrs", i64)
    a.state_slot_strides = _ptr(state_slot_strides, "state_slot_strides", i64)
    a.x_cache_ptrs = _ptr(x_cache_ptrs, "x_cache_ptrs", i64)
    a.x_cache_slot_strides = _ptr(x_cache_slot_strides, "x_cache_slot_strides", i64)
    a.B_cache_ptrs = _ptr(B_cache_ptrs, "B_cache_ptrs", i64)
    a.B_cache_slot_strides = _ptr(B_cache_slot_strides, "B_cache_slot_strides", i64)
    a.dt_cache_ptrs = _ptr(dt_cache_ptrs, "dt_cache_ptrs", i64)
    a.dt_cache_slot_strides = _ptr(dt_cache_slot_strides, "dt_cache_slot_strides", i64)
    a.A_ptrs = _ptr(A_ptrs, "A_ptrs", i64)
    a.state_scale_ptrs = _ptr(state_scale_ptrs, "state_scale_ptrs", i64, optional=True)
    a.state_scale_slot_strides = _ptr(state_scale_slot_strides, "state_scale_slot_strides", i64, optional=True)
    a.src_slots = _ptr(src_slots, "src_slots", i32)
    a.dst_slots = _ptr(dst_slots, "dst_slots", i32)
    a.ring_start = _ptr(ring_start, "ring_start", i32)
    a.replay_prefix_len = _ptr(replay_prefix_len, "replay_prefix_len", i32)
    a.active_request_indices = _ptr(active_request_indices, "active_request_indices", i32)
    a.rand_seed = _ptr(rand_seed, "rand_seed", i64, optional=True)
    a.device_status = _ptr(device_status, "device_status", optional=True)
    if src_slots.dim() != 2 or dst_slots.shape != src_slots.shape:
        raise ValueError("src_slots and dst_slots must both be [L, B]")
    L, B = src_slots.shape
    for name, t in (("state_ptrs", state_ptrs), ("x_cache_ptrs", x_cache_ptrs), ("A_ptrs", A_ptrs)):
        if t.numel() != L:
            raise ValueError(f"{name} must have L={L} entries")
    for name, t in (("ring_start", ring_start), ("replay_prefix_len", replay_prefix_len),
                    ("active_request_indices", active_request_indices)):
        if t.numel() != B:
            raise ValueError(f"{name} must have B={B} entries")
    a.num_layers, a.batch = int(L), int(B)
    a.state_dtype = _dtype_code(state_dtype)
    a.input_dtype = _dtype_code(input_dtype)
    a.matrixA_dtype = _dtype_code(matrixA_dtype)
    a.dim, a.dstate = int(dim), int(dstate)
    a.num_heads = int(num_heads)
    a.heads_per_group = int(heads_per_group)
    a.max_window = int(max_window)
    a.ring_buffer_len = int(ring_buffer_len)
    a.pad_slot_id = int(pad_slot_id)
    a.philox_rounds = int(philox_rounds)
    a.num_slots = int(num_slots or 0)
    return a


def replayssm_materialize(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs,
                          B_cache_slot_strides, dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs,
                          state_scale_slot_strides, src_slots, dst_slots, ring_start, replay_prefix_len,
                          active_request_indices, *, state_dtype, input_dtype, matrixA_dtype, dim, dstate,
                          num_heads, heads_per_group, max_window, ring_buffer_len, pad_slot_id=-1, rand_seed=None,
                          philox_rounds=0, dependency_inputs=None, dependency_outputs=None, device_status=None,
                          num_slots=0, stream=None) -> None:
    """Materialize SSM states at selected tokens from older states plus their replay rings.

    Same arguments as flashinfer.mamba.replayssm_materialize; all tensors live
    on the current CUDA device.  `device_status` (optional uint32/int32 [1]
    CUDA tensor) receives RSM_STATUS_* bits for skipped out-of-range metadata.
    `num_slots` (optional) states the slot count of every layer's pools, so that
    a slot at or past it is skipped and flagged instead of addressed; 0 leaves
    it unchecked.  `stream` defaults to torch's current stream.  Asynchronous:
    returns once the kernel is enqueued.
    """
    import torch
    lib = load_library()
    a = _build_args(state_ptrs, state_slot_strides, x_cache_ptrs, x_cache_slot_strides, B_cache_ptrs,
                    B_cache_slot_strides, dt_cache_ptrs, dt_cache_slot_strides, A_ptrs, state_scale_ptrs,
                    state_scale_slot_strides, src_slots, dst_slots, ring_start, replay_prefix_len,
                    active_request_indices, state_dtype=state_dtype, input_dtype=input_dtype,
                    matrixA_dtype=matrixA_dtype, dim=dim, dstate=dstate, num_heads=num_heads,
                    heads_per_group=heads_per_group, max_window=max_window, ring_buffer_len=ring_buffer_len,
                    pad_slot_id=pad_slot_id, rand_seed=rand_seed, philox_rounds=philox_rounds,
                    device_status=device_status, num_slots=num_slots)
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.rsm_materialize(ctypes.byref(a), ctypes.c_void_p(handle))
    if rc != 0:
        raise ReplaySSMError(rc, lib.rsm_last_error().decode())


class Prepared:
    """A materialization whose arguments were marshalled once: calling it only
    enqueues the kernel (for serving loops and CUDA-graph capture).  The
    tensors it points at must stay alive and in place."""

    def __init__(self, lib, args, keep):
        self._lib, self._args, self._keep = lib, args, keep

    def __call__(self, stream=None) -> None:
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        rc = self._lib.rsm_materialize(ctypes.byref(self._args), ctypes.c_void_p(handle))
        if rc != 0:
            raise ReplaySSMError(rc, self._lib.rsm_last_error().decode())


def prepare(*args, **kwargs) -> Prepared:
    """Marshals replayssm_materialize's arguments once; returns a callable."""
    lib = load_library()
    kwargs.pop("stream", None)
    kwargs.pop("dependency_inputs", None)
    kwargs.pop("dependency_outputs", None)
    a = _build_args(*args, **kwargs)
    return Prepared(lib, a, (args, kwargs))


def launch_config(*args, **kwargs) -> dict:
    """The (grid, block, smem_bytes, stages) rsm_materialize would use for these arguments."""
    lib = load_library()
    kwargs.pop("stream", None)
    kwargs.pop("dependency_inputs", None)
    kwargs.pop("dependency_outputs", None)
    a = _build_args(*args, **kwargs)
    out = [ctypes.c_int() for _ in range(4)]
    rc = lib.rsm_launch_config(ctypes.byref(a), *[ctypes.byref(o) for o in out])
    if rc != 0:
        raise ReplaySSMError(rc, lib.rsm_last_error().decode())
    return dict(zip(("grid", "block", "smem_bytes", "stages"), (o.value for o in out)))


def kernel_name(*args, **kwargs) -> str:
    """Name of the kernel replayssm_materialize launches for these arguments
    ("materialize_kernel", "materialize_q8_kernel", "materialize_q8tc_kernel"
    or "materialize_tc_kernel")."""
    lib = load_library()
    kwargs.pop("stream", None)
    kwargs.pop("dependency_inputs", None)
    kwargs.pop("dependency_outputs", None)
    a = _build_args(*args, **kwargs)
    name = lib.rsm_kernel_name(ctypes.byref(a)).decode()
    if not name:
        raise ReplaySSMError(-1, lib.rsm_last_error().decode())
    return name


def pointer_table(tensors, device=None):
    """int64 CUDA tensor of base addresses (0 for None), one per layer."""
    import torch
    dev = device or next(t.device for t in tensors if t is not None)
    return torch.tensor([0 if t is None else t.data_ptr() for t in tensors], dtype=torch.int64, device=dev)


def stride_table(tensors, device=None):
    """int64 CUDA tensor of outer-slot strides in elements (dim 0 of each tensor)."""
    import torch
    dev = device or next(t.device for t in tensors if t is not None)
    return torch.tensor([0 if t is None else t.stride(0) for t in tensors], dtype=torch.int64, device=dev)


def _gdn_args(checkpoint_state, rawv_cache, rawk_cache, g_cache, beta_cache, state_indices, accept_lens, *,
              track_state_indices=None, track_steps=None, use_qk_l2norm=True, null_block_id=-1, backend="auto",
              device_status=None):
    import torch
    if checkpoint_state.dim() != 5 or tuple(checkpoint_state.shape[3:]) != (128, 128):
        raise ValueError("checkpoint_state must be [layers, slots, HV, 128, 128]")
    L, SL, HV = checkpoint_state.shape[:3]
    if rawv_cache.dim() != 5 or tuple(rawv_cache.shape[:3]) != (L, SL, HV) or rawv_cache.shape[4] != 128:
        raise ValueError("rawv_cache must be [layers, slots, HV, T, 128]")
    T = rawv_cache.shape[3]
    if rawk_cache.dim() != 5 or tuple(rawk_cache.shape[:2]) != (L, SL) or tuple(rawk_cache.shape[3:]) != (T, 128):
        raise ValueError("rawk_cache must be [layers, slots, H, T, 128]")
    for name, t in (("g_cache", g_cache), ("beta_cache", beta_cache)):
        if tuple(t.shape) != (L, SL, HV, T):
            raise ValueError(f"{name} must be [layers, slots, HV, T]")
    if (track_state_indices is None) != (track_steps is None):
        raise ValueError("track_state_indices and track_steps come together")
    B = state_indices.numel()
    for name, t in (("accept_lens", accept_lens), ("track_state_indices", track_state_indices),
                    ("track_steps", track_steps)):
        if t is not None and t.numel() != B:
            raise ValueError(f"{name} must have B={B} entries")
    a = GdnArgs()
    a.checkpoint_state = _ptr(checkpoint_state, "checkpoint_state", torch.float32)
    a.rawv_cache = _ptr(rawv_cache, "rawv_cache", torch.bfloat16)
    a.rawk_cache = _ptr(rawk_cache, "rawk_cache", torch.bfloat16)
    a.g_cache = _ptr(g_cache, "g_cache", torch.float32)
    a.beta_cache = _ptr(beta_cache, "beta_cache", torch.float32)
    a.state_indices = _ptr(state_indices, "state_indices", torch.int32)
    a.accept_lens = _ptr(accept_lens, "accept_lens", torch.int32)
    a.track_state_indices = _ptr(track_state_indices, "track_state_indices", torch.int32, optional=True)
    a.track_steps = _ptr(track_steps, "track_steps", torch.int32, optional=True)
    a.device_status = _ptr(device_status, "device_status", optional=True)
    a.layers, a.slots, a.num_v_heads, a.num_k_heads = int(L), int(SL), int(HV), int(rawk_cache.shape[2])
    a.window, a.batch = int(T), int(B)
    a.use_qk_l2norm = int(bool(use_qk_l2norm))
    a.null_block_id = int(null_block_id)
    if backend not in GDN_BACKENDS:
        raise ValueError(f"backend must be one of {sorted(GDN_BACKENDS)} (got {backend!r})")
    a.backend = GDN_BACKENDS[backend]
    return a


def gated_delta_rule_replayssm_commit(checkpoint_state, rawv_cache, rawk_cache, g_cache, beta_cache, state_indices,
                                      accept_lens, *, track_state_indices=None, track_steps=None,
                                      use_qk_l2norm=True, null_block_id=-1, backend="auto", device_status=None,
                                      stream=None) -> None:
    """Commit accepted ReplaySSM prefixes into every layer's gated-delta-rule
    checkpoints, in place.

    Same arguments as flashinfer.gdn_decode.gated_delta_rule_replayssm_commit
    (API page).  `backend` "auto" and "simt" run the kernel with fp32
    contractions on the CUDA cores; "tcgen05" runs the contractions on the
    tensor cores with TF32 operands, and (as on the page) requires
    use_qk_l2norm, no tracking and a window of 4 to 8 tokens.
    `device_status` (optional int32 [1] CUDA tensor) receives RSM_STATUS_* bits
    for skipped out-of-range metadata.  Asynchronous on `stream` (default:
    torch's current stream).
    """
    import torch
    lib = load_library()
    a = _gdn_args(checkpoint_state, rawv_cache, rawk_cache, g_cache, beta_cache, state_indices, accept_lens,
                  track_state_indices=track_state_indices, track_steps=track_steps, use_qk_l2norm=use_qk_l2norm,
                  null_block_id=null_block_id, device_status=device_status, backend=backend)
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.rsm_gdn_commit(ctypes.byref(a), ctypes.c_void_p(handle))
    if rc != 0:
        raise ReplaySSMError(rc, lib.rsm_last_error().decode())
