"""Python handle on the plain C oracle for ReplaySSM prefix materialization.

TEST INFRASTRUCTURE ONLY.  The oracle is the slow, obviously-correct CPU
checker that the CUDA library is compared against.  Only the test suite, the
package's smoke entry and the benchmark's CPU-baseline leg may import it; the
product path never does.  It shares no code with the CUDA library and imports
nothing from it.

The operation follows the flashinfer.mamba.replayssm_materialize API page
(signature, Parameters, Notes); the readings of what the pages leave open are
listed at the top of replayssm_oracle.c.

Parity status: every function here is pinned by tests/test_oracle_pins.py
and tests/test_oracle_gdn_pins.py (closed form, copy, composition, ring wrap,
pad/-1 skipping, brute force over ring_start x prefix, format conversions
against numpy/torch, Philox against the published known-answer vectors, the
stochastic-rounding counter layout and the one-byte quotient through stored
bytes predicted from their written statements, the GDN epsilon placement).
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, F16, I8, FP8_E4M3 = 0, 1, 2, 3, 4
DTYPE_CODES = {"f32": F32, "bf16": BF16, "f16": F16, "i8": I8, "fp8_e4m3": FP8_E4M3}

_P64 = ctypes.POINTER(ctypes.c_int64)
_P32 = ctypes.POINTER(ctypes.c_int32)


class OracleArgs(ctypes.Structure):
    _fields_ = [
        ("state_ptrs", _P64), ("state_slot_strides", _P64),
        ("x_cache_ptrs", _P64), ("x_cache_slot_strides", _P64),
        ("B_cache_ptrs", _P64), ("B_cache_slot_strides", _P64),
        ("dt_cache_ptrs", _P64), ("dt_cache_slot_strides", _P64),
        ("A_ptrs", _P64),
        ("state_scale_ptrs", _P64), ("state_scale_slot_strides", _P64),
        ("src_slots", _P32), ("dst_slots", _P32),
        ("ring_start", _P32), ("replay_prefix_len", _P32),
        ("active_request_indices", _P32),
        ("rand_seed", _P64),
        ("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32), ("input_dtype", ctypes.c_int32),
        ("matrixA_dtype", ctypes.c_int32),
        ("dim", ctypes.c_int32), ("dstate", ctypes.c_int32),
        ("num_heads", ctypes.c_int64),
        ("heads_per_group", ctypes.c_int32), ("max_window", ctypes.c_int32),
        ("ring_buffer_len", ctypes.c_int32), ("pad_slot_id", ctypes.c_int32),
        ("philox_rounds", ctypes.c_int32),
        ("sr_counter_slots", _P32), ("sr_counter_layers", _P32),
        ("num_slots", ctypes.c_int32),
    ]


class GdnArgs(ctypes.Structure):
    """Mirror of oracle_gdn_args (gdn_commit_oracle.h)."""
    _fields_ = [
        ("state", ctypes.c_void_p), ("rawv", ctypes.c_void_p), ("rawk", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("state_indices", _P32), ("accept_lens", _P32),
        ("track_state_indices", _P32), ("track_steps", _P32),
        ("layers", ctypes.c_int32), ("slots", ctypes.c_int32), ("hv", ctypes.c_int32), ("h", ctypes.c_int32),
        ("t", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("use_qk_l2norm", ctypes.c_int32), ("null_block_id", ctypes.c_int32),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_materialize.argtypes = [ctypes.POINTER(OracleArgs)]
        L.oracle_materialize.restype = ctypes.c_int
        L.oracle_last_error.restype = ctypes.c_char_p
        L.oracle_philox4x32.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                                        ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)]
        L.oracle_round.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_uint32]
        L.oracle_round.restype = ctypes.c_double
        L.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
        L.oracle_decode.restype = ctypes.c_double
        L.oracle_encode.argtypes = [ctypes.c_int, ctypes.c_double]
        L.oracle_encode.restype = ctypes.c_uint32
        L.oracle_args_size.restype = ctypes.c_int
        L.oracle_gdn_commit.argtypes = [ctypes.POINTER(GdnArgs)]
        L.oracle_gdn_commit.restype = ctypes.c_int
        L.oracle_gdn_last_error.restype = ctypes.c_char_p
        if L.oracle_args_size() != ctypes.sizeof(OracleArgs):
            raise RuntimeError("oracle argument struct layout mismatch")
        _lib = L
    return _lib


def _addr_table(arrays):
    return np.array([0 if a is None else a.ctypes.data for a in arrays], dtype=np.int64)


def _slot_stride(a):
    """Outer-slot stride in elements of a C-contiguous per-layer array [slots, ...]."""
    return int(np.prod(a.shape[1:])) if a is not None else 0


def materialize(world) -> None:
    """Runs the oracle on a host world in place: writes the destination slots
    of world.state / world.scale.  `world` is a workloads.HostWorld (any object
    with the same attributes works)."""
    L = lib()
    for arrs in (world.state, world.x, world.B, world.dt, world.A):
        for a in arrs:
            assert a.flags["C_CONTIGUOUS"]
    keep = []

    def tab(arr):
        keep.append(arr)
        return arr.ctypes.data_as(_P64)

    def tab32(arr):
        arr = np.ascontiguousarray(arr, dtype=np.int32)
        keep.append(arr)
        return arr.ctypes.data_as(_P32)

    quant = world.state_dtype in ("i8", "fp8_e4m3")
    args = OracleArgs()
    args.state_ptrs = tab(_addr_table(world.state))
    args.state_slot_strides = tab(np.array([_slot_stride(a) for a in world.state], np.int64))
    args.x_cache_ptrs = tab(_addr_table(world.x))
    args.x_cache_slot_strides = tab(np.array([_slot_stride(a) for a in world.x], np.int64))
    args.B_cache_ptrs = tab(_addr_table(world.B))
    args.B_cache_slot_strides = tab(np.array([_slot_stride(a) for a in world.B], np.int64))
    args.dt_cache_ptrs = tab(_addr_table(world.dt))
    args.dt_cache_slot_strides = tab(np.array([_slot_stride(a) for a in world.dt], np.int64))
    args.A_ptrs = tab(_addr_table(world.A))
    if quant:
        args.state_scale_ptrs = tab(_addr_table(world.scale))
        args.state_scale_slot_strides = tab(np.array([_slot_stride(a) for a in world.scale], np.int64))
    else:
        zeros = np.zeros(world.L, np.int64)
        args.state_scale_ptrs = tab(zeros)
        args.state_scale_slot_strides = tab(zeros.copy())
    args.src_slots = tab32(world.src_slots)
    args.dst_slots = tab32(world.dst_slots)
    args.ring_start = tab32(world.ring_start)
    args.replay_prefix_len = tab32(world.replay_prefix_len)
    args.active_request_indices = tab32(world.active)
    if world.philox_rounds > 0:
        args.rand_seed = tab(np.array([world.rand_seed], np.int64))
    args.num_layers = world.L
    args.batch = world.Bt
    args.state_dtype = DTYPE_CODES[world.state_dtype]
    args.input_dtype = DTYPE_CODES[world.input_dtype]
    args.matrixA_dtype = DTYPE_CODES[world.A_dtype]
    args.dim = world.D
    args.dstate = world.N
    args.num_heads = world.H
    args.heads_per_group = world.hpg
    args.max_window = world.W
    args.ring_buffer_len = world.R
    args.pad_slot_id = world.pad_slot_id
    args.philox_rounds = world.philox_rounds
    args.num_slots = min(int(a.shape[0]) for a in world.state)
    # a one-request copy of a larger call (workloads.host_subworld) names the
    # destination slot and layer of that call: the Philox counter uses them
    meta = getattr(world, "meta", None) or {}
    if "dst_slot_in_call" in meta:
        args.sr_counter_slots = tab32(np.full((world.L, world.Bt), meta["dst_slot_in_call"], np.int32))
        args.sr_counter_layers = tab32(np.full(world.L, meta["layer_in_call"], np.int32))
    rc = L.oracle_materialize(ctypes.byref(args))
    if rc != 0:
        raise ValueError("oracle: " + L.oracle_last_error().decode())


def philox4x32(ctr, key, rounds=10):
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib().oracle_philox4x32(c, k, int(rounds), o)
    return tuple(o)


def round_to(fmt, y, stochastic=False, r16=0):
    return lib().oracle_round(DTYPE_CODES.get(fmt, fmt), float(y), int(stochastic), int(r16) & 0xFFFF)


def decode(fmt, bits):
    return lib().oracle_decode(DTYPE_CODES.get(fmt, fmt), int(bits) & 0xFFFFFFFF)


def encode(fmt, value):
    return lib().oracle_encode(DTYPE_CODES.get(fmt, fmt), float(value))


def gdn_commit(world) -> None:
    """Runs the gated-delta-rule commit oracle on a host world in place
    (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit, API page):
    world.state is updated; track slots are written.  `world` is a
    workloads.GdnWorld (any object with the same attributes works)."""
    L = lib()
    keep = []

    def arr(a, dtype):
        assert a.dtype == dtype and a.flags["C_CONTIGUOUS"], (a.dtype, dtype)
        keep.append(a)
        return a.ctypes.data

    def i32(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=np.int32)
        keep.append(a)
        return a.ctypes.data_as(_P32)

    L_, SL, HV, T = world.state.shape[0], world.state.shape[1], world.state.shape[2], world.rawv.shape[3]
    args = GdnArgs()
    args.state = arr(world.state, np.float32)
    args.rawv = arr(world.rawv, np.uint16)
    args.rawk = arr(world.rawk, np.uint16)
    args.g = arr(world.g, np.float32)
    args.beta = arr(world.beta, np.float32)
    args.state_indices = i32(world.state_indices)
    args.accept_lens = i32(world.accept_lens)
    args.track_state_indices = i32(world.track_state_indices)
    args.track_steps = i32(world.track_steps)
    args.layers, args.slots, args.hv, args.h, args.t = L_, SL, HV, world.rawk.shape[2], T
    args.batch = len(world.state_indices)
    args.use_qk_l2norm = int(bool(world.use_qk_l2norm))
    args.null_block_id = int(world.null_block_id)
    if L.oracle_gdn_commit(ctypes.byref(args)) != 0:
        raise ValueError("oracle: " + L.oracle_gdn_last_error().decode())
