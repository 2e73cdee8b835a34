"""Seeded synthetic workloads for ReplaySSM prefix materialization.

This module only draws random inputs and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it.  There is no dataset: the shapes are model shapes (no weights needed) and
every value is drawn from a seeded generator.

Layouts (per layer; "slots" is the outer slot dimension the pointer tables'
slot strides step over):
  state  [slots, H, D, N]   f32 / bf16 bits (uint16) / f16 / int8 / fp8 bits (uint8)
  scale  [slots, H, D]      fp32, one-byte state only
  x      [slots, R, H, D]   bf16 bits (uint16) or f32
  B      [slots, R, G, N]   bf16 bits (uint16) or f32
  dt     [slots, R, H]      fp32, the final step size
  A      [H]                fp32, negative

Value recipe: state, x, B ~ N(0,1); dt ~ U(0.001, 0.1); A = -U(0.5, 2).  One-byte
state draws its codes and its positive per-row scales at random (no quantizer
involved).  Source slots are a random permutation of the low half of the pool
per layer, destination slots one of the high half; destination slots start as
0xFF bytes so that an unwritten slot is recognisable.  The active list is a
random subset in random order, then -1s.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

STORAGE_NP = {"f32": np.float32, "bf16": np.uint16, "f16": np.float16, "i8": np.int8, "fp8_e4m3": np.uint8}
ELEM_SIZE = {"f32": 4, "bf16": 2, "f16": 2, "i8": 1, "fp8_e4m3": 1}
QUANTIZED = ("i8", "fp8_e4m3")


@dataclass(frozen=True)
class Shape:
    name: str
    L: int
    Bt: int
    H: int
    hpg: int
    D: int
    N: int
    R: int
    W: int
    state_dtype: str
    input_dtype: str = "bf16"
    A_dtype: str = "f32"
    n_active: int = 0
    pool: int = 0                 # total slots per layer; 0 -> 2*Bt (src low half, dst high half)
    ring_start: tuple = (0, 8)    # U[lo, hi)
    prefix: tuple = ("uniform", 0, 8)  # ("uniform", lo, hi_inclusive) or ("fixed", k)
    pad_frac: float = 0.0         # fraction of (layer, request) entries given a pad slot
    philox_rounds: int = 0
    rand_seed: int = 0
    pad_slot_id: int = -1
    special: str = ""             # named edge cases, see _apply_special

    @property
    def G(self) -> int:
        return self.H // self.hpg

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# The workloads, named by what they are.
SHAPES = {
    # tiny fp32: everything fits in the oracle's reach in milliseconds
    "tiny_fp32": Shape("tiny_fp32", L=2, Bt=4, H=4, hpg=2, D=16, N=16, R=8, W=8,
                       state_dtype="f32", input_dtype="f32", n_active=4, pool=16,
                       ring_start=(0, 8), prefix=("uniform", 0, 8), special="tiny"),
    # Mamba-2-2.7B-like: 64 layers, 80 heads in one group, fp32 state, forced ring wrap
    "mamba2_2p7b_fp32": Shape("mamba2_2p7b_fp32", L=64, Bt=64, H=80, hpg=80, D=64, N=128, R=16, W=16,
                              state_dtype="f32", n_active=16, ring_start=(9, 16),
                              prefix=("uniform", 0, 16), special="wrap"),
    # large hybrid 48 layers x 256 heads x 64x128, bf16 state (the headline shape)
    "hybrid48_bf16": Shape("hybrid48_bf16", L=48, Bt=256, H=256, hpg=32, D=64, N=128, R=8, W=8,
                           state_dtype="bf16", n_active=256, ring_start=(0, 8), prefix=("uniform", 0, 8)),
    "hybrid48_int8": Shape("hybrid48_int8", L=48, Bt=64, H=256, hpg=32, D=64, N=128, R=8, W=8,
                           state_dtype="i8", n_active=32, ring_start=(0, 8), prefix=("uniform", 0, 8)),
    "hybrid48_fp8_sr": Shape("hybrid48_fp8_sr", L=48, Bt=64, H=256, hpg=32, D=64, N=128, R=8, W=8,
                             state_dtype="fp8_e4m3", n_active=32, ring_start=(0, 8),
                             prefix=("uniform", 0, 8), philox_rounds=10, rand_seed=0x5EED),
    # ring/prefix sweep: long ring, fixed prefix, start near the wrap, 10% pads
    "ring_sweep_fp16": Shape("ring_sweep_fp16", L=24, Bt=128, H=128, hpg=16, D=64, N=128, R=64, W=64,
                             state_dtype="f16", n_active=128, ring_start=(56, 64),
                             prefix=("fixed", 16), pad_frac=0.10),
}


@dataclass
class HostWorld:
    """All inputs of one call, in host memory (numpy), per layer."""
    shape: Shape
    state: list
    scale: list
    x: list
    B: list
    dt: list
    A: list
    src_slots: np.ndarray
    dst_slots: np.ndarray
    ring_start: np.ndarray
    replay_prefix_len: np.ndarray
    active: np.ndarray
    rand_seed: int = 0
    meta: dict = field(default_factory=dict)

    # flat views of the shape's scalars, so the world reads like the call
    def __getattr__(self, name):
        if name in ("L", "Bt", "H", "hpg", "D", "N", "R", "W", "state_dtype", "input_dtype",
                    "A_dtype", "philox_rounds", "pad_slot_id", "G"):
            return getattr(self.shape, name)
        raise AttributeError(name)

    def copy(self) -> "HostWorld":
        cp = lambda lst: [None if a is None else a.copy() for a in lst]
        return HostWorld(self.shape, cp(self.state), cp(self.scale), cp(self.x), cp(self.B),
                         cp(self.dt), cp(self.A), self.src_slots.copy(), self.dst_slots.copy(),
                         self.ring_start.copy(), self.replay_prefix_len.copy(), self.active.copy(),
                         self.rand_seed, dict(self.meta))


def bf16_bits_from_f32(v: np.ndarray) -> np.ndarray:
    """Storage cast of random draws to bfloat16 bit patterns (torch's CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def fp8_bits_from_f32(v: np.ndarray) -> np.ndarray:
    """Storage cast of random draws to fp8 e4m3fn bit patterns (torch's CPU cast);
    draws are clipped into the finite range first."""
    import torch
    t = torch.from_numpy(np.clip(np.ascontiguousarray(v, dtype=np.float32), -440, 440))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _storage_from_normal(dtype: str, v: np.ndarray, rng) -> np.ndarray:
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_from_f32(v)
    if dtype == "f16":
        return v.astype(np.float16)
    if dtype == "i8":
        return np.clip(np.rint(v * 32.0), -127, 127).astype(np.int8)
    if dtype == "fp8_e4m3":
        return fp8_bits_from_f32(v * 64.0)
    raise ValueError(dtype)


def _input_storage(dtype: str, v: np.ndarray) -> np.ndarray:
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_from_f32(v)
    raise ValueError(dtype)


def draw_metadata(shape: Shape, rng) -> dict:
    """Slot tables, ring starts, prefix lengths and the active list."""
    L, Bt = shape.L, shape.Bt
    pool = shape.pool or 2 * Bt
    half = pool // 2
    assert half >= Bt, "pool must hold distinct source and destination slots"
    src = np.stack([rng.permutation(half)[:Bt] for _ in range(L)]).astype(np.int32)
    dst = np.stack([half + rng.permutation(pool - half)[:Bt] for _ in range(L)]).astype(np.int32)
    lo, hi = shape.ring_start
    ring_start = rng.integers(lo, hi, size=Bt).astype(np.int32)
    if shape.prefix[0] == "fixed":
        prefix = np.full(Bt, shape.prefix[1], np.int32)
    else:
        prefix = rng.integers(shape.prefix[1], shape.prefix[2] + 1, size=Bt).astype(np.int32)
    prefix = np.minimum(prefix, shape.W).astype(np.int32)
    if shape.pad_frac > 0:
        mask = rng.random((L, Bt)) < shape.pad_frac
        which = rng.random((L, Bt)) < 0.5
        src = np.where(mask & which, shape.pad_slot_id, src).astype(np.int32)
        dst = np.where(mask & ~which, shape.pad_slot_id, dst).astype(np.int32)
    n = min(shape.n_active, Bt)
    active = np.full(Bt, -1, np.int32)
    active[:n] = rng.permutation(Bt)[:n]
    meta = dict(src_slots=src, dst_slots=dst, ring_start=ring_start, replay_prefix_len=prefix,
                active=active, pool=pool)
    _apply_special(shape, meta, rng)
    return meta


def _apply_special(shape: Shape, m: dict, rng) -> None:
    if shape.special == "tiny":
        # request 1 replays nothing (exact copy); request 2 is padded on the
        # destination side in layer 0 and on the source side in layer 1
        m["replay_prefix_len"][1] = 0
        m["dst_slots"][0, 2] = shape.pad_slot_id
        if shape.L > 1:
            m["src_slots"][1, 2] = shape.pad_slot_id
    elif shape.special == "wrap":
        # one request replays the whole ring starting at its last row
        b = int(rng.integers(0, shape.Bt))
        m["ring_start"][b] = shape.R - 1
        m["replay_prefix_len"][b] = min(shape.R, shape.W)


def host_world(shape: Shape, seed: int = 0, metadata: dict | None = None) -> HostWorld:
    """Draws every input of one call into host memory."""
    rng = np.random.default_rng(seed)
    meta = metadata if metadata is not None else draw_metadata(shape, rng)
    pool = meta["pool"]
    L, H, G, D, N, R = shape.L, shape.H, shape.G, shape.D, shape.N, shape.R
    sd = shape.state_dtype
    state, scale, xs, Bs, dts, As = [], [], [], [], [], []
    for _ in range(L):
        st = _storage_from_normal(sd, rng.standard_normal((pool, H, D, N), dtype=np.float32), rng)
        st = np.ascontiguousarray(st)
        # destination half starts as 0xFF bytes
        half = pool // 2
        st.view(np.uint8).reshape(pool, -1)[half:] = 0xFF
        state.append(st)
        if sd in QUANTIZED:
            qmax = 127.0 if sd == "i8" else 448.0
            sc = (rng.uniform(0.5, 2.0, size=(pool, H, D)) * (4.0 / qmax)).astype(np.float32)
            sc.view(np.uint8).reshape(pool, -1)[half:] = 0xFF
            scale.append(sc)
        else:
            scale.append(None)
        xs.append(_input_storage(shape.input_dtype, rng.standard_normal((pool, R, H, D), dtype=np.float32)))
        Bs.append(_input_storage(shape.input_dtype, rng.standard_normal((pool, R, G, N), dtype=np.float32)))
        dts.append(rng.uniform(0.001, 0.1, size=(pool, R, H)).astype(np.float32))
        As.append((-rng.uniform(0.5, 2.0, size=H)).astype(np.float32))
    return HostWorld(shape, state, scale, xs, Bs, dts, As,
                     meta["src_slots"].copy(), meta["dst_slots"].copy(), meta["ring_start"].copy(),
                     meta["replay_prefix_len"].copy(), meta["active"].copy(),
                     rand_seed=shape.rand_seed, meta={"pool": pool, "seed": seed})


def state_bytes_per_request(shape: Shape) -> int:
    """Algorithmic state bytes one active request moves (read + write, with scales)."""
    per = shape.H * shape.D * shape.N * ELEM_SIZE[shape.state_dtype]
    if shape.state_dtype in QUANTIZED:
        per += shape.H * shape.D * 4
    return 2 * shape.L * per


def ring_bytes_per_token(shape: Shape) -> int:
    """Algorithmic ring bytes per (layer, replayed token): x per head, B per group, dt per head."""
    ie = ELEM_SIZE[shape.input_dtype]
    return shape.H * shape.D * ie + shape.G * shape.N * ie + shape.H * 4
