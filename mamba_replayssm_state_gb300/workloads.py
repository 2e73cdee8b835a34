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


# ---------------------------------------------------------------------------
# device-side worlds (torch CUDA tensors + the call's pointer tables)
# ---------------------------------------------------------------------------

TORCH_STORAGE = {"f32": "float32", "bf16": "bfloat16", "f16": "float16", "i8": "int8", "fp8_e4m3": "uint8"}


@dataclass
class DeviceWorld:
    """All inputs of one call on a CUDA device, with the call's pointer tables."""
    shape: Shape
    state: list
    scale: list
    x: list
    B: list
    dt: list
    A: list
    src_slots: object
    dst_slots: object
    ring_start: object
    replay_prefix_len: object
    active: object
    rand_seed: object
    status: object
    tables: dict
    pool: int

    def call_kwargs(self) -> dict:
        s = self.shape
        t = self.tables
        return dict(
            state_ptrs=t["state_ptrs"], state_slot_strides=t["state_slot_strides"],
            x_cache_ptrs=t["x_cache_ptrs"], x_cache_slot_strides=t["x_cache_slot_strides"],
            B_cache_ptrs=t["B_cache_ptrs"], B_cache_slot_strides=t["B_cache_slot_strides"],
            dt_cache_ptrs=t["dt_cache_ptrs"], dt_cache_slot_strides=t["dt_cache_slot_strides"],
            A_ptrs=t["A_ptrs"], state_scale_ptrs=t["state_scale_ptrs"],
            state_scale_slot_strides=t["state_scale_slot_strides"],
            src_slots=self.src_slots, dst_slots=self.dst_slots, ring_start=self.ring_start,
            replay_prefix_len=self.replay_prefix_len, active_request_indices=self.active,
            state_dtype=s.state_dtype, input_dtype=s.input_dtype, matrixA_dtype=s.A_dtype, dim=s.D,
            dstate=s.N, num_heads=s.H, heads_per_group=s.hpg, max_window=s.W, ring_buffer_len=s.R,
            pad_slot_id=s.pad_slot_id, rand_seed=self.rand_seed, philox_rounds=s.philox_rounds,
            device_status=self.status, num_slots=self.pool)

    def set_active(self, active_np) -> None:
        import torch
        self.active.copy_(torch.from_numpy(np.ascontiguousarray(active_np, np.int32)))


def _tables(state, scale, x, B, dt, A, device):
    import torch

    def ptrs(lst):
        return torch.tensor([0 if t is None else t.data_ptr() for t in lst], dtype=torch.int64, device=device)

    def strides(lst):
        return torch.tensor([0 if t is None else t.stride(0) for t in lst], dtype=torch.int64, device=device)

    return dict(state_ptrs=ptrs(state), state_slot_strides=strides(state), x_cache_ptrs=ptrs(x),
                x_cache_slot_strides=strides(x), B_cache_ptrs=ptrs(B), B_cache_slot_strides=strides(B),
                dt_cache_ptrs=ptrs(dt), dt_cache_slot_strides=strides(dt), A_ptrs=ptrs(A),
                state_scale_ptrs=ptrs(scale), state_scale_slot_strides=strides(scale))


def _np_to_torch(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a))


def _meta_tensors(meta_arrays: dict, device):
    return {k: _np_to_torch(v).to(device) for k, v in meta_arrays.items()}


def device_world_from_host(hw: HostWorld, device="cuda") -> DeviceWorld:
    """Copies a host world to the device, byte for byte."""
    import torch
    mv = lambda lst: [None if a is None else _np_to_torch(a).to(device) for a in lst]
    state, scale, x, B, dt, A = mv(hw.state), mv(hw.scale), mv(hw.x), mv(hw.B), mv(hw.dt), mv(hw.A)
    meta = _meta_tensors(dict(src_slots=hw.src_slots, dst_slots=hw.dst_slots, ring_start=hw.ring_start,
                              replay_prefix_len=hw.replay_prefix_len, active=hw.active), device)
    seed = torch.tensor([hw.rand_seed], dtype=torch.int64, device=device) if hw.philox_rounds > 0 else None
    status = torch.zeros(1, dtype=torch.int32, device=device)
    return DeviceWorld(hw.shape, state, scale, x, B, dt, A, meta["src_slots"], meta["dst_slots"],
                       meta["ring_start"], meta["replay_prefix_len"], meta["active"], seed, status,
                       _tables(state, scale, x, B, dt, A, device), hw.meta["pool"])


def device_world_random(shape: Shape, seed: int = 0, device="cuda", metadata: dict | None = None) -> DeviceWorld:
    """Draws a full-size world directly on the device (torch's seeded CUDA
    generator), same recipe as host_world; metadata is drawn on the host."""
    import torch
    rng = np.random.default_rng(seed)
    meta = metadata if metadata is not None else draw_metadata(shape, rng)
    pool = meta["pool"]
    half = pool // 2
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    L, H, G, D, N, R = shape.L, shape.H, shape.G, shape.D, shape.N, shape.R
    sd, idt = shape.state_dtype, shape.input_dtype
    tdt = getattr(torch, TORCH_STORAGE[sd])
    in_t = torch.float32 if idt == "f32" else torch.bfloat16
    state, scale, x, B, dt, A = [], [], [], [], [], []
    for _ in range(L):
        if sd in ("f32", "bf16", "f16"):
            st = torch.randn((pool, H, D, N), generator=g, device=device, dtype=tdt)
        elif sd == "i8":
            st = torch.randint(-127, 128, (pool, H, D, N), generator=g, device=device, dtype=torch.int8)
        else:  # fp8 codes: any byte except the two NaN patterns
            st = torch.randint(0, 254, (pool, H, D, N), generator=g, device=device, dtype=torch.uint8)
            st = torch.where(st >= 0x7F, st + 1, st)
        st.view(torch.uint8).view(pool, -1)[half:].fill_(0xFF)
        state.append(st)
        if sd in QUANTIZED:
            qmax = 127.0 if sd == "i8" else 448.0
            sc = torch.empty((pool, H, D), device=device, dtype=torch.float32).uniform_(0.5, 2.0, generator=g)
            sc.mul_(4.0 / qmax)
            sc.view(torch.uint8).view(pool, -1)[half:].fill_(0xFF)
            scale.append(sc)
        else:
            scale.append(None)
        x.append(torch.randn((pool, R, H, D), generator=g, device=device, dtype=in_t))
        B.append(torch.randn((pool, R, G, N), generator=g, device=device, dtype=in_t))
        dt.append(torch.empty((pool, R, H), device=device, dtype=torch.float32).uniform_(0.001, 0.1, generator=g))
        A.append(-torch.empty(H, device=device, dtype=torch.float32).uniform_(0.5, 2.0, generator=g))
    mt = _meta_tensors(dict(src_slots=meta["src_slots"], dst_slots=meta["dst_slots"],
                            ring_start=meta["ring_start"], replay_prefix_len=meta["replay_prefix_len"],
                            active=meta["active"]), device)
    seed_t = torch.tensor([shape.rand_seed], dtype=torch.int64, device=device) if shape.philox_rounds > 0 else None
    status = torch.zeros(1, dtype=torch.int32, device=device)
    return DeviceWorld(shape, state, scale, x, B, dt, A, mt["src_slots"], mt["dst_slots"], mt["ring_start"],
                       mt["replay_prefix_len"], mt["active"], seed_t, status,
                       _tables(state, scale, x, B, dt, A, device), pool)


def _to_np(t) -> np.ndarray:
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def host_subworld(dw: DeviceWorld, layer: int, request: int, k=None, rs=None) -> HostWorld:
    """A one-layer, one-request host world holding the source slot (as slot 0,
    with its ring) of (layer, request) of a device world; the destination is
    slot 1.  Used to check sampled outputs of full-size calls one by one."""
    src = int(dw.src_slots[layer, request])
    shape = dw.shape.replace(L=1, Bt=1, n_active=1, pool=2, special="", pad_frac=0.0)
    grab = lambda t: None if t is None else _to_np(t[src:src + 1])
    state = _to_np(dw.state[layer][src:src + 1])
    state = np.concatenate([state, np.full_like(state, 0)])
    state.view(np.uint8)[1:] = 0xFF
    scale = None
    if dw.scale[layer] is not None:
        sc = _to_np(dw.scale[layer][src:src + 1])
        scale = np.concatenate([sc, np.zeros_like(sc)])
        scale.view(np.uint8)[1:] = 0xFF
    x = np.concatenate([grab(dw.x[layer])] * 2)
    B = np.concatenate([grab(dw.B[layer])] * 2)
    dt = np.concatenate([grab(dw.dt[layer])] * 2)
    A = _to_np(dw.A[layer])
    kk = int(dw.replay_prefix_len[request]) if k is None else k
    rr = int(dw.ring_start[request]) if rs is None else rs
    dst = int(dw.dst_slots[layer, request])
    w = HostWorld(shape, [np.ascontiguousarray(state)], [scale], [x], [B], [dt], [A],
                  np.array([[0]], np.int32), np.array([[1]], np.int32), np.array([rr], np.int32),
                  np.array([kk], np.int32), np.array([0], np.int32),
                  rand_seed=dw.shape.rand_seed, meta={"pool": 2, "dst_slot_in_call": dst, "layer_in_call": layer})
    return w
