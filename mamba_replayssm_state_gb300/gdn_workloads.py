"""Seeded synthetic inputs for the gated-delta-rule ReplaySSM commit
(flashinfer.gdn_decode.gated_delta_rule_replayssm_commit, API page).

Like workloads.py, this module only draws random inputs and lays them out; it
holds none of the method's arithmetic, so both the CUDA path and the CPU
oracle are fed from it.

Layouts (the API page's, contiguous):
  state  [L, slots, HV, 128, 128]  fp32, K-last
  rawv   [L, slots, HV, T, 128]    bf16 bits (uint16)
  rawk   [L, slots, H, T, 128]     bf16 bits (uint16), before normalisation
  g      [L, slots, HV, T]         fp32 log-decay
  beta   [L, slots, HV, T]         fp32 sigmoid-beta

Value recipe: state, rawv ~ N(0,1); rawk ~ N(0,1) when K is normalised by the
kernel, N(0, 1/128) otherwise (so that |k| is about 1 and the update stays
contractive); g ~ -U(0.01, 2); beta ~ U(0.05, 0.95).  State slots are distinct
random slots of the low half of the pool, track slots distinct random slots of
the high half; a fraction of requests gets a null slot.  Accepted lengths are
U[0, T]; track steps U[-1, T] (some fall outside the accepted prefix).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

from .workloads import bf16_bits_from_f32

DK = DV = 128


@dataclass(frozen=True)
class GdnShape:
    name: str
    L: int
    B: int
    HV: int
    H: int
    T: int
    slots: int = 0             # 0 -> 2*B (state slots low half, track slots high half)
    accept: tuple = ("uniform",)  # ("uniform",) -> U[0, T]; ("fixed", n)
    use_qk_l2norm: bool = True
    null_block_id: int = -1
    track: bool = False
    null_frac: float = 0.0

    def replace(self, **kw) -> "GdnShape":
        return dataclasses.replace(self, **kw)

    @property
    def pool(self) -> int:
        return self.slots or 2 * self.B


GDN_SHAPES = {
    # small: the oracle finishes in well under a second
    "gdn_tiny": GdnShape("gdn_tiny", L=2, B=4, HV=4, H=2, T=8, track=True),
    # 36 linear-attention layers, 32 value heads over 16 key heads, 8-token
    # windows, 64 requests with tracking (the full-size benchmark shape)
    "gdn36_hv32_t8": GdnShape("gdn36_hv32_t8", L=36, B=64, HV=32, H=16, T=8, track=True),
}


@dataclass
class GdnWorld:
    shape: GdnShape
    state: np.ndarray
    rawv: np.ndarray
    rawk: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    state_indices: np.ndarray
    accept_lens: np.ndarray
    track_state_indices: np.ndarray | None
    track_steps: np.ndarray | None

    @property
    def use_qk_l2norm(self) -> bool:
        return self.shape.use_qk_l2norm

    @property
    def null_block_id(self) -> int:
        return self.shape.null_block_id

    def copy(self) -> "GdnWorld":
        c = lambda a: None if a is None else a.copy()
        return GdnWorld(self.shape, self.state.copy(), self.rawv.copy(), self.rawk.copy(), self.g.copy(),
                        self.beta.copy(), self.state_indices.copy(), self.accept_lens.copy(),
                        c(self.track_state_indices), c(self.track_steps))


def draw_gdn_metadata(shape: GdnShape, rng) -> dict:
    B, pool = shape.B, shape.pool
    half = pool // 2
    assert half >= B, "pool must hold distinct state and track slots"
    state_indices = rng.permutation(half)[:B].astype(np.int32)
    if shape.null_frac > 0:
        state_indices = np.where(rng.random(B) < shape.null_frac, shape.null_block_id, state_indices)
    if shape.accept[0] == "fixed":
        accept = np.full(B, shape.accept[1], np.int32)
    else:
        accept = rng.integers(0, shape.T + 1, size=B).astype(np.int32)
    track_idx = track_steps = None
    if shape.track:
        track_idx = (half + rng.permutation(pool - half)[:B]).astype(np.int32)
        track_steps = rng.integers(-1, shape.T + 1, size=B).astype(np.int32)
    return dict(state_indices=state_indices.astype(np.int32), accept_lens=accept,
                track_state_indices=track_idx, track_steps=track_steps)


def gdn_host_world(shape: GdnShape, seed: int = 0) -> GdnWorld:
    rng = np.random.default_rng(seed)
    L, SL, HV, H, T = shape.L, shape.pool, shape.HV, shape.H, shape.T
    state = rng.standard_normal((L, SL, HV, DV, DK), dtype=np.float32)
    rawv = bf16_bits_from_f32(rng.standard_normal((L, SL, HV, T, DV), dtype=np.float32))
    kscale = 1.0 if shape.use_qk_l2norm else 1.0 / np.sqrt(DK)
    rawk = bf16_bits_from_f32(kscale * rng.standard_normal((L, SL, H, T, DK), dtype=np.float32))
    g = -rng.uniform(0.01, 2.0, size=(L, SL, HV, T)).astype(np.float32)
    beta = rng.uniform(0.05, 0.95, size=(L, SL, HV, T)).astype(np.float32)
    meta = draw_gdn_metadata(shape, rng)
    return GdnWorld(shape, state, rawv, rawk, g, beta, **meta)


@dataclass
class GdnDeviceWorld:
    shape: GdnShape
    state: object
    rawv: object
    rawk: object
    g: object
    beta: object
    state_indices: object
    accept_lens: object
    track_state_indices: object
    track_steps: object
    status: object

    def call_kwargs(self) -> dict:
        return dict(checkpoint_state=self.state, rawv_cache=self.rawv, rawk_cache=self.rawk, g_cache=self.g,
                    beta_cache=self.beta, state_indices=self.state_indices, accept_lens=self.accept_lens,
                    track_state_indices=self.track_state_indices, track_steps=self.track_steps,
                    use_qk_l2norm=self.shape.use_qk_l2norm, null_block_id=self.shape.null_block_id,
                    device_status=self.status)


def _meta_to_device(meta, device):
    import torch
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)
    return dict(state_indices=t(meta["state_indices"]), accept_lens=t(meta["accept_lens"]),
                track_state_indices=t(meta["track_state_indices"]), track_steps=t(meta["track_steps"]))


def gdn_device_world_from_host(hw: GdnWorld, device="cuda") -> GdnDeviceWorld:
    """Copies a host world to the device, byte for byte."""
    import torch
    bf = lambda a: torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    meta = _meta_to_device(dict(state_indices=hw.state_indices, accept_lens=hw.accept_lens,
                                track_state_indices=hw.track_state_indices, track_steps=hw.track_steps), device)
    return GdnDeviceWorld(hw.shape, torch.from_numpy(hw.state).to(device), bf(hw.rawv), bf(hw.rawk),
                          torch.from_numpy(hw.g).to(device), torch.from_numpy(hw.beta).to(device),
                          status=torch.zeros(1, dtype=torch.int32, device=device), **meta)


def gdn_device_world_random(shape: GdnShape, seed: int = 0, device="cuda") -> GdnDeviceWorld:
    """The same recipe drawn on the device (full-size runs), with torch's
    seeded CUDA generator; metadata drawn on the host."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    L, SL, HV, H, T = shape.L, shape.pool, shape.HV, shape.H, shape.T
    state = torch.randn((L, SL, HV, DV, DK), generator=gen, device=device, dtype=torch.float32)
    rawv = torch.randn((L, SL, HV, T, DV), generator=gen, device=device).to(torch.bfloat16)
    kscale = 1.0 if shape.use_qk_l2norm else 1.0 / np.sqrt(DK)
    rawk = (kscale * torch.randn((L, SL, H, T, DK), generator=gen, device=device)).to(torch.bfloat16)
    g = -(0.01 + 1.99 * torch.rand((L, SL, HV, T), generator=gen, device=device))
    beta = 0.05 + 0.9 * torch.rand((L, SL, HV, T), generator=gen, device=device)
    meta = _meta_to_device(draw_gdn_metadata(shape, np.random.default_rng(seed)), device)
    return GdnDeviceWorld(shape, state, rawv, rawk, g, beta, status=torch.zeros(1, dtype=torch.int32, device=device),
                          **meta)


def gdn_bytes(shape: GdnShape, state_indices, accept_lens, track_state_indices, track_steps) -> int:
    """Algorithmic bytes of one call: per live request with a non-zero accepted
    length, every (layer, value head) state read and written once, the track
    copy written when the step is inside the prefix, and the windows' accepted
    rows (v per value head, k per key head, g and beta per value head)."""
    total = 0
    head = DV * DK * 4
    for b in range(len(state_indices)):
        n = int(accept_lens[b])
        if state_indices[b] <= shape.null_block_id or n == 0:
            continue
        per_layer = shape.HV * 2 * head
        if track_state_indices is not None and track_state_indices[b] > shape.null_block_id and \
                0 <= track_steps[b] < n:
            per_layer += shape.HV * head
        per_layer += n * (shape.HV * DV * 2 + shape.H * DK * 2 + shape.HV * 8)
        total += shape.L * per_layer
    return total
