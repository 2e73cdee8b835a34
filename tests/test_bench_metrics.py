"""The benchmark's roofline arithmetic on the CPU: algorithmic bytes per call
against their closed form, and the committed profile traffic it reports only
while the kernel sources match the profile."""
import importlib.util
import os

import numpy as np
import pytest

from mamba_replayssm_state_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _meta(shape, n, k, pad=None):
    Bt, L = shape.Bt, shape.L
    active = np.full(Bt, -1, np.int32)
    active[:n] = np.arange(n)
    src = np.tile(np.arange(Bt, dtype=np.int32), (L, 1))
    dst = src + Bt
    if pad is not None:
        src[pad] = shape.pad_slot_id
    prefix = np.full(Bt, k, np.int32)
    return active, prefix, src, dst


@pytest.mark.parametrize("k", [0, 4, 8])
def test_headline_bytes_match_the_closed_form(bench, k):
    """48 layers x 256 heads x 64x128 bf16: 402,653,184 B of state read and
    written per request, plus 48 * k * 35,840 B of ring (x 256*64*2, B 8*128*2,
    dt 256*4 per token and layer)."""
    shape = wl.SHAPES["hybrid48_bf16"]
    n = 256
    state_b, ring_b, got_n = bench.workload_bytes(shape, *_meta(shape, n, k))
    assert got_n == n
    assert state_b == n * 402_653_184
    assert ring_b == n * 48 * k * 35_840


def test_one_byte_state_adds_scales_and_pads_are_skipped(bench):
    shape = wl.SHAPES["hybrid48_int8"]
    n, k = 32, 5
    active, prefix, src, dst = _meta(shape, n, k, pad=(3, 7))  # layer 3 of request 7 padded
    state_b, ring_b, _ = bench.workload_bytes(shape, active, prefix, src, dst)
    tile = 256 * 64 * 128 * 1 + 256 * 64 * 4  # codes + per-row fp32 scales
    pairs = n * shape.L - 1
    assert state_b == pairs * 2 * tile
    assert ring_b == pairs * k * (256 * 64 * 2 + 8 * 128 * 2 + 256 * 4)


def test_active_list_ends_at_the_first_terminator(bench):
    shape = wl.SHAPES["hybrid48_bf16"].replace(Bt=8)
    active, prefix, src, dst = _meta(shape, 8, 2)
    active[3] = -1  # entries after the first -1 are not requests
    _, _, n = bench.workload_bytes(shape, active, prefix, src, dst)
    assert n == 3


def test_profile_traffic_follows_the_source_hash(bench):
    """The committed headline summary's traffic is reported for the sources it
    was taken on, and for no others."""
    import re
    text = open(os.path.join(ROOT, "profiles", "materialize_kernel_hybrid48_bf16.md")).read()
    taken_on = re.search(r"source_hash:\s*([0-9a-f]+)", text).group(1)
    traffic = bench.profile_traffic("hybrid48_bf16", taken_on)
    assert traffic is not None and 9.0e10 < traffic < 1.1e11
    current = bench.kernel_source_hash()
    assert (bench.profile_traffic("hybrid48_bf16", current) is not None) == (current == taken_on)
    assert bench.profile_traffic("hybrid48_bf16", "0" * 16) is None
    assert bench.profile_traffic("no_such_workload", taken_on) is None


def test_lane_operations_and_philox_fraction(bench):
    """Per replayed element: k FFMA + 1 FMUL; with Philox rounding one call
    (10 rounds x 6 integer operations, four words) per 16 one-byte or 8
    16-bit elements; copies cost nothing."""
    for name, per_call in (("hybrid48_fp8_sr", 16), ("hybrid48_bf16", 8)):
        shape = wl.SHAPES[name].replace(philox_rounds=10)
        n, k = 4, 3
        active, prefix, src, dst = _meta(shape, n, k, pad=(0, 1))
        prefix[2] = 0                                    # request 2 is a copy
        fp32, integer, words, flops = bench.lane_ops(shape, active, prefix, src, dst)
        elems = 256 * 64 * 128
        live = (n - 1) * shape.L - 1                     # one copy request, one padded layer
        assert fp32 == live * elems * (k + 1) and flops == 0
        assert integer == int(live * elems * 60 / per_call)
        assert words == live * elems * 4 // per_call
        # the replay on the tensor cores: 2 FLOPs per element and token there,
        # one FFMA per element on the lanes
        fp32_t, integer_t, words_t, flops_t = bench.lane_ops(shape, active, prefix, src, dst, tensor=True)
        assert fp32_t == live * elems and flops_t == live * elems * 2 * k
        assert (integer_t, words_t) == (integer, words)
    fr = bench._fractions(1e9, fp32, integer, 1.0, 6790.0, 152, {"sm_mhz": 2070.0}, words, 10)
    words_peak = 6.8 * 152 * 2070e6
    assert abs(fr["philox_frac"] - words / 1e-3 / words_peak) < 1e-12
    assert "philox_frac" not in bench._fractions(1e9, 1, 0, 1.0, 6790.0, 152, None)
    ft = bench._fractions(1e9, 1, 0, 1.0, 6790.0, 152, None, tensor_flops=1.9e12, tensor_peak=1.9e15)
    assert abs(ft["tensor_frac"] - 1.0) < 1e-12 and ft["bound"] == "tensor"
    assert "tensor_frac" not in bench._fractions(1e9, 1, 0, 1.0, 6790.0, 152, None)
