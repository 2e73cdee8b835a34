#!/usr/bin/env python
"""Benchmark of ReplaySSM prefix materialization on GB300.

Workload (default): the large-hybrid shape, 48 layers x 256 heads x 64x128
bf16 state, bf16 x/B rings of 8 rows, fp32 dt/A, batch 256 with all 256
requests active and replay_prefix_len ~ U[0, 8].  One step = one call of the
whole path (one kernel launch over every layer).  Inputs are synthetic and
seeded, drawn on the device; 51.5 GB of state move per step, far more than L2.

Printed (rank 0, one JSON line): state GB/s of the step (`value`), ms per
step, microseconds per active request ((T(n) - T(0)) / n, the "additional
cost" convention) for n in {1, 16, 256}, the empty-list latency, the roofline
of the kernel against the measured HBM copy bandwidth, an end-to-end figure
through the public API with pinned host buffers, the oracle timed on a
bounded sample on the host cores, and the SM clocks seen while timing.

`--impl reference` times the CPU oracle (the only reference this method has)
on bounded samples of the same workload instead.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mamba_replayssm_state_gb300 import dist  # noqa: E402
from mamba_replayssm_state_gb300 import gdn_workloads as gw  # noqa: E402
from mamba_replayssm_state_gb300 import workloads as wl  # noqa: E402

METRIC = "state GB/s & µs/active request (48L×256H×64×128); empty-active-list µs"
KERNEL_NAME = "materialize_kernel"
SPEC_HBM_GBS = 8000.0  # the GB300's nominal HBM3e bandwidth, the denominator the target is stated against
_CSRC = "mamba_replayssm_state_gb300/csrc/"
_SHARED_SOURCES = ["include/replayssm.h", _CSRC + "rsm_api.cu", _CSRC + "rsm_ptx.cuh", _CSRC + "rsm_params.h",
                   _CSRC + "rsm_instances.h"]
# every source file whose edit can change a kernel's code, per kernel: a profile
# summary is valid only for the hash of the files it was taken on
KERNEL_SOURCES = {
    "materialize_kernel": _SHARED_SOURCES + [_CSRC + f for f in (
        "rsm_kernel.cuh", "rsm_formats.cuh", "rsm_inst_f32.cu", "rsm_inst_bf16.cu", "rsm_inst_f16.cu")],
    "materialize_q8_kernel": _SHARED_SOURCES + [_CSRC + f for f in (
        "rsm_kernel.cuh", "rsm_formats.cuh", "rsm_q8_kernel.cuh", "rsm_inst_q8.cu", "rsm_inst_q8sr.cu")],
    "materialize_tc_kernel": _SHARED_SOURCES + [_CSRC + f for f in (
        "rsm_kernel.cuh", "rsm_formats.cuh", "rsm_tc_kernel.cuh", "rsm_tc.cuh", "rsm_inst_tc.cu")],
    "materialize_q8tc_kernel": _SHARED_SOURCES + [_CSRC + f for f in (
        "rsm_kernel.cuh", "rsm_formats.cuh", "rsm_q8tc_kernel.cuh", "rsm_tc.cuh", "rsm_inst_q8tc.cu")],
    "gdn_commit_kernel": _SHARED_SOURCES + [_CSRC + f for f in ("gdn_kernel.cuh", "gdn_params.h", "gdn_inst.cu")],
    "gdn_commit_tc_kernel": _SHARED_SOURCES + [_CSRC + f for f in (
        "gdn_tc_kernel.cuh", "gdn_params.h", "gdn_inst.cu", "rsm_tc.cuh")],
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", default="hybrid48_bf16", choices=sorted(wl.SHAPES))
    p.add_argument("--n-active", type=int, default=None, help="active requests per step (default: the workload's)")
    p.add_argument("--batch", type=int, default=None, help="batch size (default: the workload's)")
    p.add_argument("--prefix", type=int, default=None, help="fixed replay_prefix_len for every request")
    p.add_argument("--state-dtype", default=None, choices=sorted(wl.ELEM_SIZE), help="override the state format")
    p.add_argument("--input-dtype", default=None, choices=["bf16", "f32"], help="override the x/B input format")
    p.add_argument("--window", type=int, default=None, help="override max_window (and ring_buffer_len)")
    p.add_argument("--no-extras", action="store_true", help="skip the n sweep, empty latency, e2e and CPU baseline")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work for the oracle baseline sample")
    p.add_argument("--e2e-requests", type=int, default=16)
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--all-workloads", action="store_true",
                   help="measure the other named workloads even with --no-extras")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other named workloads (measured by default, under 'workloads')")
    p.add_argument("--only", default=None,
                   help="comma-separated names of the named workloads to measure (default: all of them)")
    p.add_argument("--gdn", action="store_true",
                   help="measure only the gated-delta-rule commit (gdn36_hv32_t8; --batch overrides B)")
    p.add_argument("--gdn-backend", default="auto", choices=["auto", "simt", "tcgen05"],
                   help="the commit's backend with --gdn (tcgen05: the shape without tracking)")
    return p.parse_args()


def kernel_source_hash(kernel: str = KERNEL_NAME) -> str:
    """SHA-256 prefix of every source file that builds `kernel`."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def workload_bytes(shape, active, prefix, src, dst):
    """Algorithmic bytes of one call: state read + write (+ scales) of every
    non-padded (layer, request), and the ring rows it replays (x per head,
    B per group, dt per head)."""
    import numpy as np
    n = int(np.argmax(active == -1)) if (active == -1).any() else len(active)
    es = wl.ELEM_SIZE[shape.state_dtype]
    tile = shape.H * shape.D * shape.N * es + (shape.H * shape.D * 4 if shape.state_dtype in wl.QUANTIZED else 0)
    per_tok = wl.ring_bytes_per_token(shape)
    state_b = ring_b = 0
    for b in active[:n]:
        b = int(b)
        for l in range(shape.L):
            if src[l, b] == shape.pad_slot_id or dst[l, b] == shape.pad_slot_id:
                continue
            state_b += 2 * tile
            ring_b += int(prefix[b]) * per_tok
    return state_b, ring_b, n


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while timing."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_uuid=None):
        self.proc = None
        self.uuid = device_uuid
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]
        sm, smax, reasons, power = [], [], set(), []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(self.REASONS, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def profile_traffic(workload: str, src_hash: str, kernel: str = KERNEL_NAME):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_hash = re.search(r"source_hash:\s*([0-9a-f]+)", txt)
    m_bytes = re.search(r"dram_bytes_per_launch_full:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_bytes or m_hash.group(1) != src_hash:
        return None
    return float(m_bytes.group(1))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            return float(json.load(open(path))["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return 6800.0, "fallback"


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ----------------------------------------------------------------------------

def oracle_pair_seconds(hw):
    import oracle
    w = hw.copy()
    t0 = time.perf_counter()
    oracle.materialize(w)
    return time.perf_counter() - t0


def oracle_parallel_seconds(worlds, threads):
    """Wall time of the oracle over independent host worlds on `threads`
    threads (the C oracle runs outside Python's lock, so the threads run it
    on as many cores)."""
    import concurrent.futures
    import oracle
    copies = [w.copy() for w in worlds]
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(oracle.materialize, copies))
    return time.perf_counter() - t0


def cpu_baseline_from_device(dw, shape, seconds):
    """Times the oracle, as it stands, on (layer, request) pairs of the device
    world (their inputs copied to the host): single-threaded until ~`seconds`
    of CPU work, then the same pairs spread over every host core."""
    import numpy as np
    active = dw.active.cpu().numpy()
    n = int(np.argmax(active == -1)) if (active == -1).any() else len(active)
    rng = np.random.default_rng(123)
    spent, pairs, state_b = 0.0, 0, 0
    tile = shape.H * shape.D * shape.N * wl.ELEM_SIZE[shape.state_dtype]
    subs = []
    while spent < seconds and pairs < 400:
        l = int(rng.integers(shape.L))
        b = int(active[int(rng.integers(n))])
        sub = wl.host_subworld(dw, l, b)
        spent += oracle_pair_seconds(sub)
        pairs += 1
        state_b += 2 * tile
        if len(subs) < 64:
            subs.append(sub)
    single = state_b / spent / 1e9
    cores = os.cpu_count() or 1
    # at least two pairs per core, so that every core stays busy
    batch = (subs * ((2 * cores + len(subs) - 1) // len(subs)))[: max(2 * cores, len(subs))]
    wall = oracle_parallel_seconds(batch, cores)
    multi = len(batch) * 2 * tile / wall / 1e9
    return {"value": multi, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(batch)} (layer, request) pairs of the timed workload on {cores} threads "
                      f"({wall:.1f} s wall); single-threaded, {pairs} pairs took {spent:.1f} s",
            "single_thread_value": single,
            "us_per_request": spent / pairs * shape.L * 1e6}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle timed on bounded samples of the workload."""
    if rank != 0:
        return 0
    import numpy as np
    shape = wl.SHAPES[args.workload]
    one = shape.replace(L=1, Bt=1, n_active=1, pool=2, special="", pad_frac=0.0)
    tile = shape.H * shape.D * shape.N * wl.ELEM_SIZE[shape.state_dtype]
    rng = np.random.default_rng(0)

    cores = os.cpu_count() or 1

    def world(seed):
        meta = wl.draw_metadata(one, np.random.default_rng(seed))
        return wl.host_world(one, seed=seed, metadata=meta)

    # one step: `cores` independent (layer, request) pairs on `cores` threads
    for i in range(args.warmup):
        oracle_parallel_seconds([world(10_000 + 100 * i + c) for c in range(cores)], cores)
    times = []
    for _ in range(args.steps):
        worlds = [world(int(rng.integers(1 << 30))) for _ in range(cores)]
        times.append(oracle_parallel_seconds(worlds, cores))
    total = sum(times)
    gbs = args.steps * cores * 2 * tile / total / 1e9
    sample = (f"each step: {cores} (layer, request) pairs of {shape.name} (all {shape.H} heads, prefix ~ the "
              f"workload's distribution), the C oracle on {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name, "layers": shape.L, "heads": shape.H, "dim": shape.D,
                   "dstate": shape.N, "state_dtype": shape.state_dtype, "batch": shape.Bt,
                   "sample": f"{cores} (layer, request) pairs per step"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "us_per_request": total / args.steps / cores * shape.L * 1e6,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def time_graph(torch, fn_list, reps=3):
    """Mean device time (ms) of one launch, from a CUDA graph of the given launches."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for fn in fn_list[:2]:
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for fn in fn_list:
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * len(fn_list))


def bind_to_gpu_numa_node(torch, device):
    """Runs this process on the CPUs of the NUMA node closest to `device` (so
    that pinned host buffers allocated next are local to the GPU's CPU link);
    returns that node, or None when the topology cannot be read."""
    try:
        prop = torch.cuda.get_device_properties(device)
        bus = f"{prop.pci_domain_id:04x}:{prop.pci_bus_id:02x}:{prop.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        if cpus:
            os.sched_setaffinity(0, cpus)
        return node
    except (OSError, ValueError, AttributeError):
        return None


def e2e_measure(torch, rsm, shape, n_req, steps, device, groups=8):
    """End to end through the public API: every step copies the inputs of n_req
    requests (their source state slots, rings and the call's metadata) from
    pinned host memory, materializes, and copies the destination slots back.
    The layers go through in `groups` groups, one public call each, on three
    streams: group g's inputs go up while group g-1 computes and group g-2's
    results come back (host-to-device and device-to-host copies overlap)."""
    import numpy as np
    saved_affinity = os.sched_getaffinity(0)
    node = bind_to_gpu_numa_node(torch, device)
    sh = shape.replace(Bt=n_req, n_active=n_req)
    meta = wl.draw_metadata(sh, np.random.default_rng(77))
    # contiguous source block (slots 0..n-1) and destination block (n..2n-1) per layer
    meta["src_slots"] = np.tile(np.arange(n_req, dtype=np.int32), (sh.L, 1))
    meta["dst_slots"] = np.tile(np.arange(n_req, 2 * n_req, dtype=np.int32), (sh.L, 1))
    dw = wl.device_world_random(sh, seed=77, device=device, metadata=meta)
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    h_state = [pin(s[:n_req]) for s in dw.state]
    h_x = [pin(x[:n_req]) for x in dw.x]
    h_B = [pin(b[:n_req]) for b in dw.B]
    h_dt = [pin(d[:n_req]) for d in dw.dt]
    h_meta = {k: pin(getattr(dw, k)) for k in ("src_slots", "dst_slots", "ring_start", "replay_prefix_len",
                                               "active")}
    h_out = [torch.empty(s[n_req:].shape, dtype=s.dtype, pin_memory=True) for s in dw.state]
    h2d = sum(t.numel() * t.element_size() for t in h_state + h_x + h_B + h_dt + list(h_meta.values()))
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    # one public call per layer group: the per-layer tables and slot rows sliced
    bounds = np.linspace(0, sh.L, groups + 1).astype(int)
    spans = [(int(bounds[g]), int(bounds[g + 1])) for g in range(groups) if bounds[g + 1] > bounds[g]]
    calls = [rsm.prepare(**dist.layer_shard_kwargs(dw.call_kwargs(), l0, l1)) for l0, l1 in spans]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ng = len(spans)
    ev_in = [torch.cuda.Event() for _ in range(ng)]
    ev_cmp = [torch.cuda.Event() for _ in range(ng)]
    ev_out = [torch.cuda.Event() for _ in range(ng)]
    first = [True]

    def one_step():
        with torch.cuda.stream(s_in):
            for k, t in h_meta.items():
                getattr(dw, k).copy_(t, non_blocking=True)
            for g, (l0, l1) in enumerate(spans):
                if not first[0]:
                    s_in.wait_event(ev_cmp[g])  # the previous step has read these source slots
                for l in range(l0, l1):
                    dw.state[l][:n_req].copy_(h_state[l], non_blocking=True)
                    dw.x[l][:n_req].copy_(h_x[l], non_blocking=True)
                    dw.B[l][:n_req].copy_(h_B[l], non_blocking=True)
                    dw.dt[l][:n_req].copy_(h_dt[l], non_blocking=True)
                ev_in[g].record(s_in)
        for g in range(ng):
            s_cmp.wait_event(ev_in[g])
            if not first[0]:
                s_cmp.wait_event(ev_out[g])  # the previous step's results have left
            calls[g](s_cmp)
            ev_cmp[g].record(s_cmp)
        with torch.cuda.stream(s_out):
            for g, (l0, l1) in enumerate(spans):
                s_out.wait_event(ev_cmp[g])
                for l in range(l0, l1):
                    h_out[l].copy_(dw.state[l][n_req:], non_blocking=True)
                ev_out[g].record(s_out)
        first[0] = False

    for _ in range(3):
        one_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / steps
    state_b, _, _ = workload_bytes(sh, meta["active"], meta["replay_prefix_len"], meta["src_slots"],
                                   meta["dst_slots"])
    del dw, h_state, h_x, h_B, h_dt, h_out, calls
    torch.cuda.empty_cache()
    os.sched_setaffinity(0, saved_affinity)
    return {"value": state_b / sec / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": sec * 1e3, "host_numa_node": node,
            "workload": f"{sh.name} with {n_req} active requests, inputs from pinned host memory, "
                        f"{ng} layer groups streamed through the public call (copies in, compute and copies out "
                        f"overlapped on three streams)"}


ALU_LANES_PER_SM = 128  # FP32 lanes per SM (Blackwell: 4 sub-partitions x 32)
INT_LANES_PER_SM = 64   # 32-bit integer lanes per SM (4 sub-partitions x 16): LOP3, IADD3, SHF, IMAD
# Philox-4x32 output words per SM per clock at 10 rounds, measured on GB300 by
# a loop of independent generator calls (bound by the 32x32->64-bit multiplies);
# the rate scales as 10 / rounds.  Stochastic rounding uses 16 bits per element.
PHILOX10_WORDS_PER_SM_CLK = 6.8


# kernels whose replay (sum_t w_t x_t B_t^T) runs on the tensor cores
TENSOR_KERNELS = {"materialize_tc_kernel", "materialize_q8tc_kernel", "gdn_commit_tc_kernel"}
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense TF32 : BF16 tensor rate of the part


def tensor_peak_flops():
    """Dense bf16 tensor FLOP/s: the measured burst GEMM rate, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            return float(json.load(open(path))["bf16_tflops"]) * 1e12
        except (KeyError, ValueError):
            pass
    return 1.9e15


def lane_ops(shape, active, prefix, src, dst, tensor=False):
    """(fp32 lane-operations, 32-bit integer lane-operations, Philox words,
    tensor FLOPs) one call needs, counted from the method, not from the code.
    Per element of a replayed tile: one FMUL (the decay product) and one FFMA
    per token; where the replay runs on the tensor cores (`tensor`), the
    tokens' multiply-adds are tensor FLOPs (2 per element and token) and one
    FFMA per element (P S_0 + the accumulator) stays on the lanes.
    With Philox rounding, one call (four words) serves 8 elements of 16-bit
    state or 16 of one-byte state, and costs philox_rounds * 6 integer
    operations (a round is two 32x32->64-bit multiplies, two three-way XORs
    and two key additions); the rounding decision itself is the conversion
    instruction's (bf16, f16, fp8) and is not counted.  Copies (prefix 0) cost
    nothing."""
    import numpy as np
    n = int(np.argmax(active == -1)) if (active == -1).any() else len(active)
    elems = shape.H * shape.D * shape.N
    per_call = 16 if wl.ELEM_SIZE[shape.state_dtype] == 1 else 8
    fp32 = integer = words = flops = 0
    for b in active[:n]:
        b = int(b)
        k = int(prefix[b])
        if k == 0:
            continue
        live = sum(1 for l in range(shape.L) if src[l, b] != shape.pad_slot_id and dst[l, b] != shape.pad_slot_id)
        if tensor:
            fp32 += live * elems
            flops += live * elems * 2 * k
        else:
            fp32 += live * elems * (k + 1)
        if shape.philox_rounds > 0:
            integer += live * elems * shape.philox_rounds * 6 / per_call
            words += live * elems * 4 // per_call
    return fp32, int(integer), words, flops


def timed_calls(torch, call, stream, uuid, seconds=1.0):
    """Device time per call (ms) over about `seconds` of back-to-back calls,
    with the SM clocks sampled while they run (the sampler needs ~1 s)."""
    for _ in range(3):
        call(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(3):
        call(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    one = e0.elapsed_time(e1) / 3
    steps = int(min(5000, max(20, seconds * 1e3 / max(one, 1e-3))))
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    e0.record(stream)
    for _ in range(steps):
        call(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    info = clocks.stop()
    return e0.elapsed_time(e1) / steps, steps, info


def _fractions(nbytes, fp32_ops, int_ops, ms, peak_gbs, sms, clock_info, words=0, rounds=0, tensor_flops=0,
               tensor_peak=0.0):
    mhz = (clock_info or {}).get("sm_mhz") or 2070.0
    sec = ms * 1e-3
    fr = {"hbm_frac": nbytes / sec / 1e9 / peak_gbs, "hbm_frac_spec": nbytes / sec / 1e9 / SPEC_HBM_GBS,
          "fp32_lane_frac": fp32_ops / sec / (sms * ALU_LANES_PER_SM * mhz * 1e6),
          "int_lane_frac": int_ops / sec / (sms * INT_LANES_PER_SM * mhz * 1e6)}
    if rounds > 0:
        # Philox words the rounding needs against the measured generator rate
        words_peak = PHILOX10_WORDS_PER_SM_CLK * 10.0 / rounds * sms * mhz * 1e6
        fr["philox_frac"] = words / sec / words_peak
    cands = [("hbm", fr["hbm_frac"]), ("fp32", fr["fp32_lane_frac"]), ("int", fr["int_lane_frac"])]
    if "philox_frac" in fr:
        cands.append(("philox", fr["philox_frac"]))
    if tensor_flops:
        fr["tensor_frac"] = tensor_flops / sec / tensor_peak
        cands.append(("tensor", fr["tensor_frac"]))
    fr["bound"] = max(cands, key=lambda kv: kv[1])[0]
    return fr


def measure_workload(torch, rsm, shape, device, peak_gbs, sms, uuid):
    """State GB/s, microseconds per active request and roofline fractions of
    one named workload (its own seeded world, timed with CUDA events over
    about a second, clocks sampled meanwhile)."""
    dw = wl.device_world_random(shape, seed=5, device=device)
    active = dw.active.cpu().numpy()
    prefix = dw.replay_prefix_len.cpu().numpy()
    src, dst = dw.src_slots.cpu().numpy(), dw.dst_slots.cpu().numpy()
    state_b, ring_b, n = workload_bytes(shape, active, prefix, src, dst)
    kw = dw.call_kwargs()
    call = rsm.prepare(**kw)
    kernel = rsm.kernel_name(**kw)
    fp32_ops, int_ops, words, tflops = lane_ops(shape, active, prefix, src, dst, tensor=kernel in TENSOR_KERNELS)
    launch = rsm.launch_config(**kw)
    ms, steps, clock_info = timed_calls(torch, call, torch.cuda.current_stream(), uuid)
    status = int(dw.status.item())
    del dw, call, kw
    torch.cuda.empty_cache()
    out = {"kernel": kernel, "source_hash": kernel_source_hash(kernel), "launch": launch,
           "state_dtype": shape.state_dtype,
           "layers": shape.L, "heads": shape.H, "batch": shape.Bt, "n_active": n, "prefix": list(shape.prefix),
           "philox_rounds": shape.philox_rounds, "pad_frac": shape.pad_frac, "ms_per_call": ms, "steps": steps,
           "algorithmic_bytes": state_b + ring_b, "state_gbs": state_b / (ms * 1e-3) / 1e9,
           "us_per_request": ms * 1e3 / max(n, 1), "fp32_lane_ops": fp32_ops, "int_lane_ops": int_ops}
    if tflops:
        out["tensor_flops"] = tflops
    out.update(_fractions(state_b + ring_b, fp32_ops, int_ops, ms, peak_gbs, sms, clock_info, words,
                          shape.philox_rounds, tflops, tensor_peak_flops()))
    out["clocks"] = clock_info
    out["device_status"] = status
    return out


def measure_gdn(torch, rsm, shape, device, peak_gbs, sms, uuid, backend="auto"):
    """Time of one gated-delta-rule commit call over a seeded full-size world
    (state updated in place, so every timed call is a fresh commit of the same
    shape), its algorithmic bytes against the HBM peak, and its FP32 lane
    operations (per element and accepted token: the dot-product FMA, the decay
    multiply and the update FMA) against the lane peak.  `backend` as the
    call's ("tcgen05": the TF32 tensor-core kernel, no tracking)."""
    dw = gw.gdn_device_world_random(shape, seed=5, device=device)
    kw = dw.call_kwargs()
    kw["backend"] = backend
    idx, lens = dw.state_indices.cpu().numpy(), dw.accept_lens.cpu().numpy()
    tidx = None if dw.track_state_indices is None else dw.track_state_indices.cpu().numpy()
    tst = None if dw.track_steps is None else dw.track_steps.cpu().numpy()
    nbytes = gw.gdn_bytes(shape, idx, lens, tidx, tst)
    live = [b for b in range(shape.B) if idx[b] > shape.null_block_id and lens[b] > 0]
    tokens = sum(int(lens[b]) for b in live) * shape.L * shape.HV * gw.DV * gw.DK
    if backend == "tcgen05":  # the two contractions (W = S0 K^, the rank-n update) in TF32 on the tensor cores
        lane_ops_, tflops = tokens, 4 * tokens
    else:
        lane_ops_, tflops = 3 * tokens, 0
    stream = torch.cuda.current_stream()
    call = lambda st: rsm.gated_delta_rule_replayssm_commit(**kw, stream=st)
    ms, steps, clock_info = timed_calls(torch, call, stream, uuid)
    status = int(dw.status.item())
    del dw, kw
    torch.cuda.empty_cache()
    kernel = "gdn_commit_tc_kernel" if backend == "tcgen05" else "gdn_commit_kernel"
    out = {"kernel": kernel, "source_hash": kernel_source_hash(kernel), "backend": backend,
           "layers": shape.L, "v_heads": shape.HV, "k_heads": shape.H, "window": shape.T, "batch": shape.B,
           "live_requests": len(live), "track": shape.track, "accept": list(shape.accept), "ms_per_call": ms,
           "steps": steps, "algorithmic_bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9}
    if tflops:
        out["tensor_flops"] = tflops
    out.update(_fractions(nbytes, lane_ops_, 0, ms, peak_gbs, sms, clock_info, tensor_flops=tflops,
                          tensor_peak=tensor_peak_flops() * TF32_PER_BF16))
    out["clocks"] = clock_info
    out["device_status"] = status
    return out


def named_workloads():
    """The other named workloads, each at its full size on one GPU: the
    Mamba-2-like fp32 state, int8 state, fp8 state with Philox stochastic
    rounding and with round-to-nearest, the 64-token ring sweep at every
    prefix length, and the gated-delta-rule commit.  name -> (kind, shape)."""
    out = {name: ("materialize", wl.SHAPES[name]) for name in ("mamba2_2p7b_fp32", "hybrid48_int8", "hybrid48_fp8_sr")}
    out["hybrid48_fp8_rne"] = ("materialize",
                               wl.SHAPES["hybrid48_fp8_sr"].replace(name="hybrid48_fp8_rne", philox_rounds=0))
    for k in (0, 1, 4, 16, 64):
        out[f"ring_sweep_fp16_k{k}"] = ("materialize", wl.SHAPES["ring_sweep_fp16"].replace(prefix=("fixed", k)))
    gshape = gw.GDN_SHAPES["gdn36_hv32_t8"]
    out["gdn36_hv32_t8"] = ("gdn", gshape)
    out["gdn36_hv32_t8_full"] = ("gdn", gshape.replace(accept=("fixed", 8)))
    # the two backends side by side on the conditions the tcgen05 one takes (no tracking)
    out["gdn36_hv32_t8_notrack"] = ("gdn", gshape.replace(track=False))
    out["gdn36_hv32_t8_notrack_tcgen05"] = ("gdn_tcgen05", gshape.replace(track=False))
    return out


def measure_named_workloads(torch, rsm, device, peak_gbs, sms, uuid, only=None):
    sweep = {}
    for name, (kind, shape) in named_workloads().items():
        if only and name not in only:
            continue
        if kind == "gdn_tcgen05":
            sweep[name] = measure_gdn(torch, rsm, shape, device, peak_gbs, sms, uuid, backend="tcgen05")
            continue
        measure = measure_gdn if kind == "gdn" else measure_workload
        sweep[name] = measure(torch, rsm, shape, device, peak_gbs, sms, uuid)
    return sweep


def main():
    args = parse_args()
    rank, local_rank, world = dist.env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch

    import mamba_replayssm_state_gb300 as rsm
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist.init("nccl")
    rsm.load_library()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        uuid = None
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peak, peak_kind = measured_peak()

    if args.gdn:
        gshape = gw.GDN_SHAPES["gdn36_hv32_t8"]
        if args.batch is not None:
            gshape = gshape.replace(B=args.batch)
        if args.prefix is not None:
            gshape = gshape.replace(accept=("fixed", args.prefix))
        if args.gdn_backend == "tcgen05":
            gshape = gshape.replace(track=False)
        res = measure_gdn(torch, rsm, gshape, device, peak, sms, uuid, backend=args.gdn_backend)
        if rank == 0:
            print(json.dumps({"metric": "gated-delta-rule commit: algorithmic GB/s", "unit": "GB/s",
                              "value": res["gbs"], "peak_gbs": peak, "peak_source": peak_kind, **res}), flush=True)
        return 0

    shape = wl.SHAPES[args.workload]
    if args.batch is not None:
        shape = shape.replace(Bt=args.batch, n_active=min(shape.n_active, args.batch))
    if args.n_active is not None:
        shape = shape.replace(n_active=args.n_active)
    if args.prefix is not None:
        shape = shape.replace(prefix=("fixed", args.prefix))
    if args.state_dtype is not None:
        shape = shape.replace(state_dtype=args.state_dtype)
    if args.input_dtype is not None:
        shape = shape.replace(input_dtype=args.input_dtype)
    if args.window is not None:
        shape = shape.replace(W=args.window, R=max(args.window, shape.R),
                              ring_start=(0, max(args.window, shape.R)))
    # each rank materializes its own batch (weak scaling: independent shards)
    dw = wl.device_world_random(shape, seed=1000 * rank, device=device)
    active = dw.active.cpu().numpy()
    prefix = dw.replay_prefix_len.cpu().numpy()
    src, dst = dw.src_slots.cpu().numpy(), dw.dst_slots.cpu().numpy()
    state_b, ring_b, n = workload_bytes(shape, active, prefix, src, dst)
    call = rsm.prepare(**dw.call_kwargs())
    cfg = rsm.launch_config(**dw.call_kwargs())
    stream = torch.cuda.current_stream()

    clocks = ClockSampler(uuid)

    for _ in range(max(args.warmup, 0)):
        call(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    e0.record(stream)
    for _ in range(args.steps):
        call(stream)
    e1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    dist.barrier()
    clock_info = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = dist.max_over_ranks(ms, device)
    status = int(dw.status.item())

    out = {
        "metric": METRIC,
        "value": world * state_b / (ms_max * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": shape.name, "layers": shape.L, "heads": shape.H, "heads_per_group": shape.hpg,
                   "dim": shape.D, "dstate": shape.N, "state_dtype": shape.state_dtype,
                   "input_dtype": shape.input_dtype, "batch": shape.Bt, "n_active": n,
                   "ring_buffer_len": shape.R, "max_window": shape.W,
                   "prefix": "U[0,8]" if shape.prefix[0] == "uniform" else f"fixed {shape.prefix[1]}",
                   "l2": f"inputs larger than L2 ({state_b / 1e9:.1f} GB of state per step), no flush",
                   "launch": cfg, "parallelism": f"dp{world} (independent request shards)" if world > 1 else "1 GPU"},
        "gpu_launches": args.steps,
        "device_status": status,
    }
    achieved = (state_b + ring_b) / (ms * 1e-3) / 1e9
    kernel = rsm.kernel_name(**dw.call_kwargs())
    src_hash = kernel_source_hash(kernel)
    traffic = profile_traffic(shape.name, src_hash, kernel) if n == shape.Bt else None
    out["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                       "frac": achieved / peak, "traffic": traffic,
                       "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                       "frac_spec": achieved / SPEC_HBM_GBS, "spec_peak": SPEC_HBM_GBS,
                       "spec_source": "nominal GB300 HBM3e bandwidth (8 TB/s), the target's denominator",
                       "algorithmic_bytes_per_launch": state_b + ring_b, "kernel": kernel,
                       "source_hash": src_hash}
    out["clocks"] = clock_info

    if not args.no_extras:
        # latency with an empty active list: a CUDA graph of 1000 launches
        kw = dw.call_kwargs()
        empty = torch.full_like(dw.active, -1)
        kw["active_request_indices"] = empty
        empty_call = rsm.prepare(**kw)
        t_empty = time_graph(torch, [empty_call] * 1000)
        # host cost of one call (argument marshalling done once)
        t0 = time.perf_counter()
        for _ in range(1000):
            empty_call(stream)
        host_us = (time.perf_counter() - t0) / 1000 * 1e6
        torch.cuda.synchronize()
        # T(n) for small n, rotating over requests so no launch re-reads what the previous one read
        sweep = {}
        rng = np.random.default_rng(9)
        for nn in (1, 16):
            if nn > shape.Bt:
                continue
            calls, keep = [], []
            for r in range(max(64 // nn, 8)):
                a = np.full(shape.Bt, -1, np.int32)
                a[:nn] = rng.permutation(shape.Bt)[:nn]
                t = torch.from_numpy(a).to(device)
                keep.append(t)
                kw2 = dw.call_kwargs()
                kw2["active_request_indices"] = t
                calls.append(rsm.prepare(**kw2))
            sweep[nn] = time_graph(torch, calls, reps=2)
        sweep[n] = ms
        out["empty_us"] = t_empty * 1e3
        out["host_call_us"] = host_us
        out["ms_per_call"] = {str(k): v for k, v in sorted(sweep.items())}
        out["us_per_request"] = {str(k): (v - t_empty) * 1e3 / k for k, v in sorted(sweep.items()) if k > 0}
        out["us_per_request_total"] = {str(k): v * 1e3 / k for k, v in sorted(sweep.items()) if k > 0}
        if rank == 0:
            try:
                out["e2e"] = e2e_measure(torch, rsm, shape, min(args.e2e_requests, shape.Bt), args.e2e_steps,
                                         device)
                if out["e2e"]["h2d_bytes_per_step"] < state_b:
                    out["e2e"]["note"] = (
                        f"measured on {min(args.e2e_requests, shape.Bt)} of the {n} requests: the whole step's "
                        f"{state_b / 2e9:.0f} GB of source state (and as much of results) would not fit in pinned "
                        f"host memory, and the figure is bound by the CPU-GPU link, not by the request count")
            except RuntimeError as ex:  # pinned memory exhausted etc.
                out["e2e"] = {"value": None, "error": str(ex)[:200]}
            if world == 1:
                out["cpu_baseline"] = cpu_baseline_from_device(dw, shape, args.cpu_seconds)
    if args.all_workloads or not (args.no_extras or args.no_workloads):
        del dw, call
        torch.cuda.empty_cache()
        only = set(args.only.split(",")) if args.only else None
        out["workloads"] = measure_named_workloads(torch, rsm, device, peak, sms, uuid, only)
        out["lane_peaks_note"] = (f"fp32: {sms} SMs x {ALU_LANES_PER_SM} lanes x the sampled SM clock; 32-bit "
                                  f"integer: {sms} SMs x {INT_LANES_PER_SM} lanes x the sampled SM clock; Philox: "
                                  f"{PHILOX10_WORDS_PER_SM_CLK} words per SM per clock at 10 rounds (measured); a word "
                                  f"rounds two 16-bit or four one-byte elements; tensor: the measured dense bf16 "
                                  f"GEMM rate (MEASURED_PEAKS.json bf16_tflops), x {TF32_PER_BF16:.3f} (the nominal "
                                  f"TF32 : BF16 ratio) for TF32")
    if rank == 0:
        print(json.dumps(out), flush=True)
    dist.barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
