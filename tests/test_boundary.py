"""The C-ABI library without a GPU: it loads, exports what include/replayssm.h
declares, and rejects bad host arguments before it touches CUDA."""
import ctypes
import os
import re

import pytest

import mamba_replayssm_state_gb300 as rsm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names += re.findall(r"RSM_API\s+[\w\s\*]+?\b(rsm_\w+)\s*\(", txt)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return rsm.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "rsm_materialize" in names and len(names) >= 5
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(rsm.EXPORTS)


def test_struct_layout_and_version(lib):
    assert lib.rsm_args_size() == ctypes.sizeof(rsm.RsmArgs)
    assert lib.rsm_abi_version() == 4


def test_oracle_library_loads():
    import oracle
    L = oracle.lib()
    assert L.oracle_args_size() == ctypes.sizeof(oracle.OracleArgs)


REQUIRED_TABLES = ("state_ptrs", "state_slot_strides", "x_cache_ptrs", "x_cache_slot_strides", "B_cache_ptrs",
                   "B_cache_slot_strides", "dt_cache_ptrs", "dt_cache_slot_strides", "A_ptrs", "src_slots",
                   "dst_slots", "ring_start", "replay_prefix_len", "active_request_indices")


def good_args():
    """The headline shape with fake device pointers: never dereferenced, since
    each test breaks one rule and validation stops before any CUDA call."""
    a = rsm.RsmArgs()
    for name in REQUIRED_TABLES:
        setattr(a, name, 0x1000)
    a.num_layers, a.batch = 48, 256
    a.state_dtype, a.input_dtype, a.matrixA_dtype = rsm.RSM_BF16, rsm.RSM_BF16, rsm.RSM_F32
    a.dim, a.dstate, a.num_heads, a.heads_per_group = 64, 128, 256, 32
    a.max_window, a.ring_buffer_len, a.pad_slot_id, a.philox_rounds = 8, 8, -1, 0
    return a


BAD_CASES = [
    ("null table", lambda a: setattr(a, "x_cache_ptrs", None), "x_cache_ptrs is NULL"),
    ("null active", lambda a: setattr(a, "active_request_indices", None), "active_request_indices"),
    ("layers", lambda a: setattr(a, "num_layers", 0), "num_layers"),
    ("batch", lambda a: setattr(a, "batch", -3), "batch"),
    ("heads zero", lambda a: setattr(a, "num_heads", 0), "num_heads"),
    ("heads > int32", lambda a: setattr(a, "num_heads", 2 ** 31), "num_heads"),
    ("group", lambda a: setattr(a, "heads_per_group", 33), "heads_per_group"),
    ("group zero", lambda a: setattr(a, "heads_per_group", 0), "heads_per_group"),
    ("window 0", lambda a: setattr(a, "max_window", 0), "max_window"),
    ("window 65", lambda a: setattr(a, "max_window", 65), "max_window"),
    ("ring", lambda a: setattr(a, "ring_buffer_len", 0), "ring_buffer_len"),
    ("input fp16", lambda a: setattr(a, "input_dtype", rsm.RSM_F16), "input_dtype"),
    ("A bf16", lambda a: setattr(a, "matrixA_dtype", rsm.RSM_BF16), "matrixA_dtype"),
    ("state dtype", lambda a: setattr(a, "state_dtype", 9), "state_dtype"),
    ("num_slots", lambda a: setattr(a, "num_slots", -1), "num_slots"),
    ("int8 shape", lambda a: (setattr(a, "state_dtype", rsm.RSM_I8), setattr(a, "dstate", 64)), "one-byte"),
    ("int8 scales", lambda a: setattr(a, "state_dtype", rsm.RSM_I8), "scale"),
    ("seed", lambda a: setattr(a, "philox_rounds", 10), "rand_seed"),
    ("rounds", lambda a: setattr(a, "philox_rounds", -1), "philox_rounds"),
]


@pytest.mark.parametrize("name,mutate,msg", BAD_CASES, ids=[c[0] for c in BAD_CASES])
def test_host_validation_rejects(lib, name, mutate, msg):
    a = good_args()
    mutate(a)
    rc = lib.rsm_materialize(ctypes.byref(a), None)
    assert rc == -1, (name, rc, lib.rsm_last_error())
    assert msg in lib.rsm_last_error().decode()
    rc = lib.rsm_launch_config(ctypes.byref(a), None, None, None, None)
    assert rc == -1


def test_unsupported_shape_is_enotsup(lib):
    a = good_args()
    a.dim, a.dstate = 32, 96
    assert lib.rsm_materialize(ctypes.byref(a), None) == -2
    assert "no kernel" in lib.rsm_last_error().decode()


def test_null_args(lib):
    assert lib.rsm_materialize(None, None) == -1


def test_python_binding_rejects_host_tensors():
    import torch
    t = torch.zeros(2, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        rsm._build_args(t, t, t, t, t, t, t, t, t, None, None, torch.zeros((2, 2), dtype=torch.int32),
                        torch.zeros((2, 2), dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                        torch.zeros(2, dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                        state_dtype=torch.bfloat16, input_dtype=torch.bfloat16, matrixA_dtype=torch.float32,
                        dim=64, dstate=128, num_heads=4, heads_per_group=2, max_window=8, ring_buffer_len=8)


def test_no_oracle_on_the_product_path():
    """The package never imports the oracle: no CPU fallback can hide behind it."""
    pkg = os.path.join(ROOT, "mamba_replayssm_state_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "replayssm_oracle" not in txt, f


# ----------------------------------------------------------------------------
# rsm_gdn_commit: host-side validation (no CUDA call is reached)
# ----------------------------------------------------------------------------

def good_gdn_args():
    a = rsm.GdnArgs()
    for name in ("checkpoint_state", "rawv_cache", "rawk_cache", "g_cache", "beta_cache", "state_indices",
                 "accept_lens"):
        setattr(a, name, 0x10000)
    a.layers, a.slots, a.num_v_heads, a.num_k_heads, a.window, a.batch = 36, 128, 32, 16, 8, 64
    a.use_qk_l2norm, a.null_block_id = 1, -1
    return a


def test_gdn_struct_layout(lib):
    assert lib.rsm_gdn_args_size() == ctypes.sizeof(rsm.GdnArgs)


@pytest.mark.parametrize("rule", ["null_state", "misaligned", "track_half", "heads", "window_lo", "window_hi",
                                  "null_id", "layers"])
def test_gdn_validation_rejects(lib, rule):
    a = good_gdn_args()
    if rule == "null_state":
        a.checkpoint_state = None
    elif rule == "misaligned":
        a.rawk_cache = 0x10008
    elif rule == "track_half":
        a.track_state_indices = 0x10000
    elif rule == "heads":
        a.num_k_heads = 5
    elif rule == "window_lo":
        a.window = 0
    elif rule == "window_hi":
        a.window = 65
    elif rule == "null_id":
        a.null_block_id = -2
    else:
        a.layers = 0
    assert lib.rsm_gdn_commit(ctypes.byref(a), None) == -1
    assert lib.rsm_last_error()


@pytest.mark.parametrize("rule", ["unknown", "no_l2norm", "tracking", "window_3", "window_9"])
def test_gdn_tcgen05_backend_preconditions(lib, rule):
    """The tcgen05 backend takes what the GDN page gives it (normalised K, no
    tracking, windows of 4 to 8 tokens) and refuses the rest on the host."""
    a = good_gdn_args()
    a.backend = rsm.GDN_BACKENDS["tcgen05"]
    if rule == "unknown":
        a.backend = 3
    elif rule == "no_l2norm":
        a.use_qk_l2norm = 0
    elif rule == "tracking":
        a.track_state_indices = a.track_steps = 0x10000
    elif rule == "window_3":
        a.window = 3
    else:
        a.window = 9
    assert lib.rsm_gdn_commit(ctypes.byref(a), None) == -1
    msg = lib.rsm_last_error()
    assert (b"backend" in msg) if rule == "unknown" else (b"tcgen05" in msg), msg


def test_gdn_empty_batch_enqueues_nothing(lib):
    a = good_gdn_args()
    a.batch = 0
    assert lib.rsm_gdn_commit(ctypes.byref(a), None) == 0


def test_kernel_name_follows_the_launch_rule(lib):
    """rsm_kernel_name needs no GPU: the CUDA-core kernel for the 8-token
    headline shape and fp32 state, the tensor-core kernel for 16-bit state with
    bf16 inputs at 64 x 128 once max_window reaches 16, for int8 and fp8 state
    the one-byte tensor-core kernel when the inputs are bf16 and a B group has
    an even number of heads and the one-byte kernel otherwise, and "" (with
    the reason) when the arguments fail validation."""
    a = good_args()
    assert lib.rsm_kernel_name(ctypes.byref(a)) == b"materialize_kernel"
    a.max_window = a.ring_buffer_len = 64
    for sd in (rsm.RSM_BF16, rsm.RSM_F16):
        a.state_dtype = sd
        assert lib.rsm_kernel_name(ctypes.byref(a)) == b"materialize_tc_kernel"
    a.state_dtype = rsm.RSM_F32
    assert lib.rsm_kernel_name(ctypes.byref(a)) == b"materialize_kernel"
    a.state_scale_ptrs = a.state_scale_slot_strides = 0x1000
    assert a.input_dtype == rsm.RSM_BF16 and a.heads_per_group % 2 == 0
    for sd in (rsm.RSM_I8, rsm.RSM_FP8_E4M3):
        a.state_dtype = sd
        assert lib.rsm_kernel_name(ctypes.byref(a)) == b"materialize_q8tc_kernel"
        a.input_dtype = rsm.RSM_F32
        assert lib.rsm_kernel_name(ctypes.byref(a)) == b"materialize_q8_kernel"
        a.input_dtype = rsm.RSM_BF16
        hpg = a.heads_per_group
        a.heads_per_group = 1
        assert lib.rsm_kernel_name(ctypes.byref(a)) == b"materialize_q8_kernel"
        a.heads_per_group = hpg
    a.heads_per_group = 33
    assert lib.rsm_kernel_name(ctypes.byref(a)) == b""
    assert b"heads_per_group" in lib.rsm_last_error()
