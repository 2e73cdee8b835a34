"""The torch.library custom op (torch.ops.replayssm.materialize): its schema
declares the dependency outputs mutated, its fake implementation traces on
meta tensors (no GPU), and on a GPU a torch.compile'd call writes what the
eager call writes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_replayssm_state_gb300.torch_op as top  # noqa: E402


def _meta_args(L=2, B=4):
    m = lambda *s, dt=torch.int64: torch.zeros(*s, dtype=dt, device="meta")
    return ([m(L) for _ in range(11)] +
            [m(L, B, dt=torch.int32), m(L, B, dt=torch.int32), m(B, dt=torch.int32), m(B, dt=torch.int32),
             m(B, dt=torch.int32)])


KW = dict(state_dtype="bf16", input_dtype="bf16", matrixA_dtype="f32", dim=64, dstate=128, num_heads=4,
          heads_per_group=2, max_window=8, ring_buffer_len=8)


def test_schema_marks_dependency_outputs_mutated():
    schema = top.OP.default._schema
    mutated = [a.name for a in schema.arguments if a.alias_info is not None and a.alias_info.is_write]
    assert mutated == ["dependency_outputs"]
    assert len(schema.returns) == 0


def test_fake_implementation_on_meta_tensors():
    st = torch.zeros(3, 5, device="meta")
    top.materialize(*_meta_args(), dependency_inputs=[st], dependency_outputs=[st], **KW)


def test_traces_under_torch_compile_without_graph_breaks():
    def f(st, *a):
        top.materialize(*a, dependency_inputs=[st], dependency_outputs=[st], **KW)
        return st + 1

    st = torch.zeros(3, 5, device="meta")
    out = torch.compile(f, backend="aot_eager", fullgraph=True)(st, *_meta_args())
    assert out.shape == (3, 5)


# ----------------------------------------------------------------------------
# GPU: compiled against eager, and against the oracle
# ----------------------------------------------------------------------------

def _world():
    from mamba_replayssm_state_gb300 import workloads as wl
    shape = wl.Shape("op", L=2, Bt=5, H=6, hpg=3, D=64, N=128, R=8, W=8, state_dtype="bf16", n_active=4)
    return wl, wl.host_world(shape, seed=17)


def _compiled_call(dw, backend):
    kw = dw.call_kwargs()
    kw.pop("device_status")
    inputs = [t for t in dw.x + dw.B + dw.dt + dw.A if t is not None]
    outputs = list(dw.state)

    def step(*states):
        top.materialize(**kw, dependency_inputs=inputs, dependency_outputs=list(states))
        return [s.clone() for s in states]

    return torch.compile(step, backend=backend, fullgraph=True)(*outputs)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("backend", ["eager", "inductor"])
def test_compiled_call_matches_oracle(backend):
    if backend == "inductor":
        pytest.importorskip("triton")
    import oracle
    from parity import compare_worlds
    wl, hw = _world()
    dw = wl.device_world_from_host(hw)
    got_states = _compiled_call(dw, backend)
    torch.cuda.synchronize()
    got = hw.copy()
    got.state = [wl._to_np(t).view(a.dtype) for t, a in zip(got_states, hw.state)]
    ref = hw.copy()
    oracle.materialize(ref)
    assert compare_worlds(got, ref, hw) >= 4
    # the state tensors themselves hold the result too
    for t, g in zip(dw.state, got.state):
        assert np.array_equal(wl._to_np(t).view(g.dtype), g)
