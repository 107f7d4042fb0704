"""jfa_bwd_static_scratch: the backward pass for callers that cannot allocate device
memory (for instance code that runs inside another runtime's memory pool and owns
no allocator of its own).  The call keeps its scratch in a fixed array of the library
instead of a caller-supplied workspace.  These tests check it through the C-ABI
against jfa_bwd, on two calls in a row: every call shares the array, so a second
call would show anything the first one left behind.  They also check that an
oversized problem is refused before anything runs.

The file name makes pytest collect it after every other test file."""
import ctypes

import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

from parity import BWD_REL_FROB, np64, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jfa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    return m


def _static_call(jfa, plan, b, O, lse, dQ, dK, dV):
    """One jfa_bwd_static_scratch call through the C-ABI, into preallocated outputs."""
    L = jfa.lib()
    bk = jfa.JFA_BIAS_RELPOS32 if b.bias is not None else jfa.JFA_BIAS_NONE
    return L.jfa_bwd_static_scratch(plan.handle, jfa.JFA_BF16, jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V),
                                    jfa._ptr(O), jfa.JFA_F32, jfa._ptr(b.dO), jfa._ptr(lse), bk,
                                    jfa._ptr(b.bias), ctypes.c_float(b.scale), jfa._ptr(dQ), jfa._ptr(dK),
                                    jfa._ptr(dV), jfa._stream())


@pytest.mark.parametrize("mode,causal,bias", [("softmax", True, True), ("softmax", False, False),
                                              ("gelu_tanh", False, True)])
def test_static_scratch_matches_jfa_bwd_on_consecutive_calls(jfa, mode, causal, bias):
    q = [300, 1, 517, 128, 64, 200]
    kv = q if causal else [257, 40, 700, 128, 1, 333]
    b = wl.make_custom(q, kv, H=4, D=128, dtype=torch.bfloat16, mode=mode, causal=causal, bias=bias,
                       value_std=1.0 if mode == "softmax" else 0.5, device="cuda", seed=777)
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, mode, causal)
    assert jfa.jfa_bwd_workspace_size(plan) <= jfa.JFA_STATIC_SCRATCH_BYTES
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    ref = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    outs = [tuple(torch.full_like(t, float("nan")) for t in (b.Q, b.K, b.V)) for _ in range(2)]
    for dQ, dK, dV in outs:  # two calls in a row, nothing in between
        assert _static_call(jfa, plan, b, O, lse, dQ, dK, dV) == jfa.JFA_OK
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    for call, got in enumerate(outs):
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.isfinite(g).all(), (call, name)
            err = rel_frob(np64(g), np64(r))
            assert err <= BWD_REL_FROB, (call, name, err)


def test_static_scratch_refuses_problems_beyond_its_size(jfa):
    # fp32 inputs keep an fp32 dQ accumulator in the scratch: T_q * H * D * 4 bytes of it
    # alone exceed the array by a little.
    D, H = 64, 1
    tq = jfa.JFA_STATIC_SCRATCH_BYTES // (4 * D * H) + 64
    b = wl.make_custom([tq], [tq], H=H, D=D, dtype=torch.float32, device="cuda", seed=5)
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, H, D, "softmax", False)
    assert jfa.jfa_bwd_workspace_size(plan, torch.float32) > jfa.JFA_STATIC_SCRATCH_BYTES
    O = torch.zeros(b.Q.shape, dtype=torch.float32, device="cuda")
    lse = torch.zeros((tq, H), dtype=torch.float32, device="cuda")
    dQ, dK, dV = (torch.zeros_like(t) for t in (b.Q, b.K, b.V))
    L = jfa.lib()
    st = L.jfa_bwd_static_scratch(plan.handle, jfa.JFA_F32, jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V),
                                  jfa._ptr(O), jfa.JFA_F32, jfa._ptr(b.dO), jfa._ptr(lse), jfa.JFA_BIAS_NONE,
                                  None, ctypes.c_float(b.scale), jfa._ptr(dQ), jfa._ptr(dK), jfa._ptr(dV),
                                  jfa._stream())
    assert st == jfa.JFA_ERR_SCRATCH_LIMIT
    assert "scratch" in jfa.jfa_status_string(jfa.JFA_ERR_SCRATCH_LIMIT)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dQ) == 0 and torch.count_nonzero(dK) == 0
