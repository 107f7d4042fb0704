"""jfa_bwd_static_scratch: the backward pass for callers that cannot allocate device
memory (for instance code that runs inside another runtime's memory pool and owns
no allocator of its own).  The call keeps its scratch in a fixed array of the library
instead of a caller-supplied workspace.  These tests call it through the C-ABI and
compare it with jfa_bwd:

- bf16 inputs: the two calls run the same launches.  With the deterministic two-pass
  backward (jfa_plan_set_deterministic) everything adds in a fixed order, so the
  gradients must be equal bit for bit.  The default fused backward adds dQ into an
  fp32 accumulator in the shared array with reduce-adds whose order varies, so there dK
  and dV must be equal bit for bit and dQ within one bf16 rounding step; a call that
  found the previous call's accumulator uncleared would be far off.  Calls on two
  different problems alternate, so anything a call left in the shared array would
  show in the next one.
- fp32 inputs: the array also holds the dQ accumulator, which every call must clear
  before adding into it; two successful calls in a row would double dQ otherwise.
  The fp32 dQ adds with atomics (order varies), so that case compares within 1e-6.
- A problem whose scratch exceeds the array is refused before anything runs.

The file name makes pytest collect it after every other test file."""
import ctypes

import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

from parity import np64, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jfa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    return m


def _static_call(jfa, plan, b, dtype, O, o_dtype, lse, dQ, dK, dV):
    """One jfa_bwd_static_scratch call through the C-ABI, into preallocated outputs."""
    L = jfa.lib()
    bk = jfa.JFA_BIAS_RELPOS32 if b.bias is not None else jfa.JFA_BIAS_NONE
    return L.jfa_bwd_static_scratch(plan.handle, dtype, jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V),
                                    jfa._ptr(O), o_dtype, jfa._ptr(b.dO), jfa._ptr(lse), bk,
                                    jfa._ptr(b.bias), ctypes.c_float(b.scale), jfa._ptr(dQ), jfa._ptr(dK),
                                    jfa._ptr(dV), jfa._stream())


def _problem(jfa, q, kv, mode, causal, bias, seed, dtype=torch.bfloat16, H=4, D=128, deterministic=False):
    b = wl.make_custom(q, kv, H=H, D=D, dtype=dtype, mode=mode, causal=causal, bias=bias,
                       value_std=1.0 if mode == "softmax" else 0.5, device="cuda", seed=seed)
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, mode, causal)
    jfa.jfa_plan_set_deterministic(plan, deterministic)
    assert jfa.jfa_bwd_workspace_size(plan, dtype) <= jfa.JFA_STATIC_SCRATCH_BYTES
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    ref = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    return b, plan, O, lse, ref


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("mode,causal,bias", [("softmax", True, True), ("softmax", False, False),
                                              ("gelu_tanh", False, True)])
def test_static_scratch_equal_to_jfa_bwd_across_alternating_problems(jfa, mode, causal, bias, deterministic):
    q1 = [300, 1, 517, 128, 64, 200]
    kv1 = q1 if causal else [257, 40, 700, 128, 1, 333]
    q2 = [129, 900, 33]
    kv2 = q2 if causal else [1000, 77, 256]
    probs = [_problem(jfa, q1, kv1, mode, causal, bias, 777, deterministic=deterministic),
             _problem(jfa, q2, kv2, mode, causal, bias, 778, deterministic=deterministic)]
    # Calls A, B, A, B in a row on one stream with nothing in between: every call finds
    # the other problem's terms in the shared array.
    outs = []
    for k in range(4):
        b, plan, O, lse, _ = probs[k % 2]
        got = tuple(torch.full_like(t, float("nan")) for t in (b.Q, b.K, b.V))
        assert _static_call(jfa, plan, b, jfa.JFA_BF16, O, jfa.JFA_F32, lse, *got) == jfa.JFA_OK
        outs.append(got)
    torch.cuda.synchronize()
    for k, got in enumerate(outs):
        b, plan, _, _, ref = probs[k % 2]
        assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            if deterministic or name != "dQ":
                assert torch.equal(g, r), (k, name, float((g.float() - r.float()).abs().max()))
            else:  # within one bf16 rounding step of the other call's dQ
                gf, rf = g.float(), r.float()
                assert bool(((gf - rf).abs() <= rf.abs() * 2.0 ** -7 + 1e-6).all()), (k, name)


@pytest.mark.parametrize("mode", ["softmax", "silu"])
def test_static_scratch_on_the_short_query_backward(jfa, mode):
    # query sets of one tile without a causal mask or a bias: the short-query kernel, which
    # keeps only row terms in the scratch and adds nothing, so every output is equal bit
    # for bit to jfa_bwd's, across calls on alternating problems
    probs = [_problem(jfa, [40, 1, 64, 0, 17], [300, 129, 1000, 77, 0], mode, False, False, 781, H=2, D=64),
             _problem(jfa, [128, 5, 90], [700, 1, 256], mode, False, False, 782, H=2, D=128)]
    assert jfa.jfa_plan_info(probs[0][1])["bwd_short"] == 64 and jfa.jfa_plan_info(probs[1][1])["bwd_short"] == 128
    outs = []
    for k in range(4):
        b, plan, O, lse, _ = probs[k % 2]
        got = tuple(torch.full_like(t, float("nan")) for t in (b.Q, b.K, b.V))
        assert _static_call(jfa, plan, b, jfa.JFA_BF16, O, jfa.JFA_F32, lse, *got) == jfa.JFA_OK
        outs.append(got)
    torch.cuda.synchronize()
    for k, got in enumerate(outs):
        b, plan, _, _, ref = probs[k % 2]
        assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(g, r), (k, name)


def test_static_scratch_fp32_consecutive_calls_clear_the_accumulator(jfa):
    # fp32 inputs keep the dQ accumulator in the shared array: a second call that did not
    # clear it would return about twice the first call's dQ.
    b, plan, O, lse, ref = _problem(jfa, [300, 1, 77, 128], [257, 40, 700, 128], "softmax", False, True, 91,
                                    dtype=torch.float32, H=2, D=64)
    outs = []
    for _ in range(2):
        got = tuple(torch.full_like(t, float("nan")) for t in (b.Q, b.K, b.V))
        assert _static_call(jfa, plan, b, jfa.JFA_F32, O, jfa.JFA_F32, lse, *got) == jfa.JFA_OK
        outs.append(got)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    for k, got in enumerate(outs):
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.isfinite(g).all(), (k, name)
            err = rel_frob(np64(g), np64(r))
            assert err <= 1e-6, (k, name, err)


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
