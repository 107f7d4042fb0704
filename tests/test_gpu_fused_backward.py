"""The fused bf16 backward (one kernel over key tiles forms dK, dV and each key tile's
part of dQ, added into an fp32 accumulator at L2) against the two-pass backward (dQ by a
second pass over query tiles, no atomics), its run-to-run behaviour, and the planner's
choice between them (fused while key tiles visit few query tiles on average).

Both compute the same gradients from the same bf16 operands; they differ only in the
order in which dQ's fp32 sums are formed.  So dK and dV agree to fp32 rounding, dQ to
about one bf16 rounding step, and the fused dQ is the same between runs except in
the last bit.  Parity with the oracle is tested everywhere else: every bf16 test of
jfa_bwd runs the fused backward by default."""
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jfa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    return m


def _bwd(jfa, b, deterministic):
    plan = jfa.plan_for(b, deterministic=deterministic)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    g = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    return plan, g


CASES = [
    # (q lengths, kv lengths, H, D, mode, causal, bias, window)
    ([300, 1, 517, 128, 64, 200], None, 2, 128, "softmax", True, True, None),
    ([129, 40, 1000], [700, 40, 1000], 2, 128, "softmax", False, False, None),
    ([77, 256, 300], [500, 256, 129], 2, 64, "gelu_tanh", False, True, None),
    ([64, 2000], None, 2, 64, "silu", True, True, 300),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_agrees_with_two_pass(jfa, case):
    q, kv, H, D, mode, causal, bias, window = CASES[case]
    kv = q if kv is None else kv
    b = wl.make_custom(q, kv, H=H, D=D, mode=mode, causal=causal, bias=bias, window=window,
                       value_std=1.0 if mode == "softmax" else 0.5, device="cuda", seed=400 + case)
    pf, gf = _bwd(jfa, b, False)
    pd, gd = _bwd(jfa, b, True)
    assert jfa.jfa_plan_info(pf)["bwd_fused"] == 1 and jfa.jfa_plan_info(pd)["bwd_fused"] == 0
    assert jfa.jfa_bwd_workspace_size(pf) > jfa.jfa_bwd_workspace_size(pd)
    for name, x, y in zip(("dQ", "dK", "dV"), gf, gd):
        err = parity.rel_frob(parity.np64(x), parity.np64(y))
        assert err <= (2e-3 if name == "dQ" else 1e-5), (name, err)


def test_fused_repeats_except_the_last_bit_of_dq(jfa):
    b = wl.make_custom([300, 1, 517, 128, 64, 200], [300, 1, 517, 128, 64, 200], H=4, D=128, causal=True,
                       bias=True, device="cuda", seed=410)
    plan = jfa.plan_for(b)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    g1 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    g2 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    a, c = g1[0].float(), g2[0].float()
    assert bool(((a - c).abs() <= c.abs() * 2.0 ** -7 + 1e-6).all())


def test_deterministic_mode_repeats_bit_for_bit(jfa):
    b = wl.make_custom([300, 1, 517, 128, 64, 200], [300, 1, 517, 128, 64, 200], H=4, D=128, causal=True,
                       bias=True, device="cuda", seed=411)
    plan = jfa.plan_for(b, deterministic=True)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    g1 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    g2 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    for x, y in zip(g1, g2):
        assert torch.equal(x, y)


def test_planner_chooses_two_pass_for_long_sequences(jfa):
    # a 4096-token causal sequence: its key tiles visit 16.5 query tiles on average
    long_plan = jfa.jfa_plan_create([0, 4096], [0, 4096], 2, 128, "softmax", True)
    short_plan = jfa.jfa_plan_create([0, 300, 600], [0, 300, 600], 2, 128, "softmax", True)
    assert jfa.jfa_plan_info(long_plan)["bwd_fused"] == 0
    assert jfa.jfa_plan_info(short_plan)["bwd_fused"] == 1
    jfa.jfa_plan_set_deterministic(short_plan, True)
    assert jfa.jfa_plan_info(short_plan)["bwd_fused"] == 0
    # the workspace follows the form: row terms only once the fused form is off
    assert jfa.jfa_bwd_workspace_size(short_plan) == (600 * 2 * 4 + 255) // 256 * 256
    jfa.jfa_plan_set_deterministic(short_plan, False)
    assert jfa.jfa_bwd_workspace_size(short_plan) > 600 * 2 * 128 * 4
