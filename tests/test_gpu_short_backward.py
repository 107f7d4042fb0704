"""The short-query bf16 backward (one kernel over (sequence, head) items: the query set's
Q and dO stay in shared memory, the key tiles stream past, dQ accumulates in TMEM and is
written once) against the oracle, the two-pass backward and itself.

The planner takes this form when every query set fits one tile (64 rows at head_dim 64,
where two CTAs share an SM; else 128 rows), with no causal mask, no window and no shared
key/value, and jfa_bwd runs it when the call has no bias.  The cases cover each tile
configuration in both modes, query sets of 0, 1 and tile-boundary lengths, key lengths
of 0, 1 and tile boundaries +-1, a batch whose last sequence ends at the end of the
buffers, and sequences without queries (their dK/dV rows must be zeros) or without keys
(their dQ rows must be zeros)."""
import dataclasses

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


CASES = [
    # (q lengths, kv lengths, D, expected query-tile rows)
    ([1, 31, 32, 33, 63, 64, 0, 17, 5], [1, 127, 128, 129, 1000, 300, 200, 0, 256], 64, 64),
    ([65, 128, 1, 100, 0, 127], [129, 40, 513, 0, 77, 128], 64, 128),
    ([128, 1, 64, 0, 90, 127, 33], [256, 700, 1, 129, 0, 383, 128], 128, 128),
]


def _batch(case, mode, seed):
    q, kv, D, _ = CASES[case]
    return wl.make_custom(q, kv, H=3, D=D, mode=mode, causal=False, bias=False,
                          value_std=1.0 if mode == "softmax" else 0.5, device="cuda", seed=seed)


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_short_backward_matches_oracle(jfa, case, mode):
    b = _batch(case, mode, 600 + case)
    g = parity.run_gpu(b)
    assert g["status"] == 0
    info = jfa.jfa_plan_info(g["plan"])
    assert info["bwd_short"] == CASES[case][3]
    m = parity.compare(g, parity.run_oracle(b), softmax=mode == "softmax")
    print(CASES[case][:3], mode, m)
    parity.assert_within(m, softmax=mode == "softmax")
    Tq = int(b.q_off[-1])
    # sequences without keys: dQ rows exactly zero; without queries: dK and dV rows zero
    for s in range(b.B):
        q0, q1 = int(b.q_off[s]), int(b.q_off[s + 1])
        k0, k1 = int(b.kv_off[s]), int(b.kv_off[s + 1])
        if k1 == k0 and q1 > q0:
            assert torch.all(g["dQ"][q0:q1] == 0)
        if q1 == q0 and k1 > k0:
            assert torch.all(g["dK"][k0:k1] == 0) and torch.all(g["dV"][k0:k1] == 0)
    assert Tq == sum(CASES[case][0])


@pytest.mark.parametrize("case", range(len(CASES)))
def test_short_backward_repeats_bit_for_bit_and_agrees_with_two_pass(jfa, case):
    b = _batch(case, "softmax", 610 + case)
    plan = jfa.plan_for(b)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    g1 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, None, b.scale)
    g2 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, None, b.scale)
    two = jfa.plan_for(b, deterministic=True)
    assert jfa.jfa_plan_info(two)["bwd_short"] == 0
    g3 = jfa.jfa_bwd(two, b.Q, b.K, b.V, O, b.dO, lse, None, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK and jfa.jfa_plan_device_status(two) == jfa.JFA_OK
    for name, x, y, z in zip(("dQ", "dK", "dV"), g1, g2, g3):
        assert torch.equal(x, y), name  # no atomics: the same bits on every run
        # the same products from the same bf16 operands, summed in another order
        err = parity.rel_frob(parity.np64(x), parity.np64(z))
        assert err <= 2e-3, (name, err)


def test_planner_takes_the_form_only_where_it_applies(jfa):
    q, kv = [0, 40, 104], [0, 300, 429]  # offsets: query sets of 40 and 64 rows
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 64, "softmax", False))["bwd_short"] == 64
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 128, "softmax", False))["bwd_short"] == 128
    assert jfa.jfa_plan_info(jfa.jfa_plan_create([0, 65], [0, 300], 2, 64, "softmax", False))["bwd_short"] == 128
    # a query set longer than one tile, a causal mask, or head_dim 32: not this form
    assert jfa.jfa_plan_info(jfa.jfa_plan_create([0, 129], [0, 300], 2, 64, "softmax", False))["bwd_short"] == 0
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 64, "softmax", True))["bwd_short"] == 0
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 32, "softmax", False))["bwd_short"] == 0
    p = jfa.jfa_plan_create(q, kv, 2, 64, "softmax", False)
    jfa.jfa_plan_set_deterministic(p, True)  # forces the two-pass form
    assert jfa.jfa_plan_info(p)["bwd_short"] == 0


def test_one_kernel_per_backward_and_bias_calls_take_another_form(jfa):
    b = wl.make_custom([40, 64, 7], [300, 129, 1000], H=2, D=64, causal=False, bias=True, device="cuda",
                       seed=620)
    p = jfa.plan_for(b)
    jfa.jfa_plan_set_timing(p, True)
    for bias in (None, b.bias):
        O, lse = jfa.jfa_fwd(p, b.Q, b.K, b.V, bias, b.scale)
        g = jfa.jfa_bwd(p, b.Q, b.K, b.V, O, b.dO, lse, bias, b.scale)
        t = {k: v[1] for k, v in jfa.jfa_plan_kernel_times(p).items()}
        if bias is None:  # the short-query kernel alone (after the row terms)
            assert t == {"fwd": 1, "bwd_pre": 1, "bwd_main": 1, "bwd_post": 0, "bwd_dq": 0}
        else:  # the relative-position bias runs the fused form
            assert t == {"fwd": 1, "bwd_pre": 1, "bwd_main": 1, "bwd_post": 1, "bwd_dq": 0}
        torch.cuda.synchronize()
        assert jfa.jfa_plan_device_status(p) == jfa.JFA_OK
        ref = parity.run_oracle(b if bias is not None else dataclasses.replace(b, bias=None))
        m = parity.compare({"O": O, "lse": lse, "dQ": g[0], "dK": g[1], "dV": g[2]}, ref)
        parity.assert_within(m)
