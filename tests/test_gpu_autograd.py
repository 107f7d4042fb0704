"""The torch.autograd form of the library (jfa.jagged_attention), on the GPU.

It marshals arguments only, so its output and gradients must be bitwise those of the direct
calls (jfa_fwd, then jfa_bwd or jfa_bwd_ex with the same upstream gradient); once more they are
compared with the CPU oracle within the usual tolerances.  Bitwise comparisons of gradients run
the deterministic two-pass backward (jfa_plan_set_deterministic): the fused one adds dQ in an
order that varies between runs."""
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()


def leaf(t):
    return t.detach().clone().requires_grad_(True)


@pytest.mark.parametrize("mode,causal,bias", [("softmax", True, True), ("gelu_tanh", False, True),
                                              ("silu", True, False)])
def test_autograd_matches_the_direct_calls_and_the_oracle(mode, causal, bias):
    from jagged_sequence_attention_gb300 import jfa
    q = [1, 127, 129, 300, 64]
    kv = [5, 200, 129, 300, 700]
    std = 1.0 if mode == "softmax" else 0.5
    b = wl.make_custom(q, kv, H=2, D=128, mode=mode, causal=causal, bias=bias, value_std=std, device="cuda",
                       seed=31)
    Q, K, V = leaf(b.Q), leaf(b.K), leaf(b.V)
    tb = leaf(b.bias) if bias else None
    O = jfa.jagged_attention(Q, K, V, b.q_off, b.kv_off, bias=tb, mode=mode, causal=causal, scale=b.scale,
                             deterministic=True)
    O.backward(b.dO)
    torch.cuda.synchronize()

    direct = jfa.attention(b, with_backward=True, out_dtype=b.Q.dtype, bias_grad=bias, deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(O.detach(), direct["O"])
    for got, key in ((Q.grad, "dQ"), (K.grad, "dK"), (V.grad, "dV")):
        assert torch.equal(got, direct[key]), key
    if bias:
        assert torch.equal(tb.grad, direct["dbias"])

    r = parity.run_oracle(b, True, bias_grads=bias)
    O64 = parity.np64(O.detach())  # bf16, as Q: the error beyond its own rounding
    assert parity.beyond_rounding(O64, r["O"]) <= parity.FWD_MAX_ABS
    assert parity.rel_frob(O64, r["O"]) <= parity.FWD_REL_FROB
    for got, key in ((Q.grad, "dQ"), (K.grad, "dK"), (V.grad, "dV")):
        assert parity.rel_frob(parity.np64(got), r[key]) <= parity.BWD_REL_FROB, key
    if bias:
        assert parity.rel_frob(parity.np64(tb.grad), r["dbias"]) <= parity.BWD_REL_FROB


def test_autograd_without_bias_gradient_and_with_a_reused_plan():
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom([40, 260], [300, 260], H=2, D=64, causal=True, bias=True, device="cuda", seed=32)
    plan = jfa.plan_for(b, deterministic=True)
    Q, K, V = leaf(b.Q), leaf(b.K), leaf(b.V)
    grads = []
    for _ in range(2):  # the same plan serves both steps
        for t in (Q, K, V):
            t.grad = None
        O = jfa.jagged_attention(Q, K, V, bias=b.bias, plan=plan, scale=b.scale)  # the table needs no grad
        O.backward(b.dO)
        grads.append([t.grad.clone() for t in (Q, K, V)])
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == 0
    for x, y in zip(*grads):
        assert torch.equal(x, y)


def test_autograd_dense_bias_gradient():
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom([33, 128, 5], [70, 128, 300], H=2, D=64, dense_bias=True, device="cuda", seed=33)
    Q, K, V, dense = leaf(b.Q), leaf(b.K), leaf(b.V), leaf(b.dense)
    O = jfa.jagged_attention(Q, K, V, b.q_off, b.kv_off, bias=dense, dense_bias=True, scale=b.scale)
    O.backward(b.dO)
    torch.cuda.synchronize()
    direct = jfa.attention(b, with_backward=True, out_dtype=b.Q.dtype, bias_grad=True)
    torch.cuda.synchronize()
    assert torch.equal(O.detach(), direct["O"])
    assert torch.equal(dense.grad, direct["dbias"])


def test_autograd_shared_key_value():
    # query sets 0..4 over two users; dK and dV sum over each user's query sets
    from jagged_sequence_attention_gb300 import jfa
    users = [300, 129]
    kv_map = [0, 1, 0, 0, 1]
    q = [40, 7, 128, 1, 64]
    b = wl.make_shared_kv(q, users, kv_map, H=2, D=128, bias=True, seed=34, device="cuda")
    Q, K, V = leaf(b.Q), leaf(b.K), leaf(b.V)
    O = jfa.jagged_attention(Q, K, V, b.q_off, b.kv_off, bias=b.bias, scale=b.scale, kv_index=b.kv_map)
    O.backward(b.dO)
    torch.cuda.synchronize()
    direct = jfa.attention(b, with_backward=True, out_dtype=b.Q.dtype)
    torch.cuda.synchronize()
    assert torch.equal(O.detach(), direct["O"])
    for got, key in ((Q.grad, "dQ"), (K.grad, "dK"), (V.grad, "dV")):
        assert torch.equal(got, direct[key]), key
