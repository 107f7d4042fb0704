"""Gradient of the relative-position bias table on the GPU (through the C-ABI,
jfa_bwd_ex) against the CPU oracle, which sums dS by bucket over every allowed pair.

Cases:
- causal and non-causal;
- q_len != kv_len, including rows with no key;
- a sliding window;
- both GDPA activations;
- the fp32 CUDA-core path and both tensor-core head dims;
- a long pair of sequences whose far buckets come from many steps of warp-constant
  chunks.

Also checked:
- the result is bitwise the same on a second run;
- dQ, dK and dV are bitwise those of jfa_bwd;
- argument errors.

Softmax's exact table gradient sums to zero per head (each row's dS does). That is
pinned on the oracle. On the GPU the sum is not zero but a small residual: the forward
forms O from bf16-rounded P, so Delta = rowsum(dO * O) differs from sum_j p_ij dp_ij
by that rounding."""
import numpy as np
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

import parity

pytestmark = pytest.mark.gpu

DBIAS_REL_FROB = parity.BWD_REL_FROB


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()


def check(batch, out_dtype=torch.float32):
    from jagged_sequence_attention_gb300 import jfa
    out = jfa.attention(batch, with_backward=True, out_dtype=out_dtype, bias_grad=True)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(out["plan"]) == 0
    r = parity.run_oracle(batch, True, bias_grads=True)
    m = parity.compare(out, r, softmax=batch.mode == "softmax", with_backward=True)
    m["dbias_rel_frob"] = parity.rel_frob(parity.np64(out["dbias"]), r["dbias"])
    print(batch.name, m)
    parity.assert_within(m, softmax=batch.mode == "softmax")
    assert m["dbias_rel_frob"] <= DBIAS_REL_FROB, m
    return out, r


LENS = [1, 37, 127, 128, 129, 255, 256, 257, 700, 1100]


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
def test_causal_self_attention(mode):
    check(wl.make_custom(LENS, LENS, H=2, D=128, mode=mode, causal=True, bias=True, value_std=0.5 if mode != "softmax"
                         else 1.0, device="cuda", seed=31))


@pytest.mark.parametrize("causal", [False, True])
def test_asymmetric_lengths(causal):
    # q > kv leaves causal rows with no key; non-causal relative positions take both signs
    q, kv = [200, 64, 900, 5, 300, 1], [500, 64, 700, 1, 129, 40]
    check(wl.make_custom(q, kv, H=3, D=128, causal=causal, bias=True, device="cuda", seed=32))


def test_window():
    check(wl.make_custom(LENS, LENS, H=2, D=128, causal=True, bias=True, device="cuda", seed=33, window=300))


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 32), (torch.float32, 64)])
def test_other_head_dims_and_fp32(dtype, D):
    check(wl.make_custom([7, 130, 64, 300], [7, 130, 90, 300], H=2, D=D, dtype=dtype, causal=True, bias=True,
                         device="cuda", seed=34))


def test_fp32_non_causal():
    check(wl.make_custom([7, 130, 64], [40, 130, 9], H=2, D=32, dtype=torch.float32, causal=False, bias=True,
                         device="cuda", seed=35))


def test_bf16_output():
    check(wl.make_custom(LENS, LENS, H=2, D=128, causal=True, bias=True, device="cuda", seed=36),
          out_dtype=torch.bfloat16)


def test_long_sequences_far_buckets():
    # 6k tokens: relative positions up to 6k (bucket 25), most chunks warp-constant
    check(wl.make_custom([6000, 2500], [6000, 2500], H=2, D=128, causal=True, bias=True, device="cuda", seed=37))


def test_deterministic_and_same_gradients_as_jfa_bwd():
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom(LENS, LENS, H=2, D=128, causal=True, bias=True, device="cuda", seed=38)
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, b.mode, b.causal)
    jfa.jfa_plan_set_deterministic(plan, True)  # jfa_bwd then runs the two-pass form, as jfa_bwd_ex does
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale)
    g1 = jfa.jfa_bwd_ex(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    g2 = jfa.jfa_bwd_ex(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    g0 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == 0
    assert torch.equal(g1[3], g2[3])
    for x, y in zip(g0, g1[:3]):
        assert torch.equal(x, y)


def test_argument_errors():
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom([10, 20], [10, 20], H=2, D=128, causal=True, bias=True, device="cuda", seed=39)
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, b.mode, b.causal)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale)
    with pytest.raises(jfa.JFAError) as e:   # a gradient needs the table
        jfa.jfa_bwd_ex(plan, b.Q, b.K, b.V, O, b.dO, lse, None, b.scale)
    assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    small = torch.empty(jfa.jfa_bwd_workspace_size(plan, b.Q.dtype), dtype=torch.uint8, device="cuda")
    assert jfa.jfa_bwd_ex_workspace_size(plan, b.Q.dtype) > small.numel()
    with pytest.raises(jfa.JFAError) as e:
        jfa.jfa_bwd_ex(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale, workspace=small)
    assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    assert jfa.jfa_bwd_ex_workspace_size(plan, b.Q.dtype, bias_grad=False) == \
        jfa.jfa_bwd_workspace_size(plan, b.Q.dtype)
