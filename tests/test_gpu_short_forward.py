"""The short-query forwards against the oracle and against the query-tile forward:
- GDPA: scores formed transposed (keys on the TMEM lanes), O^T summed in TMEM over all key
  tiles of a (sequence, head) item;
- softmax at head_dim 64 with query sets of at most 64 rows: two key tiles per score tile (one
  per half of the TMEM lanes), an online softmax per lane with deferred rescaling, and the
  two halves' partial results merged per query row.

The planner takes these forms for plans whose query sets all fit one tile, with no causal
mask, window or shared key/value, and jfa_fwd runs them when the call has no bias.  The cases
are those of the short-query backward: each tile configuration, query sets of 0, 1 and
tile-boundary lengths, key lengths of 0, 1 and tile boundaries +-1, a last sequence that ends
at the end of the buffers, and sequences without keys, whose O rows must be exact zeros."""
import numpy as np
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

import parity
from test_gpu_short_backward import CASES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jfa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    return m


def _batch(case, mode, seed):
    q, kv, D, _ = CASES[case]
    return wl.make_custom(q, kv, H=3, D=D, mode=mode, causal=False, bias=False, value_std=0.5,
                          device="cuda", seed=seed)


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["gelu_tanh", "silu"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_short_forward_matches_oracle(jfa, case, mode, out):
    b = _batch(case, mode, 700 + case)
    plan = jfa.plan_for(b)
    assert jfa.jfa_plan_info(plan)["fwd_short"] == CASES[case][3]
    O, _ = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale,
                       out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    ref = parity.run_oracle(b, with_backward=False)
    m = parity.compare({"O": O}, ref, softmax=False, with_backward=False)
    print(CASES[case][:3], mode, out, m)
    parity.assert_within(m, softmax=False)
    for s in range(b.B):  # sequences without keys: O rows exactly zero
        q0, q1 = int(b.q_off[s]), int(b.q_off[s + 1])
        if b.kv_off[s + 1] == b.kv_off[s] and q1 > q0:
            assert torch.all(O[q0:q1] == 0)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_short_forward_agrees_with_the_query_tile_forward(jfa, case):
    # a relative-position bias of zeros runs the query-tile forward on the same arithmetic
    b = _batch(case, "gelu_tanh", 710 + case)
    plan = jfa.plan_for(b)
    O1, _ = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    zero_bias = torch.zeros(b.H, 32, dtype=torch.float32, device="cuda")
    jfa.jfa_plan_set_timing(plan, True)
    O2, _ = jfa.jfa_fwd(plan, b.Q, b.K, b.V, zero_bias, b.scale, out_dtype=torch.float32)
    O3, _ = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    assert torch.equal(O1, O3)  # no atomics: the same bits on every run
    err = parity.rel_frob(parity.np64(O1), parity.np64(O2))
    assert err <= 1e-5, err


def test_which_plans_take_a_short_query_forward(jfa):
    q, kv = [0, 40, 104], [0, 300, 429]  # offsets: query sets of 40 and 64 rows
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 128, "gelu_tanh", False))["fwd_short"] == 128
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 64, "silu", False))["fwd_short"] == 64
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 64, "softmax", False))["fwd_short"] == 64
    # softmax keeps the query-tile forward at head_dim 128 or with query sets over 64 rows
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 128, "softmax", False))["fwd_short"] == 0
    assert jfa.jfa_plan_info(jfa.jfa_plan_create([0, 65], [0, 300], 2, 64, "softmax", False))["fwd_short"] == 0
    assert jfa.jfa_plan_info(jfa.jfa_plan_create([0, 129], [0, 300], 2, 64, "silu", False))["fwd_short"] == 0
    assert jfa.jfa_plan_info(jfa.jfa_plan_create(q, kv, 2, 64, "silu", True))["fwd_short"] == 0


def test_full_size_gdpa_workload_sampled(jfa):
    """The gdpa_gelu workload as the benchmark launches it (bf16 O), every sequence's O
    checked on sampled rows against the oracle, and the whole output finite."""
    batch = wl.make("gdpa_gelu", device="cuda")
    plan = jfa.plan_for(batch)
    assert jfa.jfa_plan_info(plan)["fwd_short"] == 128
    O, _ = jfa.jfa_fwd(plan, batch.Q, batch.K, batch.V, None, batch.scale, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    assert torch.isfinite(O).all()
    rng = np.random.default_rng(3)
    seqs = sorted(set(rng.choice(batch.B, size=12, replace=False).tolist() +
                      [int(np.argmax(batch.kv_lens)), int(np.argmax(batch.q_lens))]))
    sub = wl.subset(batch, seqs)
    ref = parity.run_oracle(sub, with_backward=False)
    rows = np.concatenate([np.arange(batch.q_off[s], batch.q_off[s + 1]) for s in seqs])
    m = parity.compare({"O": O[torch.as_tensor(rows, device="cuda")]}, ref, softmax=False, with_backward=False)
    print(seqs, m)
    parity.assert_within(m, softmax=False)


# ----------------------------------------------------------------------------- softmax, packed


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_packed_softmax_forward_matches_oracle(jfa, out):
    q, kv, D, bq = CASES[0]
    assert D == 64 and bq == 64
    b = wl.make_custom(q, kv, H=3, D=64, mode="softmax", causal=False, bias=False, device="cuda", seed=720)
    plan = jfa.plan_for(b)
    assert jfa.jfa_plan_info(plan)["fwd_short"] == 64
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale,
                         out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    m = parity.compare({"O": O, "lse": lse}, parity.run_oracle(b, with_backward=False), with_backward=False)
    print(out, m)
    parity.assert_within(m)
    for s in range(b.B):  # sequences without keys: O = 0 and lse = -inf
        q0, q1 = int(b.q_off[s]), int(b.q_off[s + 1])
        if b.kv_off[s + 1] == b.kv_off[s] and q1 > q0:
            assert torch.all(O[q0:q1] == 0) and torch.all(torch.isneginf(lse[q0:q1]))


@pytest.mark.parametrize("growth", ["rising", "falling"])
def test_packed_softmax_rescales_when_the_row_max_grows(jfa, growth):
    """Scores that rise along the keys make each row's maximum grow past the 2^8 margin
    many times (every such step rescales O); falling scores never rescale."""
    b = wl.make_custom([40, 64, 7], [2000, 1500, 129], H=2, D=64, mode="softmax", causal=False, bias=False,
                       device="cuda", seed=721)
    for s in range(b.B):
        k0, k1 = int(b.kv_off[s]), int(b.kv_off[s + 1])
        ramp = torch.linspace(0.2, 6.0, k1 - k0, device="cuda")
        if growth == "falling":
            ramp = ramp.flip(0)
        b.K[k0:k1] = (b.K[k0:k1].float() * ramp[:, None, None]).to(b.K.dtype)
    plan = jfa.plan_for(b)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    m = parity.compare({"O": O, "lse": lse}, parity.run_oracle(b, with_backward=False), with_backward=False)
    print(growth, m)
    parity.assert_within(m)


def test_packed_softmax_agrees_with_the_query_tile_forward(jfa):
    # a relative-position bias of zeros runs the query-tile forward on the same arithmetic
    q, kv, _, _ = CASES[0]
    b = wl.make_custom(q, kv, H=3, D=64, mode="softmax", causal=False, bias=False, device="cuda", seed=722)
    plan = jfa.plan_for(b)
    O1, l1 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    O3, l3 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    zero_bias = torch.zeros(b.H, 32, dtype=torch.float32, device="cuda")
    O2, l2 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, zero_bias, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(O1, O3) and torch.equal(l1, l3)
    # P is rounded to bf16 against each kernel's own reference maximum (this kernel's deferred
    # one, the query-tile kernel's upper bound), so O agrees to about P's rounding
    assert parity.rel_frob(parity.np64(O1), parity.np64(O2)) <= 2e-3
    fin = torch.isfinite(l2)
    assert torch.equal(fin, torch.isfinite(l1))
    assert float((l1[fin] - l2[fin]).abs().max()) <= 1e-4


def test_softmax_scale_must_be_positive(jfa):
    b = wl.make_custom([40], [300], H=2, D=64, mode="softmax", causal=False, bias=False, device="cuda", seed=723)
    plan = jfa.plan_for(b)
    for bad in (0.0, -0.125, float("inf"), float("nan")):
        with pytest.raises(jfa.JFAError) as e:
            jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, bad)
        assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    # GDPA takes any finite scale: no row maximum is formed
    g = wl.make_custom([40], [300], H=2, D=64, mode="silu", causal=False, bias=False, value_std=0.5,
                       device="cuda", seed=724)
    gp = jfa.plan_for(g)
    O, _ = jfa.jfa_fwd(gp, g.Q, g.K, g.V, None, -g.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = parity.run_oracle(__import__("dataclasses").replace(g, scale=-g.scale), with_backward=False)
    parity.assert_within(parity.compare({"O": O}, ref, softmax=False, with_backward=False), softmax=False)

