"""Parity of the CUDA path (through the C-ABI) against the CPU oracle.

Small cases are compared element by element over every output; the full-size
workloads run exactly as the benchmark launches them and are compared on sampled
outputs that the oracle computes exactly through suffix sub-problems (see
``parity.suffix_problem``).
"""
import math

import numpy as np
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


def check_full(batch, with_backward=True, out_dtype=torch.float32, form="planner"):
    """form: "planner" (the plan's own choice of bf16 backward) or "two_pass" (forced)."""
    g = parity.run_gpu(batch, with_backward, out_dtype=out_dtype, deterministic=form == "two_pass")
    assert g["status"] == 0, g["status"]
    if form == "two_pass":
        from jagged_sequence_attention_gb300 import jfa
        assert jfa.jfa_plan_info(g["plan"])["bwd_fused"] == 0
    r = parity.run_oracle(batch, with_backward)
    m = parity.compare(g, r, softmax=batch.mode == "softmax", with_backward=with_backward)
    print(batch.name, m)
    parity.assert_within(m, softmax=batch.mode == "softmax")
    return g, r


def test_tiny_workload_full():
    check_full(wl.make("tiny", device="cuda"))


def pick_sequences(batch, k_random=4, seed=0):
    lens = batch.q_lens * batch.kv_lens + batch.q_lens
    order = np.argsort(lens)
    rng = np.random.default_rng(seed)
    mid = rng.choice(order[2:-2], size=min(k_random, max(0, len(order) - 4)), replace=False)
    return sorted(set(order[:2].tolist() + order[-2:].tolist() + mid.tolist()))


@pytest.mark.parametrize("name", ["causal_bias", "cross", "gdpa_gelu", "gdpa_silu"])
@pytest.mark.parametrize("out,form", [("f32", "planner"), ("bf16", "planner"), ("f32", "two_pass")])
def test_workload_slice_full(name, out, form):
    full = wl.make(name, device="cuda")
    check_full(wl.subset(full, pick_sequences(full)), out_dtype=torch.float32 if out == "f32" else torch.bfloat16,
               form=form)


def test_long_causal_scaled_down_full():
    """The long-sequence workload's structure (causal, bias, 8 heads, head_dim 128) at
    lengths the oracle finishes in seconds, spanning many tiles with ragged tails."""
    rng = np.random.default_rng(5)
    lens = rng.integers(200, 1500, size=6)
    check_full(wl.make_custom(lens, lens, H=8, D=128, causal=True, bias=True, device="cuda", seed=77))


@pytest.mark.parametrize("form", ["planner", "two_pass"])
@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bias", [False, True])
def test_edge_lengths(mode, causal, bias, form):
    # empty sequences, single tokens, tile boundaries +-1, q > kv and q < kv, a kv tail
    # inside a tile, and the last sequence ending at the end of the buffers
    q = [0, 1, 127, 128, 129, 3, 0, 5, 1, 200, 64]
    kv = [4, 1, 127, 128, 129, 0, 0, 300, 257, 130, 1]
    std = 1.0 if mode == "softmax" else 0.5
    check_full(wl.make_custom(q, kv, H=2, D=128, mode=mode, causal=causal, bias=bias, value_std=std,
                              device="cuda", seed=11), form=form)


@pytest.mark.parametrize("dtype,D,form", [(torch.bfloat16, 64, "planner"), (torch.bfloat16, 64, "two_pass"),
                                          (torch.float32, 32, "planner"), (torch.float32, 64, "planner")])
def test_other_head_dims(dtype, D, form):
    check_full(wl.make_custom([7, 130, 64, 1], [200, 5, 64, 129], H=3, D=D, dtype=dtype, causal=True, bias=True,
                              device="cuda", seed=12), form=form)


@pytest.mark.parametrize("deterministic", [False, True])
def test_guard_bands_untouched(deterministic):
    """Rows past the last offset of every output buffer keep their canary values (both bf16
    backward forms: the fused one adds into an accumulator, the two-pass one writes rows)."""
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom([5, 130, 77], [129, 3, 200], H=2, D=128, causal=True, bias=True, device="cuda", seed=13)
    Tq, Tkv, pad = int(b.q_off[-1]), int(b.kv_off[-1]), 37
    canary = 1536.0  # exactly representable in bf16 and fp32

    def buf(T, like):
        t = torch.full((T + pad, b.H, b.D), canary, dtype=like.dtype, device="cuda")
        return t

    O, dQ, dK, dV = buf(Tq, b.Q), buf(Tq, b.Q), buf(Tkv, b.K), buf(Tkv, b.K)
    O = O.float()
    lse = torch.full((Tq + pad, b.H), canary, dtype=torch.float32, device="cuda")
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, b.mode, b.causal)
    jfa.jfa_plan_set_deterministic(plan, deterministic)
    assert jfa.jfa_plan_info(plan)["bwd_fused"] == (0 if deterministic else 1)
    jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, O=O, lse=lse)
    jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale, dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == 0
    for t, T in ((O, Tq), (dQ, Tq), (dK, Tkv), (dV, Tkv), (lse, Tq)):
        assert torch.all(t[T:] == canary)
        assert not torch.any(t[:T] == canary)
    r = parity.run_oracle(b)
    m = parity.compare({"O": O[:Tq], "lse": lse[:Tq], "dQ": dQ[:Tq], "dK": dK[:Tkv], "dV": dV[:Tkv]}, r)
    parity.assert_within(m)


def test_no_key_rows_are_exact_zero():
    b = wl.make_custom([3, 6], [0, 2], H=2, D=128, causal=True, device="cuda", seed=14)
    g = parity.run_gpu(b)
    O = g["O"].float().cpu()
    assert torch.all(O[0:3] == 0) and torch.all(torch.isneginf(g["lse"][0:3].cpu()))
    # second sequence: q=6 > kv=2, rows 0..3 see no key
    assert torch.all(O[3:7] == 0) and torch.all(g["dQ"][3:7].float().cpu() == 0)


# ----------------------------------------------------------------------------- full size

SAMPLES = {
    # (sequence selector, head, rows kept from the end)
    "causal_bias": [("longest", 0, 300), ("shortest", 3, 10**9), ("median", 7, 10**9)],
    "cross": [("longest_kv", 1, 10**9), ("shortest", 5, 10**9), ("median", 2, 10**9)],
    "gdpa_gelu": [("longest_kv", 0, 10**9), ("longest_q", 3, 10**9), ("median", 2, 10**9)],
    "gdpa_silu": [("longest_kv", 1, 10**9), ("longest_q", 2, 10**9)],
    "long_causal": [("longest", 0, 128), ("longest", 5, 128), ("shortest", 3, 200), ("median", 6, 160)],
}


def select(batch, how):
    ql, kl = batch.q_lens, batch.kv_lens
    if how == "longest":
        return int(np.argmax(ql))
    if how == "longest_kv":
        return int(np.argmax(kl))
    if how == "longest_q":
        return int(np.argmax(ql * 100000 + kl))
    if how == "shortest":
        return int(np.argmin(ql * 100000 + kl))
    if how == "median":
        return int(np.argsort(ql * 100000 + kl)[len(ql) // 2])
    raise ValueError(how)


@pytest.mark.parametrize("name", ["causal_bias", "cross", "gdpa_gelu", "gdpa_silu", "long_causal"])
def test_full_size_workload_sampled(name):
    batch = wl.make(name, device="cuda")
    # the launch configuration the benchmark times: O written in the input type
    g = parity.run_gpu(batch, out_dtype=torch.bfloat16)
    assert g["status"] == 0
    samples = []
    for how, h, keep in SAMPLES[name]:
        b = select(batch, how)
        q_len = int(batch.q_lens[b])
        samples.append((b, h, max(0, q_len - keep)))
    m = parity.sampled_parity(batch, g, samples)
    print(name, samples, m)
    parity.assert_within(m, softmax=batch.mode == "softmax")
    # whole-output sanity at full size: finite everywhere
    for k in ("O", "dQ", "dK", "dV"):
        assert torch.isfinite(g[k]).all(), k


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("causal,bias", [(False, False), (True, True)])
@pytest.mark.parametrize("long_len,split", [(300, 1), (3000, 0)])
def test_split_forward_both_kernels(mode, causal, bias, long_len, split):
    """One-tile query sequences over several key tiles (split items) next to a longer
    sequence: with a short neighbour the forward runs the kernel with split items on the
    mixed list, with a long one the plain kernel runs the short sequences unsplit."""
    from jagged_sequence_attention_gb300 import jfa
    rng = np.random.default_rng(12)
    q = rng.integers(1, 129, size=14).tolist() + [128, 1, long_len]
    kv = rng.integers(129, 1200, size=14).tolist() + [129, 4000, long_len]
    std = 1.0 if mode == "softmax" else 0.5
    b = wl.make_custom(q, kv, H=2, D=128, mode=mode, causal=causal, bias=bias, value_std=std,
                       device="cuda", seed=13)
    g, _ = check_full(b)
    assert jfa.jfa_plan_info(g["plan"])["fwd_split"] == split


@pytest.mark.parametrize("lens,split", [([2100, 600, 129, 256], 1), ([600, 1700, 129, 256], 0)])
def test_split_forward_long_odd_tile(lens, split):
    """The last, odd query tile of a longer causal sequence: split (its key range cut in two
    halves run as the pair's two tiles, then merged) when it visits 16 key tiles or more
    (2,100 tokens: 17 tiles), not otherwise (600 tokens: 5 tiles; 1,700 tokens: 14 tiles, an
    even count, has no such tile); the other sequences keep their plain pairs.  Full outputs
    and gradients against the oracle."""
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom(lens, lens, H=2, D=128, mode="softmax", causal=True, bias=True, device="cuda", seed=14)
    for o_dtype in (torch.float32, torch.bfloat16):
        g, _ = check_full(b, out_dtype=o_dtype)
        assert jfa.jfa_plan_info(g["plan"])["fwd_split"] == split
