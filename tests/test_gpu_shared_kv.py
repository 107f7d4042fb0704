"""Shared key/value attention on the GPU (the in-kernel broadcast of the PyTorch blog
"In-Kernel Broadcast Optimization: Co-Designing Kernels for RecSys Inference", section
3), through the C-ABI, against the CPU oracle.  The oracle attends to the broadcast
history and sums the key/value gradients over query sets that share a user.

Also checked on the GPU itself: the plain path run on an explicitly broadcast copy of
the batch gives bitwise the same O, lse and dQ.  Each query set's work is the same
there, while dK and dV come from one accumulation over all of a user's query sets
rather than from a sum of per-copy results."""
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


def check(batch, out_dtype=torch.float32, bias_grad=False):
    from jagged_sequence_attention_gb300 import jfa
    out = jfa.attention(batch, with_backward=True, out_dtype=out_dtype, bias_grad=bias_grad)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(out["plan"]) == 0
    info = jfa.jfa_plan_info(out["plan"])
    assert info["users"] == batch.kv_off.size - 1
    r = parity.run_oracle(batch, True, bias_grads=bias_grad)
    m = parity.compare(out, r, softmax=batch.mode == "softmax", with_backward=True)
    if bias_grad:
        m["dbias_rel_frob"] = parity.rel_frob(parity.np64(out["dbias"]), r["dbias"])
    print(batch.name, m)
    parity.assert_within(m, softmax=batch.mode == "softmax")
    if bias_grad:
        assert m["dbias_rel_frob"] <= parity.BWD_REL_FROB, m
    return out, r


def cross_batch(seed, n_users=6, ratio=5, q_max=64, kv_lo=100, kv_hi=2000, unused=True, **kw):
    g = np.random.default_rng(seed)
    users = g.integers(kv_lo, kv_hi, size=n_users).tolist()
    live = n_users - 1 if unused else n_users  # the last user: no query set
    kv_map = np.repeat(np.arange(live), ratio)
    g.shuffle(kv_map)
    q = g.integers(1, q_max + 1, size=kv_map.size).tolist()
    return wl.make_shared_kv(q, users, kv_map, seed=seed, device="cuda", **kw)


@pytest.mark.parametrize("D", [128, 64])
def test_cross_attention(D):
    b = cross_batch(81, H=4, D=D)
    out, r = check(b)
    # the unused user's rows: zero gradients
    rows = slice(int(b.kv_off[-2]), None)
    assert float(out["dK"][rows].abs().max()) == 0 and float(out["dV"][rows].abs().max()) == 0


@pytest.mark.parametrize("mode", ["gelu_tanh", "silu"])
def test_gdpa(mode):
    check(cross_batch(82, H=2, D=128, mode=mode, value_std=0.5))


def test_causal_with_bias_and_its_gradient():
    # bottom-right alignment per query set against its user's length; q > kv too
    users = [300, 129, 700, 40]
    kv_map = [0, 2, 0, 1, 2, 2, 3, 0, 1]
    q = [300, 64, 1, 129, 700, 5, 60, 257, 200]
    check(wl.make_shared_kv(q, users, kv_map, H=2, D=128, causal=True, bias=True, seed=83, device="cuda"),
          bias_grad=True)


def test_window():
    users = [900, 300]
    kv_map = [0, 1, 0, 0, 1]
    q = [900, 300, 128, 513, 37]
    check(wl.make_shared_kv(q, users, kv_map, H=2, D=128, causal=True, bias=True, seed=84, device="cuda", window=200))


def test_dense_bias_and_its_gradient():
    check(cross_batch(85, n_users=4, ratio=3, kv_hi=600, H=2, D=128, dense_bias=True), bias_grad=True)


@pytest.mark.parametrize("D", [32, 64])
def test_fp32(D):
    check(cross_batch(86, n_users=4, ratio=3, kv_hi=700, H=2, D=D, dtype=torch.float32, bias=True), bias_grad=True)


def test_bf16_output():
    check(cross_batch(87, H=2, D=128), out_dtype=torch.bfloat16)


def test_empty_users_and_query_sets():
    users = [0, 150, 0]
    kv_map = [0, 1, 1, 2, 1]
    q = [10, 0, 20, 3, 130]
    check(wl.make_shared_kv(q, users, kv_map, H=2, D=128, bias=True, seed=88, device="cuda"))


def test_same_as_the_plain_path_on_a_broadcast_copy():
    from jagged_sequence_attention_gb300 import jfa
    b = cross_batch(89, H=2, D=128, bias=True)
    shared = jfa.attention(b, with_backward=True, out_dtype=torch.float32)
    # explicit broadcast: each query set gets its own copy of its user's rows
    rows = np.concatenate([np.arange(b.kv_off[u], b.kv_off[u + 1]) for u in b.kv_map]).astype(np.int64)
    lens = np.diff(b.kv_off.astype(np.int64))[b.kv_map]
    idx = torch.from_numpy(rows).cuda()
    plain = wl.Batch("broadcast", b.q_off, wl.offsets(lens), b.Q, b.K.index_select(0, idx).contiguous(),
                     b.V.index_select(0, idx).contiguous(), b.dO, b.bias, b.scale, b.mode, b.causal, b.H, b.D)
    # the two-pass backward on the plain batch, as a shared key/value plan always runs it
    ref = jfa.attention(plain, with_backward=True, out_dtype=torch.float32, deterministic=True)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(shared["plan"]) == 0 and jfa.jfa_plan_device_status(ref["plan"]) == 0
    for k in ("O", "lse", "dQ"):
        assert torch.equal(shared[k], ref[k]), k
    dK = torch.zeros_like(b.K, dtype=torch.float32).index_add_(0, idx, ref["dK"].float())
    dV = torch.zeros_like(b.V, dtype=torch.float32).index_add_(0, idx, ref["dV"].float())
    for x, y in ((shared["dK"].float(), dK), (shared["dV"].float(), dV)):
        assert float((x - y).norm() / y.norm()) <= parity.BWD_REL_FROB


def test_argument_errors():
    from jagged_sequence_attention_gb300 import jfa
    with pytest.raises(jfa.JFAError) as e:   # an index outside [0, U)
        jfa.jfa_plan_create_shared_kv([0, 5, 9], [0, 10], [0, 1], 2, 128)
    assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    with pytest.raises(jfa.JFAError) as e:   # a window without causal
        jfa.jfa_plan_create_shared_kv([0, 5], [0, 10], [0], 2, 128, window=3)
    assert e.value.status == jfa.JFA_ERR_INVALID_ARG


def request_batch(seed, n_users=5, per_user=12, **kw):
    """Query sets of a user next to each other in Q (a request's candidates), so that
    the merged view packs them into shared tiles."""
    g = np.random.default_rng(seed)
    users = g.integers(100, 1500, size=n_users).tolist()
    kv_map = np.repeat(np.arange(n_users), per_user)
    q = g.integers(1, 65, size=kv_map.size).tolist()
    return wl.make_shared_kv(q, users, kv_map, seed=seed, device="cuda", **kw)


@pytest.mark.parametrize("mode", ["softmax", "silu"])
def test_merged_view(mode):
    from jagged_sequence_attention_gb300 import jfa
    b = request_batch(90, H=2, D=128, mode=mode, value_std=1.0 if mode == "softmax" else 0.5)
    out, _ = check(b)
    info = jfa.jfa_plan_info(out["plan"])
    assert info["merged"] == 5            # one query sequence per user


def test_merged_view_with_dense_bias():
    check(request_batch(91, H=2, D=64, dense_bias=True), bias_grad=True)


def test_merged_and_per_set_views_agree():
    # a zero relative-position table changes nothing but forces the per-set view
    from jagged_sequence_attention_gb300 import jfa
    b = request_batch(92, H=2, D=128)
    plan = jfa.plan_for(b)
    zero = torch.zeros((b.H, 32), dtype=torch.float32, device="cuda")
    O1, lse1 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    O2, lse2 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, zero, b.scale, out_dtype=torch.float32)
    g1 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O1, b.dO, lse1, None, b.scale)
    g2 = jfa.jfa_bwd(plan, b.Q, b.K, b.V, O2, b.dO, lse2, zero, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == 0
    assert float((O1 - O2).abs().max()) <= 2 * parity.FWD_MAX_ABS
    assert float((lse1 - lse2).abs().max()) <= 2 * parity.LSE_MAX_ABS
    for x, y in zip(g1, g2):
        assert float((x.float() - y.float()).norm() / y.float().norm()) <= 2 * parity.BWD_REL_FROB
