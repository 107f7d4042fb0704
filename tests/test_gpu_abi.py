"""C-ABI behaviour on a GPU: argument errors are reported as status codes before any
launch, plans report their facts, the timing hook counts launches, and the device
status word stays clear after correct runs."""
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jfa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    return m


def status_of(jfa, fn, *a, **k):
    try:
        fn(*a, **k)
    except jfa.JFAError as e:
        return e.status
    return jfa.JFA_OK


def test_plan_create_rejects_bad_arguments(jfa):
    assert status_of(jfa, jfa.jfa_plan_create, [0, 5, 3], [0, 1, 2], 2, 128) == jfa.JFA_ERR_INVALID_ARG
    assert status_of(jfa, jfa.jfa_plan_create, [1, 5], [0, 1], 2, 128) == jfa.JFA_ERR_INVALID_ARG
    assert status_of(jfa, jfa.jfa_plan_create, [0, 5], [0, 1], 0, 128) == jfa.JFA_ERR_INVALID_ARG
    assert status_of(jfa, jfa.jfa_plan_create, [0, 5], [0, 1], 2, 48) == jfa.JFA_ERR_UNSUPPORTED
    assert status_of(jfa, jfa.jfa_plan_create, [0, 5], [0, 1], 2, 128, mode=7) == jfa.JFA_ERR_INVALID_ARG


def test_plan_info_and_device_offsets(jfa):
    q, kv = [3, 0, 300], [5, 7, 129]
    p = jfa.jfa_plan_create(torch.tensor(wl.offsets(q), device="cuda"), torch.tensor(wl.offsets(kv), device="cuda"),
                            4, 128, "softmax", True)
    info = p.info()
    assert info["T_q"] == 303 and info["T_kv"] == 141 and info["B"] == 3 and info["H"] == 4
    assert info["fwd_items"] == 4 * (1 + 0 + 2) and info["bwd_items"] == 4 * (1 + 1 + 2)
    assert info["dq_items"] == 4 * (1 + 0 + 3) and 1 <= info["dq_grid"] <= info["num_sms"]
    assert 1 <= info["fwd_grid"] <= info["num_sms"]


def test_fwd_bwd_reject_bad_arguments(jfa):
    b = wl.make_custom([5, 9], [7, 9], H=2, D=128, device="cuda")
    p = jfa.jfa_plan_create(b.q_off, b.kv_off, 2, 128)
    O = torch.empty_like(b.Q)
    lse = torch.empty(b.Q.shape[0], 2, device="cuda")
    # misaligned pointer
    Qm = torch.empty(b.Q.numel() + 8, dtype=b.Q.dtype, device="cuda")[1:1 + b.Q.numel()].view(b.Q.shape)
    assert status_of(jfa, jfa.jfa_fwd, p, Qm, b.K, b.V, O=O, lse=lse) == jfa.JFA_ERR_INVALID_ARG
    # softmax needs lse
    r = jfa.lib().jfa_fwd(p.handle, jfa.JFA_BF16, jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V), 0, None, 0.1,
                          jfa._ptr(O), jfa.JFA_BF16, None, jfa._stream())
    assert r == jfa.JFA_ERR_INVALID_ARG
    # bias kind without a table
    r = jfa.lib().jfa_fwd(p.handle, jfa.JFA_BF16, jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V), 1, None, 0.1,
                          jfa._ptr(O), jfa.JFA_BF16, jfa._ptr(lse), jfa._stream())
    assert r == jfa.JFA_ERR_INVALID_ARG
    # too small a workspace (the row terms alone need 256 bytes here)
    ws = torch.empty(128, dtype=torch.uint8, device="cuda")
    jfa.jfa_fwd(p, b.Q, b.K, b.V, O=O, lse=lse)
    assert status_of(jfa, jfa.jfa_bwd, p, b.Q, b.K, b.V, O, b.dO, lse, workspace=ws) == jfa.JFA_ERR_INVALID_ARG
    # fp32 inputs need an fp32 output
    q32 = b.Q.float()
    assert status_of(jfa, jfa.jfa_fwd, p, q32, b.K.float(), b.V.float(), O=O, lse=lse) == jfa.JFA_ERR_UNSUPPORTED
    # unsupported head_dim for bf16
    p32 = jfa.jfa_plan_create(b.q_off, b.kv_off, 2, 32)
    q = torch.zeros(b.Q.shape[0], 2, 32, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(b.K.shape[0], 2, 32, dtype=torch.bfloat16, device="cuda")
    assert status_of(jfa, jfa.jfa_fwd, p32, q, k, k) == jfa.JFA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(p) == jfa.JFA_OK


def test_timing_hook_counts_launches(jfa):
    b = wl.make_custom([130, 40], [130, 300], H=2, D=128, causal=True, device="cuda")
    p = jfa.jfa_plan_create(b.q_off, b.kv_off, 2, 128, "softmax", True)
    jfa.jfa_plan_set_timing(p, True)
    for _ in range(3):
        O, lse = jfa.jfa_fwd(p, b.Q, b.K, b.V)
        jfa.jfa_bwd(p, b.Q, b.K, b.V, O, b.dO, lse)
    t = jfa.jfa_plan_kernel_times(p)
    # bf16 on a fused backward: the main kernel adds dQ into an fp32 accumulator that the
    # conversion pass scales and writes; the dQ pass does not run
    assert jfa.jfa_plan_info(p)["bwd_fused"] == 1
    assert {k: v[1] for k, v in t.items()} == {"fwd": 3, "bwd_pre": 3, "bwd_main": 3, "bwd_post": 3, "bwd_dq": 0}
    assert all(v[0] > 0 for v in t.values() if v[1])
    assert all(v[1] == 0 for v in jfa.jfa_plan_kernel_times(p).values())


def test_empty_batch_is_a_no_op(jfa):
    p = jfa.jfa_plan_create([0, 0], [0, 0], 2, 128)
    e = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(0, 2, device="cuda")
    jfa.jfa_fwd(p, e, e, e, O=e.clone(), lse=lse)
    jfa.jfa_bwd(p, e, e, e, e, e, lse)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(p) == jfa.JFA_OK
