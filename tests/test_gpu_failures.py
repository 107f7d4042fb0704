"""The kernels' own failure reports, made to happen without a GPU fault.

- Work-item checks (JFA_ERR_DEVICE_BOUNDS).  Every kernel checks each work item it reads
  against its plan before touching anything the item indexes, skips one that does not fit
  and reports it.  The planner never writes such an item, so the tests plant one with
  jfa_plan_set_work_item -- a sequence or head outside the batch, a tile past the
  sequence, or an inner count other than the one the tile ranges give -- in each pass's
  list, for the two-pass, the fused and the short-query bf16 backward, the fp32 kernels
  and a shared key/value plan.  Every planted item is caught by the check before any access it would
  steer.
- Bounded waits (JFA_ERR_TIMEOUT).  A test build of the forward kernel
  (JFA_TEST_STALL_MMA, pipeline waits limited to 20 ms) makes its tensor-core issuer wait
  on a barrier that nothing arrives on.  The wait runs out, every role of each CTA winds
  down (each still waits, with the normal limit, for the loads and products it issued)
  and the plan reports the timeout.

After each, a normal call on a fresh plan is compared with the oracle: the context stays
usable."""
import ctypes
import time

import numpy as np
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


def _check_normal_call_is_right(b):
    g = parity.run_gpu(b)
    assert g["status"] == 0
    softmax = b.mode == "softmax"
    parity.assert_within(parity.compare(g, parity.run_oracle(b), softmax=softmax), softmax=softmax)


def _bad_item(kind, b, item):
    """A copy of the real item `item` (sequence, head, tile, count) made not to fit."""
    seq, head, tile, count = (int(x) for x in item)
    if kind == "sequence":
        return [b.B + 5, head, tile, count]
    if kind == "head":
        return [seq, b.H, tile, count]
    if kind == "tile":
        return [seq, head, tile + 1000, count]
    return [seq, head, tile, count + 3]  # "count"


def _first_item(jfa, plan, b, pass_):
    """Item 0 of a pass as the host planner lists it for this batch (same code as the plan)."""
    L = jfa.lib()
    q = np.ascontiguousarray(b.q_off, dtype=np.int32)
    k = np.ascontiguousarray(b.kv_off, dtype=np.int32)
    info = jfa.jfa_plan_info(plan)
    grid = info[{0: "fwd_grid", 1: "bwd_grid", 2: "dq_grid"}[pass_]]
    n = info[{0: "fwd_items", 1: "bwd_items", 2: "dq_items"}[pass_]]
    items = np.zeros((max(1, n), 4), dtype=np.int32)
    offs = np.zeros(grid + 1, dtype=np.int32)
    win = -1 if b.window is None else int(b.window)
    st = L.jfa_worklist_build(q.ctypes.data, k.ctypes.data, b.B, b.H, int(b.causal), win, pass_, grid,
                              items.ctypes.data, offs.ctypes.data, None)
    assert st == 0
    return items[0]


CASES = [
    # (pass, kind, deterministic, dtype)
    (0, "sequence", False, torch.bfloat16),
    (0, "head", False, torch.bfloat16),
    (0, "count", False, torch.bfloat16),
    (1, "sequence", True, torch.bfloat16),
    (1, "tile", True, torch.bfloat16),
    (1, "count", True, torch.bfloat16),
    (1, "tile", False, torch.bfloat16),   # the fused backward
    (1, "count", False, torch.bfloat16),
    (2, "head", True, torch.bfloat16),
    (2, "count", True, torch.bfloat16),
    (0, "sequence", False, torch.float32),
    (1, "count", False, torch.float32),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_planted_work_item_is_skipped_and_reported(jfa, case):
    pass_, kind, deterministic, dtype = CASES[case]
    D = 64 if dtype == torch.float32 else 128
    b = wl.make_custom([300, 129, 40], [300, 129, 40], H=2, D=D, dtype=dtype, causal=True, bias=True,
                       device="cuda", seed=501 + case)
    plan = jfa.plan_for(b, deterministic=deterministic)
    if dtype == torch.bfloat16 and pass_ == 1:
        assert jfa.jfa_plan_info(plan)["bwd_fused"] == (0 if deterministic else 1)
    bad = _bad_item(kind, b, _first_item(jfa, plan, b, pass_))
    if pass_ > 0:  # the forward's outputs first, from the plan's own items
        O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    jfa.jfa_plan_set_work_item(plan, pass_, 0, bad)
    if pass_ == 0:
        jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    else:
        jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_ERR_DEVICE_BOUNDS
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK  # the status word was read and cleared
    _check_normal_call_is_right(b)


@pytest.mark.parametrize("kind", ["sequence", "tile", "count"])
def test_planted_item_in_the_short_query_backward(jfa, kind):
    # query sets of one tile, no causal mask: jfa_bwd runs the short-query kernel (pass 3)
    b = wl.make_custom([40, 7, 64], [300, 129, 1000], H=2, D=64, causal=False, device="cuda", seed=540)
    plan = jfa.plan_for(b)
    assert jfa.jfa_plan_info(plan)["bwd_short"] == 64
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_OK
    seq = [b.B + 5, 0, 0, 1] if kind == "sequence" else [0, 0, 1, 3] if kind == "tile" else [0, 0, 0, 2]
    jfa.jfa_plan_set_work_item(plan, 3, 0, seq)
    jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, None, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_ERR_DEVICE_BOUNDS
    _check_normal_call_is_right(b)


def test_planted_item_in_the_short_query_gdpa_forward(jfa):
    b = wl.make_custom([40, 7, 64], [300, 129, 1000], H=2, D=64, mode="silu", causal=False, value_std=0.5,
                       device="cuda", seed=545)
    plan = jfa.plan_for(b)
    assert jfa.jfa_plan_info(plan)["fwd_short"] == 64
    jfa.jfa_plan_set_work_item(plan, 4, 0, [0, 0, 0, 5])  # an inner count the sequence does not have
    jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_ERR_DEVICE_BOUNDS
    _check_normal_call_is_right(b)


@pytest.mark.parametrize("kind", ["sequence", "count"])
def test_planted_item_in_the_packed_softmax_forward(jfa, kind):
    b = wl.make_custom([40, 7, 64], [300, 129, 1000], H=2, D=64, causal=False, device="cuda", seed=546)
    plan = jfa.plan_for(b)
    assert jfa.jfa_plan_info(plan)["fwd_short"] == 64
    item = [b.B + 1, 0, 0, 3] if kind == "sequence" else [2, 1, 0, 2]  # sequence 2 has 8 key tiles
    jfa.jfa_plan_set_work_item(plan, 4, 0, item)
    jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_ERR_DEVICE_BOUNDS
    _check_normal_call_is_right(b)


def test_planted_item_on_a_shared_key_value_plan(jfa):
    b = wl.make_shared_kv([40, 7, 128, 1, 64], [300, 129], [0, 1, 0, 0, 1], H=2, D=128, causal=True, bias=True,
                          seed=520, device="cuda")
    plan = jfa.plan_for(b)
    O, lse = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    # dK/dV item 0 is a key tile of one of the two users; an inner count it does not have
    jfa.jfa_plan_set_work_item(plan, 1, 0, [0, 0, 0, 10**6])
    jfa.jfa_bwd(plan, b.Q, b.K, b.V, O, b.dO, lse, b.bias, b.scale)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == jfa.JFA_ERR_DEVICE_BOUNDS
    _check_normal_call_is_right(b)


def test_set_work_item_argument_errors(jfa):
    b = wl.make_custom([40], [40], H=1, D=128, device="cuda", seed=521)
    plan = jfa.plan_for(b)
    for pass_, index in ((5, 0), (-1, 0), (0, -1), (0, 10**6), (3, 10**6), (4, 10**6)):
        with pytest.raises(jfa.JFAError) as e:
            jfa.jfa_plan_set_work_item(plan, pass_, index, [0, 0, 0, 1])
        assert e.value.status == jfa.JFA_ERR_INVALID_ARG


def test_pipeline_wait_runs_out_and_is_reported(jfa):
    from jagged_sequence_attention_gb300 import _build
    path = _build.build_variant("jfa_stall", ["JFA_TEST_STALL_MMA", "JFA_WAIT_TIMEOUT_NS=20000000ull"])
    L = jfa.load_library(path)
    b = wl.make_custom([300, 129, 40], [300, 129, 40], H=2, D=128, causal=True, bias=True, device="cuda",
                       seed=530)
    q = np.ascontiguousarray(b.q_off, dtype=np.int32)
    k = np.ascontiguousarray(b.kv_off, dtype=np.int32)
    stream = jfa._stream()
    plan = ctypes.c_void_p()
    assert L.jfa_plan_create(q.ctypes.data, k.ctypes.data, b.B, b.H, b.D, jfa.JFA_SOFTMAX, 1, 0, stream,
                             ctypes.byref(plan)) == jfa.JFA_OK
    O = torch.full(b.Q.shape, float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.empty((b.Q.shape[0], b.H), dtype=torch.float32, device="cuda")
    t0 = time.time()
    assert L.jfa_fwd(plan, jfa.JFA_BF16, jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V), jfa.JFA_BIAS_RELPOS32,
                     jfa._ptr(b.bias), ctypes.c_float(b.scale), jfa._ptr(O), jfa.JFA_F32, jfa._ptr(lse),
                     stream) == jfa.JFA_OK
    st = L.jfa_plan_device_status(plan, stream)
    elapsed = time.time() - t0
    assert st == jfa.JFA_ERR_TIMEOUT, st
    assert elapsed < 10.0, elapsed  # the 20 ms limit, not a hang
    assert L.jfa_plan_destroy(plan) == jfa.JFA_OK
    torch.cuda.synchronize()
    _check_normal_call_is_right(b)
