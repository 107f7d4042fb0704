"""Thin Python binding of libjfa (include/jfa.h), same entry-point names.

Argument marshalling only: torch tensors are passed as raw device pointers with
the current CUDA stream; every step of the computation runs in the library's
kernels.  The library must have been built (``__graft_entry__.build()`` or
``python -m jagged_sequence_attention_gb300._build``); if it is missing or fails to
load, every call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libjfa.so")

JFA_OK, JFA_ERR_INVALID_ARG, JFA_ERR_UNSUPPORTED, JFA_ERR_CUDA = 0, 1, 2, 3
JFA_ERR_TIMEOUT, JFA_ERR_DEVICE_BOUNDS, JFA_ERR_PLAN_MISMATCH, JFA_ERR_NO_DEVICE = 4, 5, 6, 7
JFA_ERR_SCRATCH_LIMIT = 8
JFA_STATIC_SCRATCH_BYTES = 64 << 20
JFA_SOFTMAX, JFA_GDPA_GELU_TANH, JFA_GDPA_SILU = 0, 1, 2
JFA_BF16, JFA_F32 = 0, 1
JFA_BIAS_NONE, JFA_BIAS_RELPOS32, JFA_BIAS_DENSE = 0, 1, 2

MODES = {"softmax": JFA_SOFTMAX, "gelu_tanh": JFA_GDPA_GELU_TANH, "silu": JFA_GDPA_SILU}
DTYPES = {torch.bfloat16: JFA_BF16, torch.float32: JFA_F32}

EXPORTED = ["jfa_plan_create", "jfa_plan_create_ex", "jfa_plan_destroy", "jfa_plan_info", "jfa_fwd", "jfa_bwd_workspace_size",
            "jfa_bwd", "jfa_plan_device_status", "jfa_worklist_size", "jfa_worklist_build",
            "jfa_status_string", "jfa_plan_set_timing", "jfa_plan_kernel_times", "jfa_bwd_static_scratch",
            "jfa_partition_sequences", "jfa_bwd_ex_workspace_size", "jfa_bwd_ex", "jfa_plan_create_shared_kv",
            "jfa_partition_users", "jfa_plan_set_deterministic", "jfa_plan_set_work_item"]


class JFAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {jfa_status_string(status)} (status {status})")


_lib = None


def lib():
    """Load libjfa.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libjfa.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
        _lib = load_library(_LIB_PATH)
    return _lib


def load_library(path):
    """A build of the library at `path` (the main one, or a test build) with the C-ABI's
    argument and result types declared."""
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER
    L.jfa_plan_create.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, P(vp)]
    L.jfa_plan_create_ex.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, P(vp)]
    L.jfa_plan_create_shared_kv.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, P(vp)]
    L.jfa_plan_destroy.argtypes = [vp]
    L.jfa_plan_info.argtypes = [vp, P(i64), i32]
    L.jfa_fwd.argtypes = [vp, i32, vp, vp, vp, i32, vp, f32, vp, i32, vp, vp]
    L.jfa_bwd_workspace_size.argtypes = [vp, i32]
    L.jfa_bwd_workspace_size.restype = sz
    L.jfa_bwd.argtypes = [vp, i32, vp, vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, vp, sz, vp]
    L.jfa_bwd_ex_workspace_size.argtypes = [vp, i32, i32]
    L.jfa_bwd_ex_workspace_size.restype = sz
    L.jfa_bwd_ex.argtypes = [vp, i32, vp, vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, vp, vp, sz, vp]
    L.jfa_bwd_static_scratch.argtypes = [vp, i32, vp, vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, vp]
    L.jfa_plan_device_status.argtypes = [vp, vp]
    L.jfa_partition_sequences.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp]
    L.jfa_partition_users.argtypes = [vp, i32, vp, i32, vp, i32, i32, i32, i32, vp, vp]
    L.jfa_worklist_size.argtypes = [vp, vp, i32, i32, i32, i32, i32, P(i64)]
    L.jfa_worklist_build.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.jfa_plan_set_timing.argtypes = [vp, i32]
    L.jfa_plan_set_deterministic.argtypes = [vp, i32]
    L.jfa_plan_set_work_item.argtypes = [vp, i32, i64, vp]
    L.jfa_plan_kernel_times.argtypes = [vp, vp, vp]
    L.jfa_status_string.argtypes = [i32]
    L.jfa_status_string.restype = ctypes.c_char_p
    for name in ("jfa_plan_create", "jfa_plan_create_ex", "jfa_plan_destroy", "jfa_plan_info", "jfa_fwd", "jfa_bwd",
                 "jfa_plan_device_status", "jfa_worklist_size", "jfa_worklist_build", "jfa_plan_set_timing",
                 "jfa_plan_kernel_times", "jfa_bwd_static_scratch", "jfa_partition_sequences", "jfa_bwd_ex",
                 "jfa_plan_create_shared_kv", "jfa_partition_users", "jfa_plan_set_deterministic",
                 "jfa_plan_set_work_item"):
        getattr(L, name).restype = i32
    return L


def jfa_status_string(status: int) -> str:
    return lib().jfa_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != JFA_OK:
        raise JFAError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    """The tensor's data pointer.  The library reads and writes dense row-major arrays,
    so a tensor with any other strides is refused rather than misread."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise JFAError("tensor layout (must be contiguous)", JFA_ERR_INVALID_ARG)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class Plan:
    """Owns a jfa_plan handle."""

    def __init__(self, handle, B, H, D, mode, causal, Tq, Tkv):
        self.handle = handle
        self.B, self.H, self.D, self.mode, self.causal = B, H, D, mode, causal
        self.Tq, self.Tkv = Tq, Tkv

    def info(self) -> dict:
        return jfa_plan_info(self)

    def __del__(self):
        try:
            if self.handle is not None and _lib is not None:
                _lib.jfa_plan_destroy(self.handle)
        finally:
            self.handle = None


def _win(window) -> int:
    return -1 if window is None else int(window)


def jfa_plan_create(q_offsets, kv_offsets, H: int, D: int, mode="softmax", causal=False, stream=None,
                    window=None) -> Plan:
    """Offsets: host int32 arrays (or CUDA int32 tensors, copied with a sync).  window: sliding
    window W (query i sees keys i' - W .. i'; needs causal), None for none."""
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    on_dev = isinstance(q_offsets, torch.Tensor) and q_offsets.is_cuda
    if on_dev:
        qo = q_offsets.to(torch.int32).contiguous()
        ko = kv_offsets.to(torch.int32).contiguous()
        qp, kp, B = _ptr(qo), _ptr(ko), qo.numel() - 1
        Tq, Tkv = None, None
    else:
        qo = _i32(q_offsets.cpu() if isinstance(q_offsets, torch.Tensor) else q_offsets)
        ko = _i32(kv_offsets.cpu() if isinstance(kv_offsets, torch.Tensor) else kv_offsets)
        qp, kp, B = qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p), qo.size - 1
        Tq, Tkv = int(qo[-1]), int(ko[-1])
    if (qo.numel() if on_dev else qo.size) != (ko.numel() if on_dev else ko.size):
        raise JFAError("jfa_plan_create", JFA_ERR_INVALID_ARG)
    h = ctypes.c_void_p()
    _check("jfa_plan_create", lib().jfa_plan_create_ex(qp, kp, int(B), int(H), int(D), m, int(bool(causal)),
                                                        _win(window), int(on_dev), _stream(stream), ctypes.byref(h)))
    plan = Plan(h, int(B), int(H), int(D), m, bool(causal), Tq, Tkv)
    plan.window = window
    if Tq is None:
        inf = jfa_plan_info(plan)
        plan.Tq, plan.Tkv = inf["T_q"], inf["T_kv"]
    return plan


def jfa_plan_create_shared_kv(q_offsets, kv_offsets, kv_index, H: int, D: int, mode="softmax", causal=False,
                              stream=None, window=None) -> Plan:
    """Shared key/value plan: query set b attends to the rows of user kv_index[b]
    (kv_offsets over the users).  Host arrays."""
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    qo, ko, ki = _i32(q_offsets), _i32(kv_offsets), _i32(kv_index)
    B, U = qo.size - 1, ko.size - 1
    if ki.size != B:
        raise JFAError("jfa_plan_create_shared_kv", JFA_ERR_INVALID_ARG)
    h = ctypes.c_void_p()
    vp = ctypes.c_void_p
    _check("jfa_plan_create_shared_kv", lib().jfa_plan_create_shared_kv(
        qo.ctypes.data_as(vp), int(B), ko.ctypes.data_as(vp), int(U), ki.ctypes.data_as(vp), int(H), int(D), m,
        int(bool(causal)), _win(window), 0, _stream(stream), ctypes.byref(h)))
    plan = Plan(h, int(B), int(H), int(D), m, bool(causal), int(qo[-1]), int(ko[-1]))
    plan.window = window
    return plan


def jfa_plan_destroy(plan: Plan):
    if plan.handle is not None:
        _check("jfa_plan_destroy", lib().jfa_plan_destroy(plan.handle))
        plan.handle = None


INFO_KEYS = ["T_q", "T_kv", "B", "H", "D", "mode", "causal", "fwd_items", "fwd_grid", "bwd_items", "bwd_grid",
             "num_sms", "dq_items", "dq_grid", "window", "pairs", "users", "merged",
             "fwd_split", "bwd_fused", "bwd_short", "fwd_short"]


def jfa_plan_info(plan: Plan) -> dict:
    buf = (ctypes.c_int64 * len(INFO_KEYS))()
    _check("jfa_plan_info", lib().jfa_plan_info(plan.handle, buf, len(INFO_KEYS)))
    return dict(zip(INFO_KEYS, [int(x) for x in buf]))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in DTYPES:
        raise JFAError("dtype", JFA_ERR_UNSUPPORTED)
    return DTYPES[t.dtype]


def _bias_args(bias, dense=None):
    """(kind, pointer): the bucket table [H, 32], or a dense per-pair bias [H, P]."""
    if dense is not None:
        if bias is not None:
            raise JFAError("bias", JFA_ERR_INVALID_ARG)
        return JFA_BIAS_DENSE, _ptr(dense)
    if bias is None:
        return JFA_BIAS_NONE, None
    return JFA_BIAS_RELPOS32, _ptr(bias)


def jfa_fwd(plan: Plan, Q, K, V, bias=None, scale=None, O=None, lse=None, stream=None, out_dtype=None,
            dense_bias=None):
    """Returns (O, lse); lse is None in GDPA modes.  O is written in out_dtype (default:
    O's dtype if given, else Q's).  bias: the bucket table [H, 32]; dense_bias: a dense
    per-pair bias [H, P] instead."""
    dt = _dtype_code(Q)
    scale = 1.0 / float(plan.D) ** 0.5 if scale is None else float(scale)
    if O is None:
        O = torch.empty(Q.shape, dtype=out_dtype or Q.dtype, device=Q.device)
    if lse is None and plan.mode == JFA_SOFTMAX:
        lse = torch.empty((Q.shape[0], plan.H), dtype=torch.float32, device=Q.device)
    bk, bp = _bias_args(bias, dense_bias)
    _check("jfa_fwd", lib().jfa_fwd(plan.handle, dt, _ptr(Q), _ptr(K), _ptr(V), bk, bp, scale, _ptr(O),
                                    _dtype_code(O), _ptr(lse), _stream(stream)))
    return O, lse


def jfa_bwd_workspace_size(plan: Plan, dtype=torch.bfloat16) -> int:
    return int(lib().jfa_bwd_workspace_size(plan.handle, DTYPES[dtype]))


def jfa_bwd(plan: Plan, Q, K, V, O, dO, lse, bias=None, scale=None, dQ=None, dK=None, dV=None, workspace=None,
            stream=None, dense_bias=None):
    """Returns (dQ, dK, dV)."""
    dt = _dtype_code(Q)
    scale = 1.0 / float(plan.D) ** 0.5 if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    need = jfa_bwd_workspace_size(plan, Q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=Q.device)
    bk, bp = _bias_args(bias, dense_bias)
    _check("jfa_bwd", lib().jfa_bwd(plan.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _dtype_code(O), _ptr(dO),
                                    _ptr(lse), bk, bp, scale, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))
    return dQ, dK, dV


def jfa_bwd_ex_workspace_size(plan: Plan, dtype=torch.bfloat16, bias_grad=True, dense=False) -> int:
    kind = (JFA_BIAS_DENSE if dense else JFA_BIAS_RELPOS32) if bias_grad else JFA_BIAS_NONE
    return int(lib().jfa_bwd_ex_workspace_size(plan.handle, DTYPES[dtype], kind))


def jfa_bwd_ex(plan: Plan, Q, K, V, O, dO, lse, bias, scale=None, dQ=None, dK=None, dV=None, dbias=None,
               workspace=None, stream=None, dense_bias=None):
    """jfa_bwd plus the gradient of the bias: of the bucket table [H, 32], or with
    dense_bias of the dense per-pair bias [H, P] (fp32).  Returns (dQ, dK, dV, dbias)."""
    dt = _dtype_code(Q)
    scale = 1.0 / float(plan.D) ** 0.5 if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    if dbias is None:
        shape = (plan.H, 32) if dense_bias is None else tuple(dense_bias.shape)
        dbias = torch.empty(shape, dtype=torch.float32, device=Q.device)
    need = jfa_bwd_ex_workspace_size(plan, Q.dtype, dense=dense_bias is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=Q.device)
    bk, bp = _bias_args(bias, dense_bias)
    _check("jfa_bwd_ex", lib().jfa_bwd_ex(plan.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _dtype_code(O),
                                          _ptr(dO), _ptr(lse), bk, bp, scale, _ptr(dQ), _ptr(dK), _ptr(dV),
                                          _ptr(dbias), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream)))
    return dQ, dK, dV, dbias


def jfa_bwd_static_scratch(plan: Plan, Q, K, V, O, dO, lse, bias=None, scale=None, dQ=None, dK=None, dV=None,
                           stream=None):
    """jfa_bwd with the library's static scratch array in place of a workspace, for
    callers that cannot allocate device memory: pass dQ, dK and dV preallocated and
    this binding allocates nothing either.  Returns (dQ, dK, dV)."""
    dt = _dtype_code(Q)
    scale = 1.0 / float(plan.D) ** 0.5 if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    bk, bp = _bias_args(bias)
    _check("jfa_bwd_static_scratch", lib().jfa_bwd_static_scratch(
        plan.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _dtype_code(O), _ptr(dO), _ptr(lse), bk, bp, scale,
        _ptr(dQ), _ptr(dK), _ptr(dV), _stream(stream)))
    return dQ, dK, dV


def jfa_plan_device_status(plan: Plan, stream=None) -> int:
    return int(lib().jfa_plan_device_status(plan.handle, _stream(stream)))


KERNEL_KINDS = ["fwd", "bwd_pre", "bwd_main", "bwd_post", "bwd_dq"]


def jfa_plan_set_work_item(plan: Plan, pass_: int, index: int, item):
    """Test hook: overwrite work item `index` of pass 0 (forward), 1 (dK/dV), 2 (dQ), 3 (the
    short-query backward) or 4 (the short-query forward) with the four ints of `item` (see
    include/jfa.h)."""
    buf = np.ascontiguousarray(np.asarray(item, dtype=np.int32).reshape(4))
    _check("jfa_plan_set_work_item", lib().jfa_plan_set_work_item(plan.handle, int(pass_), int(index),
                                                                    buf.ctypes.data_as(ctypes.c_void_p)))


def jfa_plan_set_deterministic(plan: Plan, enable: bool = True):
    """enable: always the two-pass bf16 backward, the same bit for bit on every run; off
    (the default): the planner's choice, the fused backward on short sequences (whose dQ
    can differ in its last bit between runs), the two-pass one on long ones."""
    _check("jfa_plan_set_deterministic", lib().jfa_plan_set_deterministic(plan.handle, int(bool(enable))))


def jfa_plan_set_timing(plan: Plan, enable: bool = True):
    _check("jfa_plan_set_timing", lib().jfa_plan_set_timing(plan.handle, int(bool(enable))))


def jfa_plan_kernel_times(plan: Plan) -> dict:
    """{kind: (total_ms, launches)} since the previous query (synchronises)."""
    ms = (ctypes.c_double * len(KERNEL_KINDS))()
    n = (ctypes.c_int64 * len(KERNEL_KINDS))()
    _check("jfa_plan_kernel_times", lib().jfa_plan_kernel_times(plan.handle, ms, n))
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KERNEL_KINDS)}


def jfa_partition_sequences(q_offsets, kv_offsets, H: int, causal: bool, n_parts: int, window=None):
    """Host LPT split of a batch's sequences over n_parts GPUs.  Returns (part_of_seq int32 [B],
    part_cost int64 [n_parts])."""
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    B = qo.size - 1
    part = np.zeros(max(B, 1), dtype=np.int32)
    cost = np.zeros(int(n_parts), dtype=np.int64)
    _check("jfa_partition_sequences", lib().jfa_partition_sequences(
        qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p), int(B), int(H), int(bool(causal)),
        _win(window), int(n_parts), part.ctypes.data_as(ctypes.c_void_p), cost.ctypes.data_as(ctypes.c_void_p)))
    return part[:B], cost


def jfa_partition_users(q_offsets, kv_offsets, kv_index, H: int, causal: bool, n_parts: int, window=None):
    """Host LPT split of a shared key/value batch's users (with all their query sets) over
    n_parts GPUs.  Returns (part_of_user int32 [U], part_cost int64 [n_parts])."""
    qo, ko, ki = _i32(q_offsets), _i32(kv_offsets), _i32(kv_index)
    B, U = qo.size - 1, ko.size - 1
    part = np.zeros(max(U, 1), dtype=np.int32)
    cost = np.zeros(int(n_parts), dtype=np.int64)
    vp = ctypes.c_void_p
    _check("jfa_partition_users", lib().jfa_partition_users(
        qo.ctypes.data_as(vp), int(B), ko.ctypes.data_as(vp), int(U), ki.ctypes.data_as(vp), int(H),
        int(bool(causal)), _win(window), int(n_parts), part.ctypes.data_as(vp), cost.ctypes.data_as(vp)))
    return part[:U], cost


def shard(batch, rank: int, world: int):
    """The part of `batch` that rank `rank` of `world` processes (a workloads.Batch,
    repacked), by the LPT splits above: sequences, or for a shared key/value batch users
    with all their query sets.  The parts are independent, so their results are exactly
    the full batch's results for those sequences (users)."""
    from . import workloads
    if getattr(batch, "kv_map", None) is not None:
        part, _ = jfa_partition_users(batch.q_off, batch.kv_off, batch.kv_map, batch.H, batch.causal, world,
                                      window=getattr(batch, "window", None))
        return workloads.subset_users(batch, np.nonzero(part == rank)[0])
    part, _ = jfa_partition_sequences(batch.q_off, batch.kv_off, batch.H, batch.causal, world,
                                      window=getattr(batch, "window", None))
    seqs = np.nonzero(part == rank)[0]
    return workloads.subset(batch, seqs)


def jfa_worklist_size(q_offsets, kv_offsets, H: int, causal: bool, pass_: int, window=None) -> int:
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    n = ctypes.c_int64()
    _check("jfa_worklist_size", lib().jfa_worklist_size(qo.ctypes.data_as(ctypes.c_void_p),
                                                         ko.ctypes.data_as(ctypes.c_void_p), qo.size - 1, int(H),
                                                         int(bool(causal)), _win(window), int(pass_),
                                                         ctypes.byref(n)))
    return int(n.value)


def jfa_worklist_build(q_offsets, kv_offsets, H: int, causal: bool, pass_: int, n_ctas: int, window=None):
    """Host planner.  Returns (items int32 [n,4] (seq, head, tile, inner), cta_offsets [n_ctas+1],
    cta_cost [n_ctas])."""
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    n = jfa_worklist_size(qo, ko, H, causal, pass_, window)
    items = np.zeros((max(n, 1), 4), dtype=np.int32)
    offs = np.zeros(n_ctas + 1, dtype=np.int32)
    cost = np.zeros(n_ctas, dtype=np.int64)
    _check("jfa_worklist_build", lib().jfa_worklist_build(
        qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p), qo.size - 1, int(H),
        int(bool(causal)), _win(window), int(pass_), int(n_ctas), items.ctypes.data_as(ctypes.c_void_p),
        offs.ctypes.data_as(ctypes.c_void_p), cost.ctypes.data_as(ctypes.c_void_p)))
    return items[:n], offs, cost


# --------------------------------------------------------------------------- convenience


def plan_for(batch, stream=None, deterministic=False) -> Plan:
    """The plan of a workloads.Batch: shared key/value when it has a query-set-to-user map.
    deterministic: the two-pass backward (see jfa_plan_set_deterministic)."""
    if getattr(batch, "kv_map", None) is not None:
        plan = jfa_plan_create_shared_kv(batch.q_off, batch.kv_off, batch.kv_map, batch.H, batch.D, batch.mode,
                                         batch.causal, stream, window=getattr(batch, "window", None))
    else:
        plan = jfa_plan_create(batch.q_off, batch.kv_off, batch.H, batch.D, batch.mode, batch.causal, stream,
                               window=getattr(batch, "window", None))
    if deterministic:
        jfa_plan_set_deterministic(plan, True)
    return plan


class JaggedAttention(torch.autograd.Function):
    """The forward and backward passes as one torch.autograd function (argument marshalling
    only: both passes run in the library's kernels, on the current stream).

    Q [T_q, H, D], K, V [T_kv, H, D] (bf16 or fp32, contiguous); bias: the bucket table
    [H, 32], or with dense set the dense per-pair bias [H, P] (fp32), or None.  Returns O in
    Q's dtype.  The bias gradient is computed only when the bias requires one."""

    @staticmethod
    def forward(ctx, Q, K, V, bias, plan, scale, dense):
        O, lse = jfa_fwd(plan, Q, K, V, None if dense else bias, scale, dense_bias=bias if dense else None)
        ctx.plan, ctx.scale, ctx.dense = plan, scale, dense
        ctx.save_for_backward(Q, K, V, O, lse, bias)
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, lse, bias = ctx.saved_tensors
        dO = dO.to(Q.dtype).contiguous()
        table, dense = (None, bias) if ctx.dense else (bias, None)
        if bias is not None and ctx.needs_input_grad[3]:
            dQ, dK, dV, dbias = jfa_bwd_ex(ctx.plan, Q, K, V, O, dO, lse, table, ctx.scale, dense_bias=dense)
        else:
            (dQ, dK, dV), dbias = jfa_bwd(ctx.plan, Q, K, V, O, dO, lse, table, ctx.scale, dense_bias=dense), None
        return dQ, dK, dV, dbias, None, None, None


def jagged_attention(Q, K, V, q_offsets=None, kv_offsets=None, bias=None, mode="softmax", causal=False,
                     window=None, scale=None, plan=None, dense_bias=False, kv_index=None, deterministic=False):
    """Differentiable jagged attention.  Builds the plan from the offsets (kv_index: shared
    key/value, query set b attending to user kv_index[b]) unless one is given; a plan can be
    reused while the batch's shape is the same.  deterministic: a new plan runs the two-pass
    backward (see jfa_plan_set_deterministic).  See JaggedAttention for the tensors."""
    if plan is None:
        H, D = int(Q.shape[1]), int(Q.shape[2])
        if kv_index is not None:
            plan = jfa_plan_create_shared_kv(q_offsets, kv_offsets, kv_index, H, D, mode, causal, window=window)
        else:
            plan = jfa_plan_create(q_offsets, kv_offsets, H, D, mode, causal, window=window)
        if deterministic:
            jfa_plan_set_deterministic(plan, True)
    return JaggedAttention.apply(Q, K, V, bias, plan, scale, bool(dense_bias))


def attention(batch, with_backward=True, stream=None, out_dtype=None, bias_grad=False, deterministic=False):
    """Run forward (and backward) for a workloads.Batch on the GPU: returns dict of tensors
    (with bias_grad, also "dbias", the gradient of the batch's bias table).  deterministic:
    the two-pass backward (see jfa_plan_set_deterministic)."""
    plan = plan_for(batch, stream, deterministic)
    dense = getattr(batch, "dense", None)
    O, lse = jfa_fwd(plan, batch.Q, batch.K, batch.V, batch.bias, batch.scale, stream=stream, out_dtype=out_dtype,
                     dense_bias=dense)
    out = {"O": O, "lse": lse, "plan": plan}
    if with_backward and bias_grad:
        dQ, dK, dV, dbias = jfa_bwd_ex(plan, batch.Q, batch.K, batch.V, O, batch.dO, lse, batch.bias, batch.scale,
                                       stream=stream, dense_bias=dense)
        out.update(dQ=dQ, dK=dK, dV=dV, dbias=dbias)
    elif with_backward:
        dQ, dK, dV = jfa_bwd(plan, batch.Q, batch.K, batch.V, O, batch.dO, lse, batch.bias, batch.scale,
                             stream=stream, dense_bias=dense)
        out.update(dQ=dQ, dK=dK, dV=dV)
    return out
