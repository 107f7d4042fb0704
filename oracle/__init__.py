"""Oracle for jagged attention: plain fp64 CPU definition (see ``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The CUDA
library never loads it and shares no code with it.

Inputs are numpy arrays: values ``[T, H, D]`` (any float dtype; widened to fp64
exactly), offsets ``int32[B+1]``, bias table ``[H, 32]`` or ``None``, dense per-pair
bias ``[H, P]`` (``P = num_pairs(q_off, kv_off)``, sequence b's block row-major
``[q_len, kv_len]`` at ``pair_offsets(...)[b]``) or ``None``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SOFTMAX, GELU_TANH, SILU = 0, 1, 2
MODES = {"softmax": SOFTMAX, "gelu_tanh": GELU_TANH, "silu": SILU}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-D_DEFAULT_SOURCE", "-fopenmp", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER
            d, i32 = ctypes.c_double, ctypes.c_int32
            lib.oracle_relpos_bucket.argtypes = [ctypes.c_int64]
            lib.oracle_relpos_bucket.restype = ctypes.c_int
            lib.oracle_act.argtypes = [ctypes.c_int, d]
            lib.oracle_act.restype = d
            lib.oracle_act_grad.argtypes = [ctypes.c_int, d]
            lib.oracle_act_grad.restype = d
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_num_pairs.argtypes = [ctypes.c_int, P(i32), P(i32)]
            lib.oracle_num_pairs.restype = ctypes.c_int64
            common = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P(i32), P(i32)]
            lib.oracle_fwd.argtypes = common + [P(d)] * 3 + [ctypes.c_int, ctypes.c_int, ctypes.c_int, P(d), P(d), d,
                                                             P(d), P(d), ctypes.c_int]
            lib.oracle_fwd.restype = ctypes.c_int
            lib.oracle_bwd.argtypes = common + [P(d)] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.c_int, P(d), P(d), d,
                                                             P(d), P(d), P(d), P(d), P(d), ctypes.c_int]
            lib.oracle_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(q_off, kv_off, Q, K, V):
    q_off = np.ascontiguousarray(np.asarray(q_off, dtype=np.int32))
    kv_off = np.ascontiguousarray(np.asarray(kv_off, dtype=np.int32))
    if q_off.ndim != 1 or q_off.shape != kv_off.shape or q_off.size < 1:
        raise ValueError("offsets must be 1-D of equal length B+1")
    if np.any(np.diff(q_off) < 0) or np.any(np.diff(kv_off) < 0) or q_off[0] < 0 or kv_off[0] < 0:
        raise ValueError("offsets must be non-negative and non-decreasing")
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    if Q.ndim != 3 or K.shape != V.shape or K.ndim != 3 or Q.shape[1:] != K.shape[1:]:
        raise ValueError("Q [Tq,H,D], K and V [Tkv,H,D] expected")
    if Q.shape[0] < q_off[-1] or K.shape[0] < kv_off[-1]:
        raise ValueError("offsets exceed the value tensors")
    return q_off, kv_off, Q, K, V


def relpos_bucket(r: int) -> int:
    return int(_load().oracle_relpos_bucket(int(r)))


def act(mode: str, x: float) -> float:
    return float(_load().oracle_act(MODES[mode], float(x)))


def act_grad(mode: str, x: float) -> float:
    return float(_load().oracle_act_grad(MODES[mode], float(x)))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def pair_offsets(q_off, kv_off):
    """int64[B+1]: where each sequence's block of a dense per-pair array starts."""
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    out = np.zeros(q_off.size, dtype=np.int64)
    for b in range(q_off.size - 1):
        out[b + 1] = out[b] + (q_off[b + 1] - q_off[b]) * (kv_off[b + 1] - kv_off[b])
    return out


def num_pairs(q_off, kv_off) -> int:
    q_off = np.ascontiguousarray(np.asarray(q_off, dtype=np.int32))
    kv_off = np.ascontiguousarray(np.asarray(kv_off, dtype=np.int32))
    return int(_load().oracle_num_pairs(q_off.size - 1, _ptr(q_off, ctypes.c_int32), _ptr(kv_off, ctypes.c_int32)))


def _dense(dense, H, q_off, kv_off):
    if dense is None:
        return None
    d = _f64(dense)
    if d.shape != (H, num_pairs(q_off, kv_off)):
        raise ValueError("dense bias must be [H, P]")
    return d


def fwd(q_off, kv_off, Q, K, V, *, mode="softmax", causal=False, bias=None, scale=None,
        nthreads=0, window=None, dense_bias=None):
    """Returns (O [Tq,H,D] fp64, LSE [Tq,H] fp64).  window W (None: no window): key j is
    allowed for query i only if j >= i + (kv_len - q_len) - W.  dense_bias [H, P]: a
    per-pair additive bias (None: none)."""
    lib = _load()
    q_off, kv_off, Q, K, V = _check(q_off, kv_off, Q, K, V)
    B = q_off.size - 1
    _, H, D = Q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    b = None if bias is None else _f64(bias).reshape(H, 32)
    dn = _dense(dense_bias, H, q_off, kv_off)
    O = np.zeros_like(Q)
    LSE = np.zeros((Q.shape[0], H), dtype=np.float64)
    rc = lib.oracle_fwd(B, H, D, _ptr(q_off, ctypes.c_int32), _ptr(kv_off, ctypes.c_int32),
                        _ptr(Q), _ptr(K), _ptr(V), MODES[mode], int(bool(causal)),
                        -1 if window is None else int(window),
                        None if b is None else _ptr(b), None if dn is None else _ptr(dn), scale, _ptr(O),
                        _ptr(LSE), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle_fwd failed")
    return O, LSE


def bwd(q_off, kv_off, Q, K, V, dO, *, mode="softmax", causal=False, bias=None, scale=None,
        nthreads=0, window=None, dense_bias=None, bias_grads=False, dense_grad=True):
    """Returns (dQ, dK, dV), fp64, same shapes as Q, K, V; with bias_grads also the
    gradient of the bucket table [H, 32] and of a dense per-pair bias [H, P] (both are
    defined whether or not that bias was given: the gradient of the score).  With
    dense_grad=False the dense gradient is not formed (returned as None)."""
    lib = _load()
    q_off, kv_off, Q, K, V = _check(q_off, kv_off, Q, K, V)
    dO = _f64(dO)
    if dO.shape != Q.shape:
        raise ValueError("dO must match Q")
    B = q_off.size - 1
    _, H, D = Q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    b = None if bias is None else _f64(bias).reshape(H, 32)
    dn = _dense(dense_bias, H, q_off, kv_off)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dbias = np.zeros((H, 32)) if bias_grads else None
    d_dense = np.zeros((H, num_pairs(q_off, kv_off))) if bias_grads and dense_grad else None
    rc = lib.oracle_bwd(B, H, D, _ptr(q_off, ctypes.c_int32), _ptr(kv_off, ctypes.c_int32),
                        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), MODES[mode], int(bool(causal)),
                        -1 if window is None else int(window),
                        None if b is None else _ptr(b), None if dn is None else _ptr(dn), scale, _ptr(dQ),
                        _ptr(dK), _ptr(dV), None if dbias is None else _ptr(dbias),
                        None if d_dense is None else _ptr(d_dense), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle_bwd failed")
    if bias_grads:
        return dQ, dK, dV, dbias, d_dense
    return dQ, dK, dV


# --------------------------------------------------------------------------- shared key/value
# In-kernel broadcast (IKBO, PyTorch blog "In-Kernel Broadcast Optimization: Co-Designing
# Kernels for RecSys Inference", section 3 "IKBO Flash Attention" and figure 1): many
# candidate query sets of one request attend to the same user's key/value history.  The
# operation is exactly attention over the broadcast (copied) history; the kernel only avoids
# materialising the copies.  So the oracle is that definition: gather each query set's user
# rows, attend as above, and (backward of a broadcast) sum the key/value gradients of all
# query sets that share a user.


def _broadcast(kv_off_users, kv_index, K, V):
    """Per query set b, the rows of user kv_index[b]: (kv_off of the copies, row index)."""
    kv_off_users = np.asarray(kv_off_users, dtype=np.int64)
    kv_index = np.asarray(kv_index, dtype=np.int64)
    lens = kv_off_users[kv_index + 1] - kv_off_users[kv_index]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = np.concatenate([np.arange(kv_off_users[u], kv_off_users[u + 1]) for u in kv_index]
                          + [np.zeros(0, dtype=np.int64)]).astype(np.int64)
    return off, rows


def shared_kv_fwd(q_off, kv_off_users, kv_index, Q, K, V, **kw):
    """Forward with query set b attending to user kv_index[b]'s rows kv_off_users[u] ..
    kv_off_users[u+1] of K and V.  Same keywords and results as fwd (the dense bias, if
    any, is laid out over the pairs of the query sets with their users' lengths)."""
    off, rows = _broadcast(kv_off_users, kv_index, K, V)
    K, V = _f64(K), _f64(V)
    return fwd(q_off, off, Q, K[rows], V[rows], **kw)


def shared_kv_bwd(q_off, kv_off_users, kv_index, Q, K, V, dO, **kw):
    """Backward of shared_kv_fwd: (dQ, dK, dV[, bias gradients]) with dK, dV over the
    users' rows, each the sum over the query sets that share the user."""
    off, rows = _broadcast(kv_off_users, kv_index, K, V)
    K, V = _f64(K), _f64(V)
    res = bwd(q_off, off, Q, K[rows], V[rows], dO, **kw)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    np.add.at(dK, rows, res[1])
    np.add.at(dV, rows, res[2])
    return (res[0], dK, dV) + tuple(res[3:])

