"""Helpers for parity tests: run the CUDA path through the C-ABI binding and the CPU
oracle on the same seeded inputs, and measure the differences.

Tolerances (stated for this path: bf16 inputs, fp32 accumulation):
  forward O:  max-abs <= 1e-2 and relative Frobenius <= 5e-3
  dQ, dK, dV: relative Frobenius <= 1e-2
  lse:        max-abs <= 2e-3 (fp32 softmax statistics; derived from the fp32
              accumulation of bf16-exact products, far inside this bound)
When O is written in bf16 rather than fp32, its final round-to-nearest adds up to
half an ulp, at most 2^-8 |o|, that no bf16 output can avoid; the max-abs bound
then applies to the error beyond that rounding: |o - ref| <= 1e-2 + 2^-8 |ref|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from jagged_sequence_attention_gb300 import workloads as wl

FWD_MAX_ABS = 1e-2
FWD_REL_FROB = 5e-3
BWD_REL_FROB = 1e-2
LSE_MAX_ABS = 2e-3


def np64(t):
    if t is None:
        return None
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def rel_frob(got, ref):
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return float(num / den) if den > 0 else float(num)


def max_abs(got, ref):
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def run_gpu(batch, with_backward=True, out_dtype=torch.float32, deterministic=False):
    """The batch through the C-ABI (deterministic: the two-pass bf16 backward, whatever the
    planner would choose)."""
    from jagged_sequence_attention_gb300 import jfa
    out = jfa.attention(batch, with_backward=with_backward, out_dtype=out_dtype, deterministic=deterministic)
    torch.cuda.synchronize()
    status = jfa.jfa_plan_device_status(out["plan"])
    out["status"] = status
    return out


def run_oracle(batch, with_backward=True, bias_grads=False):
    """Oracle on a (CPU-copied) batch: dict of fp64 numpy arrays (with bias_grads also
    "dbias", the gradient of the bias table)."""
    b = None if batch.bias is None else np64(batch.bias)
    Q, K, V = np64(batch.Q), np64(batch.K), np64(batch.V)
    Tq, Tkv = int(batch.q_off[-1]), int(batch.kv_off[-1])
    Q, K, V = Q[:Tq], K[:Tkv], V[:Tkv]
    dn = None if getattr(batch, "dense", None) is None else np64(batch.dense)
    kv_map = getattr(batch, "kv_map", None)
    if kv_map is None:
        fwd, bwd = oracle.fwd, oracle.bwd
    else:  # shared key/value: the broadcast definition
        def fwd(q_off, kv_off, *a, **k):
            return oracle.shared_kv_fwd(q_off, kv_off, kv_map, *a, **k)

        def bwd(q_off, kv_off, *a, **k):
            return oracle.shared_kv_bwd(q_off, kv_off, kv_map, *a, **k)
    O, LSE = fwd(batch.q_off, batch.kv_off, Q, K, V, mode=batch.mode, causal=batch.causal,
                 bias=b, scale=batch.scale, window=batch.window, dense_bias=dn)
    res = {"O": O, "lse": LSE}
    if with_backward:
        dO = np64(batch.dO)[:Tq]
        g = bwd(batch.q_off, batch.kv_off, Q, K, V, dO, mode=batch.mode, causal=batch.causal, bias=b,
                scale=batch.scale, window=batch.window, bias_grads=bias_grads, dense_grad=dn is not None,
                dense_bias=dn)
        res.update(dQ=g[0], dK=g[1], dV=g[2])
        if bias_grads:
            res["dbias"] = g[3] if dn is None else g[4]
    return res


def compare(gpu, ref, softmax=True, with_backward=True, rows_q=None, rows_kv=None):
    """Error metrics of GPU outputs against oracle outputs (optionally restricted to row
    index arrays of the GPU tensors, mapped onto the oracle's rows in order)."""
    def pick(t, rows):
        a = np64(t)
        return a if rows is None else a[rows]
    m = {}
    O = pick(gpu["O"], rows_q)
    m["O_max_abs"] = max_abs(O, ref["O"])
    m["O_rel_frob"] = rel_frob(O, ref["O"])
    m["O_bf16"] = gpu["O"].dtype == torch.bfloat16
    m["O_max_abs_beyond_rounding"] = beyond_rounding(O, ref["O"])
    if softmax:
        lse = pick(gpu["lse"], rows_q)
        fin = np.isfinite(ref["lse"])
        m["lse_nonfinite_match"] = bool(np.array_equal(fin, np.isfinite(lse)))
        m["lse_max_abs"] = max_abs(lse[fin], ref["lse"][fin]) if fin.any() else 0.0
    if with_backward:
        m["dQ_rel_frob"] = rel_frob(pick(gpu["dQ"], rows_q), ref["dQ"])
        if "dK" in ref:
            m["dK_rel_frob"] = rel_frob(pick(gpu["dK"], rows_kv), ref["dK"])
            m["dV_rel_frob"] = rel_frob(pick(gpu["dV"], rows_kv), ref["dV"])
    return m


def beyond_rounding(got, ref):
    """Largest |got - ref| - 2^-8 |ref|: the error beyond a bf16 output's own rounding."""
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) - np.abs(ref) * 2.0 ** -8))


def assert_within(m, softmax=True):
    if m.get("O_bf16"):
        assert m["O_max_abs_beyond_rounding"] <= FWD_MAX_ABS, m
    else:
        assert m["O_max_abs"] <= FWD_MAX_ABS, m
    assert m["O_rel_frob"] <= FWD_REL_FROB, m
    if softmax:
        assert m["lse_nonfinite_match"], m
        assert m["lse_max_abs"] <= LSE_MAX_ABS, m
    for k in ("dQ_rel_frob", "dK_rel_frob", "dV_rel_frob"):
        if k in m:
            assert m[k] <= BWD_REL_FROB, m


def suffix_problem(batch, b, h, i0):
    """Exact sub-problem for query rows [i0, q_len) of sequence b, head h, over all of
    its keys.  With bottom-right causal alignment (and a sliding window, which is relative
    to the same aligned position) and |i + kv_len - q_len - j| bias positions, these rows'
    outputs and dQ are unchanged; for causal attention the keys
    j >= i0 + (kv_len - q_len) also keep their exact dK, dV (no earlier row sees them),
    and for non-causal attention that holds when i0 == 0.
    Returns (sub_batch, q_rows, kv_rows): GPU row indices ([T,...] first axis, head h)
    the sub-problem's rows correspond to."""
    q0, q1 = int(batch.q_off[b]), int(batch.q_off[b + 1])
    k0, k1 = int(batch.kv_off[b]), int(batch.kv_off[b + 1])
    q_len, kv_len = q1 - q0, k1 - k0
    i0 = max(0, min(i0, q_len))
    qs = slice(q0 + i0, q1)
    ks = slice(k0, k1)
    take = lambda t, s: None if t is None else t[s, h:h + 1].contiguous().cpu()  # noqa: E731
    sub = wl.Batch(batch.name + f"/seq{b}/h{h}/rows{i0}:", wl.offsets([q_len - i0]), wl.offsets([kv_len]),
                   take(batch.Q, qs), take(batch.K, ks), take(batch.V, ks), take(batch.dO, qs),
                   None if batch.bias is None else batch.bias[h:h + 1].cpu(), batch.scale, batch.mode,
                   batch.causal, 1, batch.D, window=batch.window)
    if batch.causal:
        j0 = max(0, i0 + (kv_len - q_len))
    else:
        j0 = 0 if i0 == 0 else kv_len
    q_rows = np.arange(q0 + i0, q1)
    kv_rows = np.arange(k0 + j0, k1)
    return sub, q_rows, kv_rows, j0


def _concat_batches(subs):
    """Several one-head jagged problems (same head) as one batch, so the oracle runs them
    in parallel."""
    cat = lambda xs: None if xs[0] is None else torch.cat(xs)  # noqa: E731
    q_l = [int(s.q_off[-1]) for s in subs]
    k_l = [int(s.kv_off[-1]) for s in subs]
    s0 = subs[0]
    return wl.Batch(s0.name, wl.offsets(q_l), wl.offsets(k_l), cat([s.Q for s in subs]), cat([s.K for s in subs]),
                    cat([s.V for s in subs]), cat([s.dO for s in subs]), s0.bias, s0.scale, s0.mode, s0.causal, 1,
                    s0.D, window=s0.window)


def sampled_parity(batch, gpu, samples, with_backward=True):
    """Compare GPU outputs of a full batch with the oracle on suffix sub-problems
    [(seq, head, i0), ...]; returns the metrics over the concatenated sample."""
    softmax = batch.mode == "softmax"
    got = {k: [] for k in ("O", "lse", "dQ", "dK", "dV")}
    ref = {k: [] for k in ("O", "lse", "dQ", "dK", "dV")}
    heads = sorted(set(h for (_, h, _) in samples))
    for h in heads:
        group = [(b, hh, i0) for (b, hh, i0) in samples if hh == h]
        subs = [suffix_problem(batch, b, h, i0) for (b, _, i0) in group]
        r = run_oracle(_concat_batches([s[0] for s in subs]), with_backward)
        qo = wl.offsets([int(s[0].q_off[-1]) for s in subs])
        ko = wl.offsets([int(s[0].kv_off[-1]) for s in subs])
        for k, (sub, q_rows, kv_rows, j0) in enumerate(subs):
            qs, ks = slice(int(qo[k]), int(qo[k + 1])), slice(int(ko[k]) + j0, int(ko[k + 1]))
            qi, ki = torch.as_tensor(q_rows), torch.as_tensor(kv_rows)
            got["O"].append(np64(gpu["O"][qi, h]))
            ref["O"].append(r["O"][qs, 0])
            if softmax:
                got["lse"].append(np64(gpu["lse"][qi, h]))
                ref["lse"].append(r["lse"][qs, 0])
            if with_backward:
                got["dQ"].append(np64(gpu["dQ"][qi, h]))
                ref["dQ"].append(r["dQ"][qs, 0])
                got["dK"].append(np64(gpu["dK"][ki, h]))
                ref["dK"].append(r["dK"][ks, 0])
                got["dV"].append(np64(gpu["dV"][ki, h]))
                ref["dV"].append(r["dV"][ks, 0])
    cat = lambda xs: np.concatenate(xs) if xs else np.zeros(0)  # noqa: E731
    m = {"O_max_abs": max_abs(cat(got["O"]), cat(ref["O"])),
         "O_rel_frob": rel_frob(cat(got["O"]), cat(ref["O"])),
         "O_bf16": gpu["O"].dtype == torch.bfloat16,
         "O_max_abs_beyond_rounding": beyond_rounding(cat(got["O"]), cat(ref["O"]))}
    if softmax:
        g, rr = cat(got["lse"]), cat(ref["lse"])
        fin = np.isfinite(rr)
        m["lse_nonfinite_match"] = bool(np.array_equal(fin, np.isfinite(g)))
        m["lse_max_abs"] = max_abs(g[fin], rr[fin]) if fin.any() else 0.0
    if with_backward:
        for k in ("dQ", "dK", "dV"):
            m[f"{k}_rel_frob"] = rel_frob(cat(got[k]), cat(ref[k]))
    return m


def causal_row_blocks(L, n):
    """Boundaries 0 = i_0 < ... < i_n = L giving blocks of about equal causal cost (a
    row i costs about i + 1 keys, so block k ends near L sqrt(k / n))."""
    cuts = sorted(set([0, L] + [int(round(L * np.sqrt(k / n))) for k in range(1, n)]))
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def causal_head_oracle(Q, K, V, dO, bias_h, scale, n_blocks=48):
    """Oracle O, lse, dQ, dK, dV ([L, D] / [L]) of one causal self-attention head given as
    fp64 [L, D] arrays, computed block by block so that the oracle, which parallelises
    over (sequence, head) problems, uses every core on one long sequence.

    The split is exact.  In causal self-attention (q_len = kv_len), rows [i0, i1) see
    only keys [0, i1).  As a sub-problem with q_len' = i1 - i0 and kv_len' = i1, the
    bottom-right alignment puts local row r at position r + i0, so it sees the same
    keys, at the same relative positions, as global row i0 + r: O, lse and dQ of the
    block's rows come out exactly, and dK, dV (sums over rows) are the sums of the
    blocks' contributions."""
    L, D = Q.shape
    blocks = causal_row_blocks(L, n_blocks)
    q_off = wl.offsets([b - a for a, b in blocks])
    kv_off = wl.offsets([b for _, b in blocks])
    cat = lambda X, sl: np.concatenate([X[s] for s in sl])[:, None, :]  # noqa: E731
    rows = [slice(a, b) for a, b in blocks]
    keys = [slice(0, b) for _, b in blocks]
    Qc, dOc, Kc, Vc = cat(Q, rows), cat(dO, rows), cat(K, keys), cat(V, keys)
    O, LSE = oracle.fwd(q_off, kv_off, Qc, Kc, Vc, causal=True, bias=bias_h, scale=scale)
    dQ, dKc, dVc = oracle.bwd(q_off, kv_off, Qc, Kc, Vc, dOc, causal=True, bias=bias_h, scale=scale)
    dK = np.zeros((L, D))
    dV = np.zeros((L, D))
    for k, (_, b) in enumerate(blocks):
        dK[:b] += dKc[kv_off[k]:kv_off[k + 1], 0]
        dV[:b] += dVc[kv_off[k]:kv_off[k + 1], 0]
    return {"O": O[:, 0], "lse": LSE[:, 0], "dQ": dQ[:, 0], "dK": dK, "dV": dV}
