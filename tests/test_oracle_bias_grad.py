"""Pins for the oracle's bias gradients and its dense per-pair bias.

The bias is the article's "custom attention bias" (aihot.vn GEM article, section
"Jagged Sequence Flash Attention").  Its gradient is that of the score it adds to,
so the gradient of the 32-bucket table is the bucket-wise sum of dS and that of a
dense per-pair bias is dS itself.

Each test checks the oracle against something other than itself:
- autograd in fp64 through SDPA, or through the explicit GDPA formula, with the bias
  as a leaf tensor (the library routine on a special case);
- central finite differences;
- the closed form that a softmax row's dS sums to zero (sum_j p_ij (dp_ij - sum_k
  p_ik dp_ik) = 0), so every head's table gradient sums to zero;
- the identity that a dense bias expanded from the table changes nothing;
- the relation dQ = scale dS K, which ties the dense gradient to dQ (itself pinned
  by autograd in test_oracle)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from jagged_sequence_attention_gb300 import workloads as wl

torch.set_default_dtype(torch.float64)


def bucket_ref(r: int) -> int:
    return min(31, ((1 + abs(int(r))) ** 2).bit_length() - 1)


def make(q_lens, kv_lens, H, D, seed, std=0.8):
    g = torch.Generator().manual_seed(seed)
    q_off, kv_off = wl.offsets(q_lens), wl.offsets(kv_lens)
    Q = torch.randn(int(q_off[-1]), H, D, generator=g) * std
    K = torch.randn(int(kv_off[-1]), H, D, generator=g) * std
    V = torch.randn(int(kv_off[-1]), H, D, generator=g)
    dO = torch.randn(int(q_off[-1]), H, D, generator=g)
    table = torch.randn(H, 32, generator=g) * 0.5
    P = sum(a * b for a, b in zip(q_lens, kv_lens))
    dense = torch.randn(H, P, generator=g) * 0.5
    return q_off, kv_off, Q, K, V, dO, table, dense


def autograd_reference(q_off, kv_off, Q, K, V, dO, table, dense, mode, causal, window, scale):
    """Per sequence: scores with the table (gathered by bucket) and the dense block as
    leaf tensors, SDPA (softmax) or act(S) V (GDPA), loss sum(O * dO); returns O and the
    gradients of the table and of the dense bias."""
    H = Q.shape[1]
    table = table.clone().requires_grad_(True)
    dense = dense.clone().requires_grad_(True)
    outs, pb = [], 0
    for b in range(len(q_off) - 1):
        qs, qe, ks, ke = int(q_off[b]), int(q_off[b + 1]), int(kv_off[b]), int(kv_off[b + 1])
        Lq, Lk = qe - qs, ke - ks
        if Lq == 0 or Lk == 0:
            pb += Lq * Lk
            outs.append(torch.zeros(Lq, H, Q.shape[2]))
            continue
        ip = torch.arange(Lq)[:, None] + (Lk - Lq)
        j = torch.arange(Lk)[None, :]
        allowed = torch.ones(Lq, Lk, dtype=torch.bool)
        if causal:
            allowed &= j <= ip
        if window is not None:
            allowed &= j >= ip - window
        idx = torch.tensor([[bucket_ref(int(r)) for r in row] for row in (ip - j).tolist()], dtype=torch.long)
        add = table[:, idx] + dense[:, pb:pb + Lq * Lk].reshape(H, Lq, Lk)
        pb += Lq * Lk
        q, k, v = (t.permute(1, 0, 2) for t in (Q[qs:qe], K[ks:ke], V[ks:ke]))
        row_has = allowed.any(dim=1)
        if mode == "softmax":
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=add.masked_fill(~allowed, float("-inf")), scale=scale)
            o = torch.where(row_has[None, :, None], o, torch.zeros_like(o))
        else:
            s = scale * q @ k.transpose(-1, -2) + add
            a = (F.gelu(s, approximate="tanh") if mode == "gelu_tanh" else F.silu(s)).masked_fill(~allowed, 0.0)
            o = a @ v
        outs.append(o.permute(1, 0, 2))
    O = torch.cat(outs)
    (O * dO).sum().backward()
    return O.detach(), table.grad, dense.grad


def run_oracle(q_off, kv_off, Q, K, V, dO, table, dense, mode, causal, window, scale):
    kw = dict(mode=mode, causal=causal, bias=None if table is None else table.numpy(),
              dense_bias=None if dense is None else dense.numpy(), scale=scale, window=window)
    O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), **kw)
    dQ, dK, dV, dtab, ddense = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(),
                                          bias_grads=True, **kw)
    return O, dQ, dK, dV, dtab, ddense


CASES = [
    # q_lens, kv_lens, causal, window
    ([1, 17, 40, 9, 0, 33], [1, 17, 55, 4, 3, 33], True, None),   # q > kv rows with no key, an empty sequence
    ([5, 30, 12], [40, 7, 12], False, None),
    ([20, 64, 3], [20, 70, 3], True, 6),
]


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_bias_gradients_match_autograd(mode, case):
    q, kv, causal, window = CASES[case]
    args = make(q, kv, H=2, D=8, seed=40 + case)
    scale = 0.45
    O, _, _, _, dtab, ddense = run_oracle(*args, mode, causal, window, scale)
    O_ref, dtab_ref, ddense_ref = autograd_reference(*args, mode, causal, window, scale)
    assert np.allclose(O, O_ref.numpy(), atol=1e-12, rtol=1e-10)
    assert np.allclose(dtab, dtab_ref.numpy(), atol=1e-11, rtol=1e-10), float(np.abs(dtab - dtab_ref.numpy()).max())
    assert np.allclose(ddense, ddense_ref.numpy(), atol=1e-12, rtol=1e-10)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_softmax_table_gradient_sums_to_zero_per_head(case):
    q, kv, causal, window = CASES[case]
    args = make(q, kv, H=3, D=8, seed=50 + case)
    _, _, _, _, dtab, ddense = run_oracle(*args, "softmax", causal, window, 0.4)
    assert np.abs(dtab).max() > 1e-3           # not trivially zero
    assert np.allclose(dtab.sum(axis=1), 0.0, atol=1e-12)
    # row by row: each query row's dS sums to zero
    pb = 0
    for a, b in zip(q, kv):
        blk = ddense[:, pb:pb + a * b].reshape(3, a, b)
        assert np.allclose(blk.sum(axis=2), 0.0, atol=1e-12)
        pb += a * b


def test_dense_bias_expanded_from_the_table_changes_nothing():
    q, kv = [9, 30, 4], [12, 30, 4]
    q_off, kv_off, Q, K, V, dO, table, _ = make(q, kv, H=2, D=8, seed=61)
    blocks = []
    for a, b in zip(q, kv):
        r = (np.arange(a)[:, None] + (b - a)) - np.arange(b)[None, :]
        idx = np.vectorize(bucket_ref)(r)
        blocks.append(table.numpy()[:, idx].reshape(2, a * b))
    dense = torch.from_numpy(np.concatenate(blocks, axis=1))
    for mode in ("softmax", "silu"):
        with_table = run_oracle(q_off, kv_off, Q, K, V, dO, table, None, mode, True, None, 0.3)
        with_dense = run_oracle(q_off, kv_off, Q, K, V, dO, None, dense, mode, True, None, 0.3)
        for x, y in zip(with_table[:4], with_dense[:4]):
            assert np.allclose(x, y, atol=1e-13, rtol=1e-12)
        # the table's gradient is the bucket-wise sum of the dense gradient
        dt = np.zeros((2, 32))
        pb = 0
        for a, b in zip(q, kv):
            r = (np.arange(a)[:, None] + (b - a)) - np.arange(b)[None, :]
            idx = np.vectorize(bucket_ref)(r).reshape(-1)
            for h in range(2):
                np.add.at(dt[h], idx, with_dense[5][h, pb:pb + a * b])
            pb += a * b
        assert np.allclose(dt, with_table[4], atol=1e-12)


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh"])
def test_dense_gradient_reproduces_dq(mode):
    q, kv = [7, 25], [11, 25]
    q_off, kv_off, Q, K, V, dO, table, dense = make(q, kv, H=2, D=6, seed=70)
    scale = 0.5
    _, dQ, _, _, _, ddense = run_oracle(q_off, kv_off, Q, K, V, dO, table, dense, mode, True, None, scale)
    pb = 0
    for b, (a, c) in enumerate(zip(q, kv)):
        qs, ks = int(q_off[b]), int(kv_off[b])
        for h in range(2):
            dS = ddense[h, pb:pb + a * c].reshape(a, c)
            want = scale * dS @ K.numpy()[ks:ks + c, h, :]
            assert np.allclose(dQ[qs:qs + a, h, :], want, atol=1e-12)
        pb += a * c


@pytest.mark.parametrize("mode", ["softmax", "silu"])
def test_bias_gradients_match_finite_differences(mode):
    q, kv = [5, 6], [5, 8]
    q_off, kv_off, Q, K, V, dO, table, dense = make(q, kv, H=1, D=3, seed=80)
    scale, h = 0.6, 1e-6
    _, _, _, _, dtab, ddense = run_oracle(q_off, kv_off, Q, K, V, dO, table, dense, mode, True, 3, scale)

    def loss(t, d):
        O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), mode=mode, causal=True, bias=t,
                          dense_bias=d, scale=scale, window=3)
        return float((O * dO.numpy()).sum())

    t0, d0 = table.numpy().copy(), dense.numpy().copy()
    for k in range(8):                      # the buckets relative positions 0..6 reach
        tp, tm = t0.copy(), t0.copy()
        tp[0, k] += h
        tm[0, k] -= h
        assert abs((loss(tp, d0) - loss(tm, d0)) / (2 * h) - dtab[0, k]) < 1e-7, k
    assert np.all(dtab[0, 8:] == 0)          # no allowed pair reaches bucket 8 with W = 3
    for e in range(d0.shape[1]):
        dp, dm = d0.copy(), d0.copy()
        dp[0, e] += h
        dm[0, e] -= h
        assert abs((loss(t0, dp) - loss(t0, dm)) / (2 * h) - ddense[0, e]) < 1e-7, e


def test_pair_offsets_and_count():
    q, kv = [3, 0, 5, 2], [4, 6, 5, 0]
    qo, ko = wl.offsets(q), wl.offsets(kv)
    assert oracle.num_pairs(qo, ko) == 3 * 4 + 0 + 25 + 0
    assert list(oracle.pair_offsets(qo, ko)) == [0, 12, 12, 37, 37]
