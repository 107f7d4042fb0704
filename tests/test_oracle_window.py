"""Pins for the oracle's sliding window (aihot.vn GEM article, section "BlockAttention":
each token attends only to its neighbouring events).  Reading: with window W, query i
sees keys j with i' - W <= j <= i', where i' = i + (kv_len - q_len) is the query's aligned
key position (the causal bound), i.e. itself and the W keys before it.

Each test checks the oracle against something other than itself: a library routine on a
special case (SDPA with an explicit band mask, gradients from autograd), a closed form
(W = 0 leaves one key per row), an identity (a window as long as the sequence changes
nothing) and finite differences."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from jagged_sequence_attention_gb300 import workloads as wl

torch.set_default_dtype(torch.float64)


def bucket_ref(r: int) -> int:
    return min(31, ((1 + abs(r)) ** 2).bit_length() - 1)


def batch(q_lens, kv_lens, H, D, seed, bias=True, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q_off, kv_off = wl.offsets(q_lens), wl.offsets(kv_lens)
    Q = torch.randn(int(q_off[-1]), H, D, generator=g) * std
    K = torch.randn(int(kv_off[-1]), H, D, generator=g) * std
    V = torch.randn(int(kv_off[-1]), H, D, generator=g)
    dO = torch.randn(int(q_off[-1]), H, D, generator=g)
    b = torch.randn(H, 32, generator=g) * 0.5 if bias else None
    return q_off, kv_off, Q, K, V, dO, b


def band_reference(q_off, kv_off, Q, K, V, dO, bias, window, mode, scale):
    """Per sequence: SDPA (softmax) or matmul-act-matmul (GDPA) in fp64 over an explicit
    [Lq, Lk] mask that allows i' - W <= j <= i'; gradients by autograd."""
    H = Q.shape[1]
    O, LSE = torch.zeros_like(Q), torch.zeros(Q.shape[0], H)
    dQ, dK, dV = torch.zeros_like(Q), torch.zeros_like(K), torch.zeros_like(V)
    for b in range(len(q_off) - 1):
        qs, qe, ks, ke = int(q_off[b]), int(q_off[b + 1]), int(kv_off[b]), int(kv_off[b + 1])
        Lq, Lk = qe - qs, ke - ks
        if Lq == 0:
            continue
        ip = torch.arange(Lq)[:, None] + (Lk - Lq)
        j = torch.arange(Lk)[None, :]
        allowed = (j <= ip) & (j >= ip - window)
        add = torch.zeros(H, Lq, Lk)
        if bias is not None:
            idx = torch.tensor([[bucket_ref(int(r)) for r in row] for row in (ip - j).tolist()],
                               dtype=torch.long).reshape(Lq, Lk)
            add = add + bias[:, idx]
        q = Q[qs:qe].permute(1, 0, 2).clone().requires_grad_(True)
        k = K[ks:ke].permute(1, 0, 2).clone().requires_grad_(True)
        v = V[ks:ke].permute(1, 0, 2).clone().requires_grad_(True)
        row_has = allowed.any(dim=1)
        if mode == "softmax":
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=add.masked_fill(~allowed, float("-inf")), scale=scale)
            o = torch.where(row_has[None, :, None], o, torch.zeros_like(o))
            lse = torch.logsumexp((scale * q @ k.transpose(-1, -2) + add).masked_fill(~allowed, float("-inf")), dim=-1)
        else:
            s = scale * q @ k.transpose(-1, -2) + add
            a = (F.gelu(s, approximate="tanh") if mode == "gelu_tanh" else F.silu(s)).masked_fill(~allowed, 0.0)
            o = a @ v
            lse = torch.zeros(H, Lq)
        O[qs:qe] = o.detach().permute(1, 0, 2)
        LSE[qs:qe] = lse.detach().T
        if Lk > 0:
            (o * dO[qs:qe].permute(1, 0, 2)).sum().backward()
            dQ[qs:qe], dK[ks:ke], dV[ks:ke] = (t.grad.permute(1, 0, 2) for t in (q, k, v))
    return O, LSE, dQ, dK, dV


def run(q_off, kv_off, Q, K, V, dO, bias, window, mode, scale, causal=True):
    b = None if bias is None else bias.numpy()
    O, LSE = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), mode=mode, causal=causal,
                        bias=b, scale=scale, window=window)
    dQ, dK, dV = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), mode=mode,
                            causal=causal, bias=b, scale=scale, window=window)
    return [torch.from_numpy(x) for x in (O, LSE, dQ, dK, dV)]


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("window", [0, 1, 5, 37])
def test_window_matches_sdpa_with_a_band_mask(mode, window):
    q, kv = [1, 17, 40, 9, 0, 64], [1, 17, 55, 4, 3, 64]   # q > kv leaves rows with no key
    args = batch(q, kv, H=2, D=8, seed=11 + window, std=0.7)
    scale = 0.4
    got = run(*args, window, mode, scale)
    want = band_reference(*args, window, mode, scale)
    for name, g, w in zip(("O", "LSE", "dQ", "dK", "dV"), got, want):
        if name == "LSE":
            fin = torch.isfinite(w)
            assert torch.equal(fin, torch.isfinite(g)), name
            g, w = g[fin], w[fin]
        assert torch.allclose(g, w, atol=1e-12, rtol=1e-10), (name, float((g - w).abs().max()))


def test_window_zero_leaves_one_key_per_row():
    """W = 0: row i sees only key i' = i + kv_len - q_len, so (softmax) o_i = v_i', lse_i =
    s_ii', dQ = dK = 0 (ds = p (dp - p dp) = 0 with p = 1), and dV_j sums dO over the rows
    aligned to key j."""
    q, kv = [5, 12, 3], [5, 15, 1]
    q_off, kv_off, Q, K, V, dO, bias = batch(q, kv, H=3, D=4, seed=3)
    scale = 0.3
    O, LSE, dQ, dK, dV = run(q_off, kv_off, Q, K, V, dO, bias, 0, "softmax", scale)
    for b in range(len(q)):
        for i in range(q[b]):
            ip = i + kv[b] - q[b]
            row = int(q_off[b]) + i
            if ip < 0:
                assert torch.all(O[row] == 0) and torch.all(torch.isinf(LSE[row]))
                continue
            key = int(kv_off[b]) + ip
            assert torch.equal(O[row], V[key])
            s = scale * (Q[row] * K[key]).sum(-1) + bias[:, bucket_ref(0)]
            assert torch.allclose(LSE[row], s, atol=1e-13)
    assert torch.all(dQ == 0) and torch.all(dK == 0)
    want_dV = torch.zeros_like(V)
    for b in range(len(q)):
        for i in range(q[b]):
            ip = i + kv[b] - q[b]
            if ip >= 0:
                want_dV[int(kv_off[b]) + ip] += dO[int(q_off[b]) + i]
    assert torch.allclose(dV, want_dV, atol=1e-13)


@pytest.mark.parametrize("mode", ["softmax", "silu"])
def test_window_as_long_as_the_keys_changes_nothing(mode):
    q, kv = [30, 7, 64], [30, 20, 64]
    args = batch(q, kv, H=2, D=8, seed=5)
    a = run(*args, 64, mode, 0.3)
    b = run(*args, None, mode, 0.3)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh"])
def test_window_gradients_match_finite_differences(mode):
    q, kv = [6, 4], [6, 7]
    q_off, kv_off, Q, K, V, dO, bias = batch(q, kv, H=1, D=3, seed=9, std=0.8)
    W, scale, h = 2, 0.5, 1e-6
    _, _, dQ, dK, dV = run(q_off, kv_off, Q, K, V, dO, bias, W, mode, scale)

    def loss(Qx, Kx, Vx):
        O, _ = oracle.fwd(q_off, kv_off, Qx.numpy(), Kx.numpy(), Vx.numpy(), mode=mode, causal=True,
                          bias=bias.numpy(), scale=scale, window=W)
        return float((torch.from_numpy(O) * dO).sum())

    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = torch.zeros_like(X)
        flat = X.reshape(-1)
        for idx in range(flat.numel()):
            old = float(flat[idx])
            flat[idx] = old + h
            lp = loss(Q, K, V)
            flat[idx] = old - h
            lm = loss(Q, K, V)
            flat[idx] = old
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        err = float((num - G).norm() / max(1e-30, float(G.norm())))
        assert err < 1e-6, (name, err)
