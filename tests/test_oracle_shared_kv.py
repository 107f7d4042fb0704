"""Pins for the oracle's shared key/value attention.  In IKBO, many candidate query sets
attend to one user's history, and the history is broadcast inside the kernel rather than
copied (PyTorch blog "In-Kernel Broadcast Optimization: Co-Designing Kernels for RecSys
Inference", section 3 and figure 1).

Each test checks the oracle against something other than itself:
- the identity map reproduces the plain jagged oracle;
- autograd in fp64 through an explicit broadcast (torch index_select of K and V, then
  SDPA per query set): a library routine, whose backward sums the gradients of the copies;
- central finite differences on a tiny case;
- a user that no query set uses gets zero gradients."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from jagged_sequence_attention_gb300 import workloads as wl

torch.set_default_dtype(torch.float64)


def bucket_ref(r: int) -> int:
    return min(31, ((1 + abs(int(r))) ** 2).bit_length() - 1)


def make(q_lens, user_lens, kv_index, H, D, seed, std=0.8):
    g = torch.Generator().manual_seed(seed)
    q_off, u_off = wl.offsets(q_lens), wl.offsets(user_lens)
    Q = torch.randn(int(q_off[-1]), H, D, generator=g) * std
    K = torch.randn(int(u_off[-1]), H, D, generator=g) * std
    V = torch.randn(int(u_off[-1]), H, D, generator=g)
    dO = torch.randn(int(q_off[-1]), H, D, generator=g)
    table = torch.randn(H, 32, generator=g) * 0.5
    return q_off, u_off, np.asarray(kv_index, dtype=np.int32), Q, K, V, dO, table


def broadcast_reference(q_off, u_off, kv_index, Q, K, V, dO, table, mode, causal, scale):
    """index_select of each query set's user rows (autograd sums the copies' gradients),
    SDPA or act(S) V per query set, loss sum(O * dO)."""
    H = Q.shape[1]
    K = K.clone().requires_grad_(True)
    V = V.clone().requires_grad_(True)
    Qg = Q.clone().requires_grad_(True)
    outs = []
    for b in range(len(q_off) - 1):
        u = int(kv_index[b])
        qs, qe = int(q_off[b]), int(q_off[b + 1])
        rows = torch.arange(int(u_off[u]), int(u_off[u + 1]))
        Lq, Lk = qe - qs, len(rows)
        if Lq == 0:
            continue
        if Lk == 0:
            outs.append(torch.zeros(Lq, H, Q.shape[2]))
            continue
        k = K.index_select(0, rows).permute(1, 0, 2)
        v = V.index_select(0, rows).permute(1, 0, 2)
        q = Qg[qs:qe].permute(1, 0, 2)
        ip = torch.arange(Lq)[:, None] + (Lk - Lq)
        j = torch.arange(Lk)[None, :]
        allowed = (j <= ip) if causal else torch.ones(Lq, Lk, dtype=torch.bool)
        idx = torch.tensor([[bucket_ref(r) for r in row] for row in (ip - j).tolist()], dtype=torch.long)
        add = table[:, idx]
        row_has = allowed.any(dim=1)
        if mode == "softmax":
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=add.masked_fill(~allowed, float("-inf")), scale=scale)
            o = torch.where(row_has[None, :, None], o, torch.zeros_like(o))
        else:
            s = scale * q @ k.transpose(-1, -2) + add
            a = (F.gelu(s, approximate="tanh") if mode == "gelu_tanh" else F.silu(s)).masked_fill(~allowed, 0.0)
            o = a @ v
        outs.append(o.permute(1, 0, 2))
    O = torch.cat(outs) if outs else torch.zeros(0, H, Q.shape[2])
    (O * dO).sum().backward()
    return O.detach(), Qg.grad, K.grad, V.grad


def run(q_off, u_off, kv_index, Q, K, V, dO, table, mode, causal, scale):
    kw = dict(mode=mode, causal=causal, bias=table.numpy(), scale=scale)
    O, _ = oracle.shared_kv_fwd(q_off, u_off, kv_index, Q.numpy(), K.numpy(), V.numpy(), **kw)
    dQ, dK, dV = oracle.shared_kv_bwd(q_off, u_off, kv_index, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), **kw)
    return O, dQ, dK, dV


CASES = [
    # query set lengths, user lengths, user of each query set
    ([3, 9, 1, 12, 5, 7], [20, 11, 6, 8], [0, 0, 1, 0, 3, 1]),    # user 2 unused
    ([16, 4, 4, 30], [16, 40], [0, 1, 1, 1]),                      # q > kv and q < kv
]


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_matches_autograd_through_a_broadcast(mode, causal, case):
    q, u, m = CASES[case]
    args = make(q, u, m, H=2, D=8, seed=60 + case)
    scale = 0.4
    got = run(*args, mode, causal, scale)
    want = broadcast_reference(*args, mode, causal, scale)
    for name, g, w in zip(("O", "dQ", "dK", "dV"), got, want):
        assert np.allclose(g, w.numpy(), atol=1e-12, rtol=1e-10), (name, float(np.abs(g - w.numpy()).max()))


def test_identity_map_is_the_plain_oracle():
    q = [5, 17, 0, 9]
    kv = [7, 17, 3, 12]
    q_off, u_off, m, Q, K, V, dO, table = make(q, kv, [0, 1, 2, 3], H=2, D=8, seed=70)
    kw = dict(mode="softmax", causal=True, bias=table.numpy(), scale=0.3)
    a = oracle.shared_kv_bwd(q_off, u_off, m, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), **kw)
    b = oracle.bwd(q_off, u_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), **kw)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_unused_user_has_zero_gradients():
    q, u, m = CASES[0]
    args = make(q, u, m, H=2, D=8, seed=71)
    _, _, dK, dV = run(*args, "softmax", False, 0.4)
    rows = slice(int(args[1][2]), int(args[1][3]))
    assert np.all(dK[rows] == 0) and np.all(dV[rows] == 0)
    assert np.abs(dK[:int(args[1][2])]).max() > 0


def test_finite_differences_on_the_shared_history():
    q, u, m = [3, 2, 4], [5, 3], [0, 0, 1]
    q_off, u_off, kv_index, Q, K, V, dO, table = make(q, u, m, H=1, D=3, seed=72)
    scale, h = 0.5, 1e-6
    _, dQ, dK, dV = run(q_off, u_off, kv_index, Q, K, V, dO, table, "softmax", True, scale)

    def loss(Kx, Vx):
        O, _ = oracle.shared_kv_fwd(q_off, u_off, kv_index, Q.numpy(), Kx.numpy(), Vx.numpy(), causal=True,
                                    bias=table.numpy(), scale=scale)
        return float((O * dO.numpy()).sum())

    for X, G in ((K, dK), (V, dV)):
        num = np.zeros(X.numel())
        flat = X.reshape(-1)
        for e in range(flat.numel()):
            old = float(flat[e])
            flat[e] = old + h
            lp = loss(K, V)
            flat[e] = old - h
            lm = loss(K, V)
            flat[e] = old
            num[e] = (lp - lm) / (2 * h)
        assert np.abs(num - G.reshape(-1)).max() < 1e-7
