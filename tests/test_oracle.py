"""Pins for the CPU oracle: each checks the oracle against something other than
itself -- a library routine on a special case, a closed form, an invariant, or
finite differences -- so that a dropped term, a wrong sign, a wrong index or a
transposed operand in the oracle fails at least one of them.

What the GEM articles fix and these tests encode:
  * jagged attention equals ordinary attention over each sequence alone
    ("Jagged Sequence Flash Attention"; FAQ "Jagged tensor 是什么");
  * padding with zeros and masking does not change results or gradients
    (the IKBO article's zero-padding equivalence argument, section 2.2);
  * GDPA is two matrix products with GELU or SiLU between them and no
    normalisation ("Generalized Dot-Product Attention (GDPA)").
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from jagged_sequence_attention_gb300 import workloads as wl

torch.set_default_dtype(torch.float64)


def bucket_ref(r: int) -> int:
    # floor(log2(n)) for a positive integer n is n.bit_length() - 1 (exact integers).
    return min(31, ((1 + abs(r)) ** 2).bit_length() - 1)


def rand_batch(q_lens, kv_lens, H, D, seed, std=1.0, bias=False):
    g = torch.Generator().manual_seed(seed)
    q_off, kv_off = wl.offsets(q_lens), wl.offsets(kv_lens)
    Q = torch.randn(int(q_off[-1]), H, D, generator=g) * std
    K = torch.randn(int(kv_off[-1]), H, D, generator=g) * std
    V = torch.randn(int(kv_off[-1]), H, D, generator=g)
    dO = torch.randn(int(q_off[-1]), H, D, generator=g)
    b = torch.randn(H, 32, generator=g) * 0.5 if bias else None
    return q_off, kv_off, Q, K, V, dO, b


def dense_bias_and_mask(Lq, Lk, H, bias, causal):
    """Per-sequence additive mask [H, Lq, Lk]: bias table lookup plus -inf where a key
    is not allowed (bottom-right causal)."""
    i = torch.arange(Lq)[:, None]
    j = torch.arange(Lk)[None, :]
    rel = i + (Lk - Lq) - j
    add = torch.zeros(H, Lq, Lk)
    if bias is not None:
        idx = torch.tensor([[bucket_ref(int(r)) for r in row] for row in rel.tolist()],
                           dtype=torch.long).reshape(Lq, Lk)
        add = add + bias[:, idx]
    allowed = torch.ones(Lq, Lk, dtype=torch.bool) if not causal else (j <= i + (Lk - Lq))
    add = add.masked_fill(~allowed, float("-inf"))
    return add, allowed


def torch_reference(q_off, kv_off, Q, K, V, dO, bias, causal, mode, scale):
    """Library special case: per sequence, SDPA (softmax) or matmul-act-matmul (GDPA)
    in fp64 with autograd for the gradients."""
    B = len(q_off) - 1
    H, D = Q.shape[1], Q.shape[2]
    O = torch.zeros_like(Q)
    LSE = torch.zeros(Q.shape[0], H)
    dQ, dK, dV = torch.zeros_like(Q), torch.zeros_like(K), torch.zeros_like(V)
    for b in range(B):
        qs, qe, ks, ke = int(q_off[b]), int(q_off[b + 1]), int(kv_off[b]), int(kv_off[b + 1])
        Lq, Lk = qe - qs, ke - ks
        if Lq == 0:
            continue
        q = Q[qs:qe].permute(1, 0, 2).clone().requires_grad_(True)
        k = K[ks:ke].permute(1, 0, 2).clone().requires_grad_(True)
        v = V[ks:ke].permute(1, 0, 2).clone().requires_grad_(True)
        add, allowed = dense_bias_and_mask(Lq, Lk, H, bias, causal)
        row_has = allowed.any(dim=1)  # [Lq]
        if mode == "softmax":
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=add, scale=scale)
            o = torch.where(row_has[None, :, None], o, torch.zeros_like(o))
            s = scale * q @ k.transpose(-1, -2) + add
            lse = torch.logsumexp(s, dim=-1)
        else:
            s = scale * q @ k.transpose(-1, -2) + add.masked_fill(~allowed, 0.0)
            a = F.gelu(s, approximate="tanh") if mode == "gelu_tanh" else F.silu(s)
            a = a.masked_fill(~allowed, 0.0)
            o = a @ v
            lse = torch.zeros(H, Lq)
        O[qs:qe] = o.detach().permute(1, 0, 2)
        LSE[qs:qe] = lse.detach().T
        if dO is not None and Lk > 0:
            (o * dO[qs:qe].permute(1, 0, 2)).sum().backward()
            dQ[qs:qe] = q.grad.permute(1, 0, 2)
            dK[ks:ke] = k.grad.permute(1, 0, 2)
            dV[ks:ke] = v.grad.permute(1, 0, 2)
    return O, LSE, dQ, dK, dV


def run_oracle(q_off, kv_off, Q, K, V, dO, bias, causal, mode, scale):
    b = None if bias is None else bias.numpy()
    O, LSE = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), mode=mode,
                        causal=causal, bias=b, scale=scale)
    dQ, dK, dV = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(),
                            mode=mode, causal=causal, bias=b, scale=scale)
    return [torch.from_numpy(x) for x in (O, LSE, dQ, dK, dV)]


# ---------------------------------------------------------------------------
# bias bucket


def test_relpos_bucket_matches_integer_log2():
    rs = list(range(0, 5000)) + [46339, 46340, 46341, 10**6, 2**31 - 1, -1, -7, -5000]
    for r in rs:
        assert oracle.relpos_bucket(r) == bucket_ref(r), r


def test_relpos_bucket_golden_boundaries():
    """Worked values of bucket(r) = min(31, floor(log2((1+r)^2))) written out by hand."""
    table = {0: 0, 1: 2, 2: 3, 3: 4, 4: 4, 5: 5, 6: 5, 7: 6, 10: 6, 11: 7, 15: 8, 21: 8, 22: 9,
             23: 9, 31: 10, 1023: 20, 46339: 30, 46340: 31, 10**9: 31}
    for r, b in table.items():
        assert oracle.relpos_bucket(r) == b, (r, b)


# ---------------------------------------------------------------------------
# activations


@pytest.mark.parametrize("mode", ["gelu_tanh", "silu"])
def test_activation_values_match_torch(mode):
    xs = np.linspace(-12, 12, 241)
    ref = (F.gelu(torch.tensor(xs), approximate="tanh") if mode == "gelu_tanh"
           else F.silu(torch.tensor(xs))).numpy()
    got = np.array([oracle.act(mode, x) for x in xs])
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("mode", ["gelu_tanh", "silu"])
def test_activation_grad_matches_autograd(mode):
    x = torch.linspace(-12, 12, 241).requires_grad_(True)
    y = F.gelu(x, approximate="tanh") if mode == "gelu_tanh" else F.silu(x)
    y.sum().backward()
    got = np.array([oracle.act_grad(mode, float(v)) for v in x.detach()])
    np.testing.assert_allclose(got, x.grad.numpy(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# jagged == dense attention on each sequence alone (library special case)

CASES = [
    ([5, 1, 9, 3], [5, 1, 9, 3]),           # self-attention
    ([3, 7, 1, 4], [6, 2, 11, 4]),          # q != kv, both directions
    ([2, 6], [1, 9]),
]


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_matches_dense_library_per_sequence(mode, causal, bias, case):
    q_lens, kv_lens = CASES[case]
    H, D = 2, 8
    q_off, kv_off, Q, K, V, dO, b = rand_batch(q_lens, kv_lens, H, D, seed=11 + case, bias=bias)
    scale = 1.0 / math.sqrt(D)
    ref = torch_reference(q_off, kv_off, Q, K, V, dO, b, causal, mode, scale)
    got = run_oracle(q_off, kv_off, Q, K, V, dO, b, causal, mode, scale)
    names = ["O", "LSE", "dQ", "dK", "dV"]
    for n, r, g in zip(names, ref, got):
        if n == "LSE" and mode != "softmax":
            continue
        fin = torch.isfinite(r)
        assert torch.equal(fin, torch.isfinite(g)), n
        torch.testing.assert_close(g[fin], r[fin], rtol=1e-10, atol=1e-12, msg=n)


# ---------------------------------------------------------------------------
# closed forms and special cases


def test_single_key_returns_v_exactly():
    q_lens, kv_lens = [4, 1, 3], [1, 1, 1]
    q_off, kv_off, Q, K, V, dO, b = rand_batch(q_lens, kv_lens, 3, 16, seed=5, bias=True)
    O, LSE = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), bias=b.numpy())
    for bi in range(3):
        for i in range(int(q_off[bi]), int(q_off[bi + 1])):
            np.testing.assert_array_equal(O[i], V.numpy()[kv_off[bi]])
            for h in range(3):
                qi, ki = int(i - q_off[bi]), 0
                s = (Q[i, h] @ K[kv_off[bi], h]).item() / 4.0 + \
                    b[h, bucket_ref(qi + (1 - q_lens[bi]) - ki)].item()
                assert abs(LSE[i, h] - s) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_give_mean_of_allowed_values(causal):
    q_lens, kv_lens = [4, 6, 3], [4, 9, 5]
    q_off, kv_off, Q, K, V, dO, _ = rand_batch(q_lens, kv_lens, 2, 8, seed=6)
    Q.zero_()
    O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), causal=causal)
    _, _, dV = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), causal=causal)
    for b in range(3):
        Lq, Lk = q_lens[b], kv_lens[b]
        Vb = V.numpy()[kv_off[b]:kv_off[b + 1]]
        dOb = dO.numpy()[q_off[b]:q_off[b + 1]]
        dv_ref = np.zeros_like(Vb)
        for i in range(Lq):
            n = Lk if not causal else min(Lk, i + 1 + Lk - Lq)
            np.testing.assert_allclose(O[q_off[b] + i], Vb[:n].mean(axis=0), rtol=1e-12, atol=1e-12)
            dv_ref[:n] += dOb[i] / n
        np.testing.assert_allclose(dV[kv_off[b]:kv_off[b + 1]], dv_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["gelu_tanh", "silu"])
def test_gdpa_zero_query_gives_zero(mode):
    q_off, kv_off, Q, K, V, dO, _ = rand_batch([3, 5], [7, 2], 2, 8, seed=7)
    Q.zero_()
    O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), mode=mode)
    assert np.all(O == 0.0)


def test_softmax_rows_sum_to_one():
    q_off, kv_off, Q, K, V, dO, b = rand_batch([6, 2, 5], [8, 3, 5], 2, 8, seed=8, bias=True)
    V = torch.ones_like(V)
    for causal in (False, True):
        O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), causal=causal,
                          bias=b.numpy())
        np.testing.assert_allclose(O, 1.0, rtol=1e-13)


def test_empty_rows_and_sequences():
    # seq0: kv empty; seq1: q empty; seq2: causal with q > kv (first rows see no key)
    q_lens, kv_lens = [3, 0, 5], [0, 4, 2]
    q_off, kv_off, Q, K, V, dO, _ = rand_batch(q_lens, kv_lens, 2, 4, seed=9)
    for mode in ("softmax", "gelu_tanh", "silu"):
        O, LSE = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), mode=mode, causal=True)
        dQ, dK, dV = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(),
                                mode=mode, causal=True)
        assert np.all(O[0:3] == 0) and np.all(dQ[0:3] == 0)
        # seq2 rows i=0..2 have no allowed key (j <= i - 3)
        assert np.all(O[3:6] == 0) and np.all(dQ[3:6] == 0)
        assert np.all(np.abs(O[6:8]) > 0)
        # keys of seq1 receive no gradient (no queries)
        assert np.all(dK[0:4] == 0) and np.all(dV[0:4] == 0)
        if mode == "softmax":
            assert np.all(np.isneginf(LSE[0:6])) and np.all(np.isfinite(LSE[6:8]))


# ---------------------------------------------------------------------------
# gradients by central finite differences


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
@pytest.mark.parametrize("causal,bias", [(False, False), (True, True), (False, True)])
def test_gradients_match_finite_differences(mode, causal, bias):
    q_lens, kv_lens = [3, 2], [4, 2]
    H, D = 2, 3
    q_off, kv_off, Q, K, V, dO, b = rand_batch(q_lens, kv_lens, H, D, seed=21, bias=bias)
    bn = None if b is None else b.numpy()
    Qn, Kn, Vn, dOn = Q.numpy(), K.numpy(), V.numpy(), dO.numpy()
    scale = 0.7

    def loss(Qx, Kx, Vx):
        O, _ = oracle.fwd(q_off, kv_off, Qx, Kx, Vx, mode=mode, causal=causal, bias=bn, scale=scale)
        return float((O * dOn).sum())

    grads = oracle.bwd(q_off, kv_off, Qn, Kn, Vn, dOn, mode=mode, causal=causal, bias=bn,
                       scale=scale)
    eps = 1e-6
    for which, (base, g) in enumerate(zip((Qn, Kn, Vn), grads)):
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            args = [Qn.copy(), Kn.copy(), Vn.copy()]
            args[which][idx] += eps
            lp = loss(*args)
            args[which][idx] -= 2 * eps
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, (which, err)


# ---------------------------------------------------------------------------
# invariants


@pytest.mark.parametrize("mode", ["softmax", "silu"])
def test_zero_padded_dense_equals_jagged(mode):
    """Pad every sequence with zero rows to the batch maximum and mask the padded keys:
    cropped results and gradients equal the jagged ones."""
    q_lens, kv_lens = [2, 5, 3], [4, 1, 6]
    H, D = 2, 8
    q_off, kv_off, Q, K, V, dO, b = rand_batch(q_lens, kv_lens, H, D, seed=31, bias=True)
    scale = 1.0 / math.sqrt(D)
    O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), mode=mode, bias=b.numpy(),
                      scale=scale)
    grads = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), mode=mode,
                       bias=b.numpy(), scale=scale)
    B, Lq, Lk = 3, max(q_lens), max(kv_lens)
    Qp = torch.zeros(B, H, Lq, D)
    Kp = torch.zeros(B, H, Lk, D)
    Vp = torch.zeros(B, H, Lk, D)
    dOp = torch.zeros(B, H, Lq, D)
    add = torch.zeros(B, H, Lq, Lk)
    for bi in range(B):
        lq, lk = q_lens[bi], kv_lens[bi]
        Qp[bi, :, :lq] = Q[q_off[bi]:q_off[bi + 1]].permute(1, 0, 2)
        Kp[bi, :, :lk] = K[kv_off[bi]:kv_off[bi + 1]].permute(1, 0, 2)
        Vp[bi, :, :lk] = V[kv_off[bi]:kv_off[bi + 1]].permute(1, 0, 2)
        dOp[bi, :, :lq] = dO[q_off[bi]:q_off[bi + 1]].permute(1, 0, 2)
        a, _ = dense_bias_and_mask(lq, lk, H, b, False)
        add[bi, :, :lq, :lk] = a
        add[bi, :, :, lk:] = float("-inf")
    Qp.requires_grad_(True)
    Kp.requires_grad_(True)
    Vp.requires_grad_(True)
    if mode == "softmax":
        Op = F.scaled_dot_product_attention(Qp, Kp, Vp, attn_mask=add, scale=scale)
    else:
        s = scale * Qp @ Kp.transpose(-1, -2) + add.masked_fill(torch.isinf(add), 0.0)
        Op = F.silu(s).masked_fill(torch.isinf(add), 0.0) @ Vp
    (Op * dOp).sum().backward()
    for bi in range(B):
        lq, lk = q_lens[bi], kv_lens[bi]
        np.testing.assert_allclose(O[q_off[bi]:q_off[bi + 1]],
                                   Op[bi, :, :lq].detach().permute(1, 0, 2).numpy(), rtol=1e-10,
                                   atol=1e-12)
        for g, gp, off, L in ((grads[0], Qp.grad, q_off, lq), (grads[1], Kp.grad, kv_off, lk),
                              (grads[2], Vp.grad, kv_off, lk)):
            np.testing.assert_allclose(g[off[bi]:off[bi + 1]], gp[bi, :, :L].permute(1, 0, 2).numpy(),
                                       rtol=1e-10, atol=1e-12)


def test_batch_permutation_permutes_outputs():
    q_lens, kv_lens = [3, 6, 2, 5], [4, 6, 7, 1]
    q_off, kv_off, Q, K, V, dO, b = rand_batch(q_lens, kv_lens, 2, 8, seed=41, bias=True)
    O, _ = oracle.fwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), causal=True, bias=b.numpy())
    perm = [2, 0, 3, 1]
    pq = np.concatenate([np.arange(q_off[p], q_off[p + 1]) for p in perm])
    pk = np.concatenate([np.arange(kv_off[p], kv_off[p + 1]) for p in perm])
    q2, k2 = wl.offsets([q_lens[p] for p in perm]), wl.offsets([kv_lens[p] for p in perm])
    O2, _ = oracle.fwd(q2, k2, Q.numpy()[pq], K.numpy()[pk], V.numpy()[pk], causal=True,
                       bias=b.numpy())
    np.testing.assert_array_equal(O2, O[pq])


def test_thread_count_does_not_change_results():
    q_off, kv_off, Q, K, V, dO, b = rand_batch([7, 3, 9], [5, 8, 9], 3, 8, seed=51, bias=True)
    a = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), causal=True,
                   bias=b.numpy(), nthreads=1)
    c = oracle.bwd(q_off, kv_off, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), causal=True,
                   bias=b.numpy(), nthreads=4)
    for x, y in zip(a, c):
        np.testing.assert_array_equal(x, y)
