"""Seeded synthetic jagged batches.

This module only draws inputs: sequence lengths, packed values and the bias
table.  It holds none of the attention arithmetic, and both the CUDA path and the
CPU oracle take their inputs from it.

The five named workloads follow the shapes, value distributions and length
mixes of the jagged recommendation workloads the GEM articles describe
(sequences from hundreds to tens of thousands of tokens, asymmetric query and
key/value lengths, GDPA interaction layers).  No production length histogram is
published, so these seeded distributions stand in for one:

  log-normal lengths: round(exp(ln(median) + 1.0 * N(0,1))), then clamp;
  uniform lengths:    integers drawn uniformly from the closed range.

Seeds are ``20261202 + index`` (index 1..5).  Lengths are drawn first on a CPU
``torch.Generator``; values are drawn on the target device from a generator
seeded with ``seed + 1000``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    D: int
    dtype: torch.dtype
    mode: str                 # "softmax" | "gelu_tanh" | "silu"
    causal: bool
    bias: bool
    value_std: float
    q_len: tuple              # ("fixed", [..]) | ("uniform", lo, hi) | ("lognormal", median, lo, hi)
    kv_len: Optional[tuple]   # None: self-attention (kv lengths = q lengths)
    description: str = ""
    window: Optional[int] = None  # sliding window W (query i sees keys i' - W .. i'), or None
    # shared key/value: B query sets over `users` users (kv_len draws the users' lengths),
    # B // users consecutive query sets per user, or None
    users: Optional[int] = None


WORKLOADS = {
    "tiny": Workload(
        "tiny", 1, 4, 2, 32, torch.float32, "softmax", False, False, 1.0,
        ("fixed", [7, 16, 33, 64]), None,
        "4 sequences, q=kv lengths {7,16,33,64}, 2 heads, head_dim 32, fp32 N(0,1), softmax"),
    "causal_bias": Workload(
        "causal_bias", 2, 256, 8, 128, torch.bfloat16, "softmax", True, True, 1.0,
        ("lognormal", 256, 32, 2048), None,
        "256 user histories, log-normal lengths in [32,2048] (median 256), causal self-attention, "
        "8 heads, head_dim 128, bf16, 32-bucket relative-position bias"),
    "cross": Workload(
        "cross", 3, 512, 8, 64, torch.bfloat16, "softmax", False, False, 1.0,
        ("uniform", 1, 64), ("lognormal", 1000, 100, 16384),
        "512 sequences, q lengths U{1..64}, kv lengths log-normal in [100,16384] (median 1000), "
        "8 heads, head_dim 64, bf16, softmax, non-causal"),
    "gdpa_gelu": Workload(
        "gdpa_gelu", 4, 1024, 4, 128, torch.bfloat16, "gelu_tanh", False, False, 0.5,
        ("uniform", 1, 128), ("lognormal", 512, 64, 4096),
        "1024 sequences, q lengths U{1..128}, kv lengths log-normal in [64,4096] (median 512), "
        "4 heads, head_dim 128, bf16 N(0,0.5), GDPA tanh-GELU"),
    "gdpa_silu": Workload(
        "gdpa_silu", 4, 1024, 4, 128, torch.bfloat16, "silu", False, False, 0.5,
        ("uniform", 1, 128), ("lognormal", 512, 64, 4096),
        "as gdpa_gelu with SiLU"),
    "long_causal": Workload(
        "long_causal", 5, 64, 8, 128, torch.bfloat16, "softmax", True, True, 1.0,
        ("uniform", 4096, 32768), None,
        "64 sequences, lengths U{4096..32768} (~1.2M tokens), causal self-attention, 8 heads, "
        "head_dim 128, bf16, relative-position bias"),
    # Profiling case: the long-sequence structure at a size one profiler pass covers
    # quickly, with every input and the dQ accumulator still larger than L2.
    "long_causal_profile": Workload(
        "long_causal_profile", 6, 8, 8, 128, torch.bfloat16, "softmax", True, True, 1.0,
        ("uniform", 6144, 10240), None,
        "8 sequences, lengths U{6144..10240}, causal self-attention, 8 heads, head_dim 128, bf16, "
        "relative-position bias (profiling size of the long-sequence workload)"),
    # Sliding-window form of the long-sequence workload (the GEM articles' move from full to
    # sliding-window self-attention for long user sequences; window size not published).
    "long_window": Workload(
        "long_window", 7, 64, 8, 128, torch.bfloat16, "softmax", True, True, 1.0,
        ("uniform", 4096, 32768), None,
        "64 sequences, lengths U{4096..32768} (~1.2M tokens), causal sliding window of 2048 keys, 8 heads, "
        "head_dim 128, bf16, relative-position bias", window=2048),
    # Shared key/value (in-kernel broadcast): candidate query sets of a request attending to
    # the request's user history, the shape of the cross-attention workload with 64 query sets
    # per user (the IKBO article's candidate-to-user ratio is about 70).
    "ikbo_cross": Workload(
        "ikbo_cross", 8, 1024, 8, 64, torch.bfloat16, "softmax", False, False, 1.0,
        ("uniform", 1, 64), ("lognormal", 1000, 100, 16384),
        "1024 candidate query sets, q lengths U{1..64}, 64 per user over 16 users whose histories are "
        "log-normal in [100,16384] (median 1000), keys/values shared per user, 8 heads, head_dim 64, bf16, "
        "softmax, non-causal", users=16),
}


def seed_of(w: Workload) -> int:
    return BASE_SEED + w.index


def _draw(spec, n, gen) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        vals = np.asarray(spec[1], dtype=np.int64)
        assert vals.size == n
        return vals
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, (n,), generator=gen).numpy().astype(np.int64)
    if kind == "lognormal":
        median, lo, hi = spec[1], spec[2], spec[3]
        z = torch.randn(n, generator=gen, dtype=torch.float64).numpy()
        x = np.rint(np.exp(math.log(median) + 1.0 * z))
        return np.clip(x, lo, hi).astype(np.int64)
    raise ValueError(kind)


def lengths(w: Workload, seed: Optional[int] = None):
    """(q_lens, kv_lens) as int64 numpy arrays: B of each, or with shared key/value B
    query lengths and `users` user history lengths."""
    gen = torch.Generator().manual_seed(seed_of(w) if seed is None else seed)
    q = _draw(w.q_len, w.B, gen)
    kv = q.copy() if w.kv_len is None else _draw(w.kv_len, w.B if w.users is None else w.users, gen)
    return q, kv


def kv_map_of(w: Workload) -> np.ndarray:
    """Shared key/value: consecutive blocks of B // users query sets per user."""
    return (np.arange(w.B) // (w.B // w.users)).astype(np.int32)


def offsets(lens) -> np.ndarray:
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    np.cumsum(np.asarray(lens, dtype=np.int64), out=out[1:])
    if out[-1] >= 2**31:
        raise ValueError("total length exceeds int32 offsets")
    return out.astype(np.int32)


@dataclass
class Batch:
    name: str
    q_off: np.ndarray          # int32 [B+1]
    kv_off: np.ndarray         # int32 [B+1]
    Q: torch.Tensor            # [Tq, H, D]
    K: torch.Tensor            # [Tkv, H, D]
    V: torch.Tensor            # [Tkv, H, D]
    dO: Optional[torch.Tensor]  # [Tq, H, D]
    bias: Optional[torch.Tensor]  # fp32 [H, 32] (same device as values)
    scale: float
    mode: str
    causal: bool
    H: int
    D: int
    extra: dict = field(default_factory=dict)
    window: Optional[int] = None   # sliding window W (query i sees keys i' - W .. i'), or None
    # dense per-pair bias fp32 [H, P], P = sum q_len * kv_len, sequence b's block row-major
    # [q_len, kv_len] from pair_offsets()[b] (used instead of the bucket table), or None
    dense: Optional[torch.Tensor] = None
    # shared key/value: query set b attends to the rows of user kv_map[b] (kv_off then
    # runs over the users), or None
    kv_map: Optional[np.ndarray] = None

    @property
    def B(self) -> int:
        return self.q_off.size - 1

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.q_off.astype(np.int64))

    @property
    def kv_lens(self) -> np.ndarray:
        """Key/value length of each sequence (shared key/value: of each query set's user)."""
        lens = np.diff(self.kv_off.astype(np.int64))
        return lens if self.kv_map is None else lens[self.kv_map]


def _values(shape, std, dtype, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def pair_offsets(q_off, kv_off) -> np.ndarray:
    """int64 [B+1]: where each sequence's block of a dense per-pair array starts."""
    q = np.diff(np.asarray(q_off, dtype=np.int64))
    kv = np.diff(np.asarray(kv_off, dtype=np.int64))
    return np.concatenate([[0], np.cumsum(q * kv)]).astype(np.int64)


def make_custom(q_lens, kv_lens, *, H, D, dtype=torch.bfloat16, mode="softmax", causal=False,
                bias=False, value_std=1.0, seed=BASE_SEED, device="cpu", with_grad=True,
                name="custom", pad_rows=0, window=None, dense_bias=False) -> Batch:
    """A batch with the given lengths.  ``pad_rows`` extra rows are appended to every
    value tensor (beyond the last offset) so tests can check that nothing there is read
    into a result or written."""
    q_off, kv_off = offsets(q_lens), offsets(kv_lens)
    Tq, Tkv = int(q_off[-1]) + pad_rows, int(kv_off[-1]) + pad_rows
    gen = torch.Generator(device=device).manual_seed(seed + 1000)
    Q = _values((Tq, H, D), value_std, dtype, gen, device)
    K = _values((Tkv, H, D), value_std, dtype, gen, device)
    V = _values((Tkv, H, D), value_std, dtype, gen, device)
    dO = _values((Tq, H, D), 1.0, dtype, gen, device) if with_grad else None
    b = None
    if bias:
        b = (torch.randn((H, 32), generator=gen, device=device, dtype=torch.float32) * 0.1)
    dn = None
    if dense_bias:  # N(0, 0.5) per pair
        P = int(pair_offsets(q_off, kv_off)[-1])
        dn = torch.randn((H, P), generator=gen, device=device, dtype=torch.float32) * 0.5
    return Batch(name, q_off, kv_off, Q, K, V, dO, b, 1.0 / math.sqrt(D), mode, causal, H, D, window=window,
                 dense=dn)


def make_shared_kv(q_lens, user_lens, kv_map, *, H, D, dtype=torch.bfloat16, mode="softmax", causal=False,
                   bias=False, value_std=1.0, seed=BASE_SEED, device="cpu", with_grad=True, name="shared_kv",
                   window=None, dense_bias=False) -> Batch:
    """Query sets (q_lens) attending to users' histories (user_lens) through kv_map: the
    keys and values exist once per user."""
    q_off, u_off = offsets(q_lens), offsets(user_lens)
    kv_map = np.ascontiguousarray(np.asarray(kv_map, dtype=np.int32))
    gen = torch.Generator(device=device).manual_seed(seed + 2000)
    Q = _values((int(q_off[-1]), H, D), value_std, dtype, gen, device)
    K = _values((int(u_off[-1]), H, D), value_std, dtype, gen, device)
    V = _values((int(u_off[-1]), H, D), value_std, dtype, gen, device)
    dO = _values((int(q_off[-1]), H, D), 1.0, dtype, gen, device) if with_grad else None
    b = None
    if bias:
        b = (torch.randn((H, 32), generator=gen, device=device, dtype=torch.float32) * 0.1)
    dn = None
    if dense_bias:  # one block per query set, q_len x its user's kv_len
        ul = np.diff(u_off.astype(np.int64))
        P = int(np.sum(np.diff(q_off.astype(np.int64)) * ul[kv_map])) if kv_map.size else 0
        dn = torch.randn((H, P), generator=gen, device=device, dtype=torch.float32) * 0.5
    return Batch(name, q_off, u_off, Q, K, V, dO, b, 1.0 / math.sqrt(D), mode, causal, H, D, window=window,
                 dense=dn, kv_map=kv_map)


def make(name: str, device="cpu", with_grad=True, seed: Optional[int] = None) -> Batch:
    """The named workload, seeded."""
    w = WORKLOADS[name]
    s = seed_of(w) if seed is None else seed
    q, kv = lengths(w, s)
    if w.users is not None:
        return make_shared_kv(q, kv, kv_map_of(w), H=w.H, D=w.D, dtype=w.dtype, mode=w.mode, causal=w.causal,
                              bias=w.bias, value_std=w.value_std, seed=s, device=device, with_grad=with_grad,
                              name=name, window=w.window)
    return make_custom(q, kv, H=w.H, D=w.D, dtype=w.dtype, mode=w.mode, causal=w.causal,
                       bias=w.bias, value_std=w.value_std, seed=s, device=device,
                       with_grad=with_grad, name=name, window=w.window)


def broadcast(batch: Batch) -> Batch:
    """A shared key/value batch with its broadcast made explicit: each query set gets its
    own copy of its user's key/value rows (the copies the in-kernel broadcast avoids)."""
    if batch.kv_map is None:
        return batch
    rows = [np.arange(batch.kv_off[u], batch.kv_off[u + 1]) for u in batch.kv_map]
    rows = np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, dtype=np.int64)
    idx = torch.from_numpy(rows).to(batch.K.device)
    return Batch(batch.name + "/broadcast", batch.q_off, offsets(batch.kv_lens), batch.Q,
                 batch.K.index_select(0, idx).contiguous(), batch.V.index_select(0, idx).contiguous(), batch.dO,
                 batch.bias, batch.scale, batch.mode, batch.causal, batch.H, batch.D, window=batch.window,
                 dense=batch.dense)


def subset_users(batch: Batch, users) -> Batch:
    """Users of a shared key/value batch with all their query sets, repacked: users
    renumbered in the given order, query sets kept in batch order.  extra records the
    original users ("users") and query sets ("seqs")."""
    users = [int(u) for u in users]
    new_id = {u: i for i, u in enumerate(users)}
    seqs = [b for b in range(batch.B) if int(batch.kv_map[b]) in new_id]
    qi = [torch.arange(int(batch.q_off[s]), int(batch.q_off[s + 1])) for s in seqs]
    ki = [torch.arange(int(batch.kv_off[u]), int(batch.kv_off[u + 1])) for u in users]
    qi = torch.cat(qi) if qi else torch.zeros(0, dtype=torch.long)
    ki = torch.cat(ki) if ki else torch.zeros(0, dtype=torch.long)

    def take(t, idx):
        return None if t is None else t.index_select(0, idx.to(t.device)).contiguous()

    dn = None
    if batch.dense is not None:
        lens = np.diff(batch.q_off.astype(np.int64)) * batch.kv_lens
        po = np.concatenate([[0], np.cumsum(lens)])
        blocks = [batch.dense[:, int(po[s]):int(po[s + 1])] for s in seqs]
        dn = torch.cat(blocks, dim=1).contiguous() if blocks else batch.dense[:, :0].contiguous()
    ulens = np.diff(batch.kv_off.astype(np.int64))[users] if users else np.zeros(0, dtype=np.int64)
    sub = Batch(batch.name + "/users", offsets(batch.q_lens[seqs]), offsets(ulens), take(batch.Q, qi),
                take(batch.K, ki), take(batch.V, ki), take(batch.dO, qi), batch.bias, batch.scale, batch.mode,
                batch.causal, batch.H, batch.D, window=batch.window, dense=dn,
                kv_map=np.asarray([new_id[int(batch.kv_map[s])] for s in seqs], dtype=np.int32))
    sub.extra.update(users=users, seqs=seqs, q_index=qi, kv_index=ki)
    return sub


def subset(batch: Batch, seqs, heads=None) -> Batch:
    """Independent sequences (and optionally heads) of a batch, repacked; a sequence's
    result does not depend on the others, so the oracle can check a sample this way."""
    seqs = [int(s) for s in seqs]
    heads = list(range(batch.H)) if heads is None else [int(h) for h in heads]
    qi = [torch.arange(int(batch.q_off[s]), int(batch.q_off[s + 1])) for s in seqs]
    ki = [torch.arange(int(batch.kv_off[s]), int(batch.kv_off[s + 1])) for s in seqs]
    qi = torch.cat(qi) if qi else torch.zeros(0, dtype=torch.long)
    ki = torch.cat(ki) if ki else torch.zeros(0, dtype=torch.long)
    hs = torch.tensor(heads, dtype=torch.long)

    def take(t, idx):
        if t is None:
            return None
        idx = idx.to(t.device)
        return t.index_select(0, idx).index_select(1, hs.to(t.device)).contiguous()

    dn = None
    if batch.dense is not None:
        po = pair_offsets(batch.q_off, batch.kv_off)
        blocks = [batch.dense[:, int(po[s]):int(po[s + 1])] for s in seqs]
        dn = torch.cat(blocks, dim=1) if blocks else batch.dense[:, :0]
        dn = dn[hs.to(dn.device)].contiguous()
    sub = Batch(batch.name + "/subset", offsets(batch.q_lens[seqs]), offsets(batch.kv_lens[seqs]),
                take(batch.Q, qi), take(batch.K, ki), take(batch.V, ki), take(batch.dO, qi),
                None if batch.bias is None else batch.bias[hs.to(batch.bias.device)].contiguous(),
                batch.scale, batch.mode, batch.causal, len(heads), batch.D, window=batch.window, dense=dn)
    sub.extra.update(seqs=seqs, heads=heads, q_index=qi, kv_index=ki)
    return sub
