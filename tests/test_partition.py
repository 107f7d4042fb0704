"""Data-parallel sharding (host only, no GPU): the LPT split of a batch's sequences over
GPUs, and a world-size-2 run over the gloo backend showing that the shards' results are
exactly the full batch's results.

Sequences are independent problems (each attends only within itself), so a batch
shards with no exchange; these tests check the split's invariants and the shard/gather
path end to end, with the CPU oracle standing in for each rank's GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from jagged_sequence_attention_gb300 import _build
from jagged_sequence_attention_gb300 import workloads as wl

BM = BN = 128


@pytest.fixture(scope="module")
def jfa():
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    m.lib()
    return m


def tiles_visited(q_len, kv_len, causal):
    """Brute-force count of 128x128 score tiles holding at least one allowed pair."""
    n = 0
    for t in range((q_len + BM - 1) // BM):
        rows = range(t * BM, min(q_len, (t + 1) * BM))
        for kt in range((kv_len + BN - 1) // BN):
            first_col = kt * BN
            if (not causal) or any(first_col <= r + kv_len - q_len for r in (rows[-1],)):
                n += 1
    return n


def expected_cost(q_len, kv_len, H, causal):
    nq, nk = (q_len + BM - 1) // BM, (kv_len + BN - 1) // BN
    return H * (9 * tiles_visited(q_len, kv_len, causal) + 2 * (nq + nk))


CASES = [
    ([5, 300, 129, 0, 1024, 77, 640], [5, 300, 129, 3, 1024, 77, 640], True),
    ([1, 64, 33, 700], [900, 10, 2000, 700], False),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("n_parts", [1, 2, 3, 8])
def test_partition_covers_and_balances(jfa, case, n_parts):
    q, kv, causal = CASES[case]
    H = 3
    part, cost = jfa.jfa_partition_sequences(wl.offsets(q), wl.offsets(kv), H, causal, n_parts)
    assert part.shape == (len(q),) and np.all((part >= 0) & (part < n_parts))
    seq_cost = np.array([expected_cost(a, b, H, causal) for a, b in zip(q, kv)], dtype=np.int64)
    # each part's cost is the sum of its sequences' costs
    for c in range(n_parts):
        assert cost[c] == seq_cost[part == c].sum()
    # greedy list scheduling bound
    assert cost.max() - cost.min() <= seq_cost.max()
    # the longest sequence is placed first, on part 0
    assert part[int(np.argmax(seq_cost))] == 0


def test_partition_is_deterministic_and_balanced_on_the_long_workload(jfa):
    w = wl.WORKLOADS["long_causal"]
    q, kv = wl.lengths(w)
    a = jfa.jfa_partition_sequences(wl.offsets(q), wl.offsets(kv), w.H, w.causal, 8)
    b = jfa.jfa_partition_sequences(wl.offsets(q), wl.offsets(kv), w.H, w.causal, 8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert a[1].max() / a[1].min() < 1.02


def test_partition_edge_cases_and_errors(jfa):
    part, cost = jfa.jfa_partition_sequences([0], [0], 2, False, 4)
    assert part.size == 0 and np.all(cost == 0)
    part, cost = jfa.jfa_partition_sequences([0, 5, 9], [0, 5, 9], 2, True, 1)
    assert np.all(part == 0)
    for bad in (([0, 5, 3], [0, 1, 2], 2, False, 2), ([0, 5], [0, 1], 0, False, 2), ([0, 5], [0, 1], 2, False, 0)):
        with pytest.raises(jfa.JFAError) as e:
            jfa.jfa_partition_sequences(*bad)
        assert e.value.status == jfa.JFA_ERR_INVALID_ARG


def test_shard_selects_each_ranks_sequences(jfa):
    b = wl.make_custom([5, 300, 129, 64], [5, 300, 129, 64], H=2, D=32, dtype=torch.float32, causal=True)
    parts, _ = jfa.jfa_partition_sequences(b.q_off, b.kv_off, b.H, b.causal, 2)
    seen = []
    for r in range(2):
        sub = jfa.shard(b, r, 2)
        seen += sub.extra["seqs"]
        assert list(sub.extra["seqs"]) == [int(s) for s in np.nonzero(parts == r)[0]]
        assert np.array_equal(sub.q_lens, b.q_lens[sub.extra["seqs"]])
    assert sorted(seen) == list(range(b.B))


# ------------------------------------------------------------------ world size 2 over gloo


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    # Each rank: its LPT shard of one seeded batch, forward + backward on its own "GPU"
    # (the CPU oracle here), results gathered to rank 0, which compares them with the
    # full-batch results sequence by sequence.
    import oracle
    from jagged_sequence_attention_gb300 import jfa
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        q = [37, 5, 130, 64, 1, 200]
        b = wl.make_custom(q, q, H=2, D=32, dtype=torch.float32, causal=True, bias=True, seed=99)
        sub = jfa.shard(b, rank, world)

        def run(batch):
            Tq = int(batch.q_off[-1])
            Q, K, V, dO = (t.double().numpy()[:Tq] for t in (batch.Q, batch.K, batch.V, batch.dO))
            bias = batch.bias.double().numpy()
            O, lse = oracle.fwd(batch.q_off, batch.kv_off, Q, K, V, causal=True, bias=bias, scale=batch.scale)
            dQ, dK, dV = oracle.bwd(batch.q_off, batch.kv_off, Q, K, V, dO, causal=True, bias=bias, scale=batch.scale)
            return O, dQ, dK, dV

        mine = run(sub)
        gathered = [None] * world
        dist.all_gather_object(gathered, {"seqs": list(sub.extra["seqs"]), "q_off": sub.q_off.tolist(),
                                          "out": [a.tolist() for a in mine]})
        if rank == 0:
            full = run(b)
            covered = []
            for g in gathered:
                offs = g["q_off"]
                for k, s in enumerate(g["seqs"]):
                    covered.append(s)
                    lo, hi = int(b.q_off[s]), int(b.q_off[s + 1])
                    for name, part_out, full_out in zip(("O", "dQ", "dK", "dV"), g["out"], full):
                        got = np.asarray(part_out)[offs[k]:offs[k + 1]]
                        assert np.array_equal(got, full_out[lo:hi]), (name, s)
            assert sorted(covered) == list(range(b.B))
            open(os.path.join(out_dir, "ok"), "w").write("ok")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo_reproduce_the_full_batch(jfa, tmp_path):
    import oracle
    oracle.build()
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    assert (tmp_path / "ok").exists()


# ------------------------------------------------------------ shared key/value: split by user


def shared_case(seed=5):
    g = np.random.default_rng(seed)
    users = g.integers(50, 700, size=7).tolist()
    kv_map = g.integers(0, 6, size=30)            # user 6 has no query set
    q = g.integers(0, 200, size=30).tolist()
    return q, users, kv_map


@pytest.mark.parametrize("n_parts", [1, 2, 3])
def test_partition_users_covers_and_balances(jfa, n_parts):
    q, users, kv_map = shared_case()
    H = 2
    part, cost = jfa.jfa_partition_users(wl.offsets(q), wl.offsets(users), kv_map, H, False, n_parts)
    assert part.shape == (len(users),) and np.all((part >= 0) & (part < n_parts))
    ucost = np.array([H * 2 * ((L + BN - 1) // BN) for L in users], dtype=np.int64)
    for b, u in enumerate(kv_map):
        nq = (q[b] + BM - 1) // BM
        ucost[u] += H * (9 * tiles_visited(q[b], users[u], False) + 2 * nq)
    for c in range(n_parts):
        assert cost[c] == ucost[part == c].sum()
    assert cost.max() - cost.min() <= ucost.max()


def test_shard_of_a_shared_batch_keeps_users_whole(jfa):
    q, users, kv_map = shared_case()
    b = wl.make_shared_kv(q, users, kv_map, H=2, D=32, dtype=torch.float32)
    seen_users, seen_seqs = [], []
    for r in range(3):
        sub = jfa.shard(b, r, 3)
        seen_users += sub.extra["users"]
        seen_seqs += sub.extra["seqs"]
        # every query set of a kept user is kept, mapped to its renumbered user
        for i, s in enumerate(sub.extra["seqs"]):
            assert sub.extra["users"][sub.kv_map[i]] == kv_map[s]
    assert sorted(seen_users) == list(range(len(users)))
    assert sorted(seen_seqs) == list(range(len(q)))


def _rank_main_shared(rank, world, port, out_dir):
    # Each rank: its users (with all their query sets) of one seeded shared key/value
    # batch, forward + backward with the CPU oracle standing in for its GPU; rank 0
    # checks every query set's O, dQ and every user's dK, dV against the full batch.
    import oracle
    from jagged_sequence_attention_gb300 import jfa
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        q, users, kv_map = shared_case(6)
        b = wl.make_shared_kv(q, users, kv_map, H=2, D=16, dtype=torch.float32, bias=True, seed=77)
        sub = jfa.shard(b, rank, world)

        def run(batch):
            Q, K, V, dO = (t.double().numpy() for t in (batch.Q, batch.K, batch.V, batch.dO))
            kw = dict(bias=batch.bias.double().numpy(), scale=batch.scale)
            O, _ = oracle.shared_kv_fwd(batch.q_off, batch.kv_off, batch.kv_map, Q, K, V, **kw)
            dQ, dK, dV = oracle.shared_kv_bwd(batch.q_off, batch.kv_off, batch.kv_map, Q, K, V, dO, **kw)
            return O, dQ, dK, dV

        mine = run(sub)
        gathered = [None] * world
        dist.all_gather_object(gathered, {"users": list(sub.extra["users"]), "seqs": list(sub.extra["seqs"]),
                                          "q_off": sub.q_off.tolist(), "kv_off": sub.kv_off.tolist(),
                                          "out": [a.tolist() for a in mine]})
        if rank == 0:
            full = run(b)
            for g in gathered:
                O, dQ, dK, dV = (np.asarray(a) for a in g["out"])
                for k, s in enumerate(g["seqs"]):
                    lo, hi = int(b.q_off[s]), int(b.q_off[s + 1])
                    assert np.array_equal(O[g["q_off"][k]:g["q_off"][k + 1]], full[0][lo:hi])
                    assert np.array_equal(dQ[g["q_off"][k]:g["q_off"][k + 1]], full[1][lo:hi])
                for k, u in enumerate(g["users"]):
                    lo, hi = int(b.kv_off[u]), int(b.kv_off[u + 1])
                    assert np.array_equal(dK[g["kv_off"][k]:g["kv_off"][k + 1]], full[2][lo:hi])
                    assert np.array_equal(dV[g["kv_off"][k]:g["kv_off"][k + 1]], full[3][lo:hi])
            open(os.path.join(out_dir, "ok"), "w").write("ok")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo_reproduce_a_shared_batch(jfa, tmp_path):
    import oracle
    oracle.build()
    mp.spawn(_rank_main_shared, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    assert (tmp_path / "ok").exists()
