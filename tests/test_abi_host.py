"""Host-side checks of libjfa: it builds, loads without a GPU, exports every entry
point include/jfa.h declares, and its planner (pure host code) produces correct,
balanced work lists.  No CUDA call is made here."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from jagged_sequence_attention_gb300 import _build
from jagged_sequence_attention_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jfa.h")

BM_FWD, BN_FWD = 128, 128
PAIR_FWD = 2 * BM_FWD
BN_BWD, BM_BWD = 128, 128


@pytest.fixture(scope="module")
def jfa():
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jfa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("jfa_plan_create", "jfa_plan_destroy", "jfa_fwd", "jfa_bwd", "jfa_bwd_workspace_size",
              "jfa_plan_device_status", "jfa_status_string", "jfa_worklist_size", "jfa_worklist_build",
              "jfa_plan_info"):
        assert n in names


def test_library_exports_every_declared_symbol(jfa):
    lib = jfa.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", jfa._LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (jfa_[a-z_]+)\b", out))
    assert set(declared_functions()) <= exported
    assert set(jfa.EXPORTED) <= exported


def test_binding_constants_match_the_header(jfa):
    """The binding restates a few of the header's numbers; they must agree."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+JFA_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "JFA_STATIC_SCRATCH_BYTES not found in the header"
    assert jfa.JFA_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
    body = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(JFA_[A-Z0-9_]+)\s*=\s*(\d+)", body))
    for name, value in enums.items():
        assert getattr(jfa, name) == value, name


def test_status_strings(jfa):
    for s in range(8):
        assert jfa.jfa_status_string(s) and jfa.jfa_status_string(s) != "unknown status"
    assert jfa.jfa_status_string(99) == "unknown status"


def visited_fwd(q_len, kv_len, t, causal):
    """Brute force: key tiles that hold at least one allowed (row, key) pair for query
    tile t (bottom-right causal)."""
    rows = range(t * BM_FWD, min(q_len, (t + 1) * BM_FWD))
    n = 0
    for kt in range((kv_len + BN_FWD - 1) // BN_FWD):
        cols = range(kt * BN_FWD, min(kv_len, (kt + 1) * BN_FWD))
        if any((not causal) or c <= r + kv_len - q_len for r in rows for c in (cols[0],)):
            n = kt + 1
    return n


def tiles_np(q_len, kv_len, tile, causal):
    """Vectorised closed form of the forward tile count (checked against the brute
    force `visited_fwd` in test_tile_count_closed_form)."""
    q_len, kv_len, tile = (np.asarray(a, dtype=np.int64) for a in (q_len, kv_len, tile))
    n = (kv_len + BN_FWD - 1) // BN_FWD
    if causal:
        last = np.minimum(q_len, (tile + 1) * BM_FWD) - 1
        max_col = last + kv_len - q_len
        n = np.where(max_col < 0, 0, np.minimum(n, max_col // BN_FWD + 1))
    return np.where(tile * BM_FWD < q_len, n, 0)


def test_tile_count_closed_form():
    rng = np.random.default_rng(0)
    for _ in range(300):
        q, kv = int(rng.integers(0, 700)), int(rng.integers(0, 700))
        for t in range(0, 7):
            for causal in (False, True):
                want = visited_fwd(q, kv, t, causal) if t * BM_FWD < q else 0
                assert tiles_np(q, kv, t, causal) == want, (q, kv, t, causal)


def visited_bwd(q_len, kv_len, t, causal):
    """Brute force: query tiles (128 rows) with at least one allowed pair for key tile t."""
    cols = range(t * BN_BWD, min(kv_len, (t + 1) * BN_BWD))
    tiles = set()
    for r in range(q_len):
        if (not causal) or cols[0] <= r + kv_len - q_len:
            tiles.add(r // BM_BWD)
    if not tiles:
        return 0, None
    # the kernel visits a contiguous range ending at the last query tile
    assert max(tiles) == (q_len - 1) // BM_BWD
    assert tiles == set(range(min(tiles), max(tiles) + 1))
    return len(tiles), min(tiles)


CASES = [
    ([0, 1, 127, 128, 129, 300, 5], [4, 1, 127, 128, 129, 300, 0]),
    ([3, 200, 64, 1], [700, 130, 1, 257]),
    ([1000, 1, 513], [1000, 1, 513]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("pass_", [0, 1, 2])
@pytest.mark.parametrize("n_ctas", [1, 3, 148])
def test_worklist_covers_every_tile_once(jfa, case, causal, pass_, n_ctas):
    q, kv = CASES[case]
    H = 3
    qo, ko = wl.offsets(q), wl.offsets(kv)
    items, offs, cost = jfa.jfa_worklist_build(qo, ko, H, causal, pass_, n_ctas)
    assert offs[0] == 0 and offs[-1] == len(items) and np.all(np.diff(offs) >= 0)
    expect = {}
    for b in range(len(q)):
        L = kv[b] if pass_ == 1 else q[b]
        T = {0: PAIR_FWD, 1: BN_BWD, 2: BM_FWD}[pass_]
        for h in range(H):
            for t in range((L + T - 1) // T):
                if pass_ == 2:
                    # dQ: one query tile, the forward's key tiles
                    expect[(b, h, t)] = visited_fwd(q[b], kv[b], t, causal)
                elif pass_ == 0:
                    # a pair of query tiles streams the larger of the two tiles' counts
                    nb = visited_fwd(q[b], kv[b], 2 * t + 1, causal) if (2 * t + 1) * BM_FWD < q[b] else 0
                    expect[(b, h, t)] = max(visited_fwd(q[b], kv[b], 2 * t, causal), nb)
                else:
                    n, first = visited_bwd(q[b], kv[b], t, causal)
                    expect[(b, h, t)] = n
                    if n:
                        assert first == (q[b] + BM_BWD - 1) // BM_BWD - n
    got = {(int(i[0]), int(i[1]), int(i[2])): int(i[3]) for i in items}
    assert len(got) == len(items), "duplicate work items"
    assert got == expect


@pytest.mark.parametrize("name", ["causal_bias", "long_causal", "cross"])
def test_worklist_is_balanced_and_group_major(jfa, name):
    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    qo, ko = wl.offsets(q), wl.offsets(kv)
    for pass_ in (0, 1, 2):
        items, offs, cost = jfa.jfa_worklist_build(qo, ko, w.H, w.causal, pass_, 148)
        if pass_ == 0:
            qi, ki, t = q[items[:, 0]], kv[items[:, 0]], items[:, 2].astype(np.int64)
            c = 2 * (tiles_np(qi, ki, 2 * t, w.causal) + tiles_np(qi, ki, 2 * t + 1, w.causal)) + 2
        elif pass_ == 1:
            c = 4 * items[:, 3].astype(np.int64) + 2
        else:
            qi, ki, t = q[items[:, 0]], kv[items[:, 0]], items[:, 2].astype(np.int64)
            assert np.array_equal(items[:, 3], tiles_np(qi, ki, t, w.causal))
            c = 3 * items[:, 3].astype(np.int64) + 2
        gid = items[:, 0].astype(np.int64) * w.H + items[:, 1]
        gcost = {}
        for g, x in zip(gid.tolist(), c.tolist()):
            gcost[g] = gcost.get(g, 0) + x
        for k in range(148):
            seg = slice(offs[k], offs[k + 1])
            # per-CTA cost matches the items assigned to it
            assert c[seg].sum() == cost[k]
            # a CTA runs its items group by group, largest groups first
            gs = [gcost[g] for g in gid[seg].tolist()]
            assert all(a >= b for a, b in zip(gs, gs[1:]))
        # greedy list scheduling: no CTA exceeds the least loaded one by more than the
        # largest item
        assert cost.max() - cost.min() <= c.max()
        assert cost.sum() == c.sum()


def test_worklist_rejects_bad_offsets(jfa):
    with pytest.raises(jfa.JFAError) as e:
        jfa.jfa_worklist_build([0, 5, 3], [0, 1, 2], 2, False, 0, 4)
    assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    with pytest.raises(jfa.JFAError):
        jfa.jfa_worklist_build([1, 5], [0, 1], 2, False, 0, 4)
    with pytest.raises(jfa.JFAError):
        jfa.jfa_worklist_size([0, 5], [0, 1], 0, False, 0)


def test_empty_batches(jfa):
    items, offs, cost = jfa.jfa_worklist_build([0], [0], 4, True, 0, 8)
    assert len(items) == 0 and np.all(offs == 0) and np.all(cost == 0)
    items, offs, cost = jfa.jfa_worklist_build([0, 0, 0], [0, 5, 5], 2, True, 1, 8)
    # the key tile still gets an item (with 0 query tiles) so its gradients are written
    assert len(items) == 2 and np.all(items[:, 3] == 0)


def test_worklist_is_deterministic(jfa):
    q, kv = wl.lengths(wl.WORKLOADS["cross"])
    qo, ko = wl.offsets(q), wl.offsets(kv)
    a = jfa.jfa_worklist_build(qo, ko, 8, False, 0, 148)
    b = jfa.jfa_worklist_build(qo, ko, 8, False, 0, 148)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_binding_refuses_non_contiguous_tensors():
    # the library takes dense row-major arrays; a strided view would be misread
    import torch
    from jagged_sequence_attention_gb300 import jfa
    t = torch.zeros(4, 6)
    assert jfa._ptr(t) is not None
    with pytest.raises(jfa.JFAError) as e:
        jfa._ptr(t.t())
    assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    assert jfa._ptr(None) is None


def test_planning_without_a_gpu_fails_loudly():
    # no CPU fallback: with no CUDA device, plan creation (and so every call and the autograd
    # form) raises -- the library's NO_DEVICE, or CUDA's own error when the binding asks for the
    # current stream first -- instead of computing anything on the host
    import torch
    from jagged_sequence_attention_gb300 import jfa
    if torch.cuda.is_available():
        pytest.skip("checks the behaviour without a GPU")
    with pytest.raises((jfa.JFAError, RuntimeError)) as e:
        jfa.jfa_plan_create([0, 3, 5], [0, 4, 9], 2, 64)
    if isinstance(e.value, jfa.JFAError):
        assert e.value.status == jfa.JFA_ERR_NO_DEVICE
    Q = torch.zeros(5, 2, 64, dtype=torch.bfloat16, requires_grad=True)
    K = torch.zeros(9, 2, 64, dtype=torch.bfloat16, requires_grad=True)
    with pytest.raises((jfa.JFAError, RuntimeError)):
        jfa.jagged_attention(Q, K, K, [0, 3, 5], [0, 4, 9])


def test_worklist_of_the_short_query_pass(jfa):
    # pass 3: one item per (sequence, head) with a query or a key, visiting all of the
    # sequence's key tiles; the pass has no causal or windowed form
    q = [0, 3, 0, 64, 1]
    kv = [0, 0, 129, 256, 1000]
    qo, ko = np.cumsum([0] + q), np.cumsum([0] + kv)
    items, offs, cost = jfa.jfa_worklist_build(qo, ko, 2, False, 3, 3)
    got = sorted(map(tuple, items.tolist()))
    want = sorted((s, h, 0, -(-kv[s] // 128)) for s in range(5) for h in range(2) if q[s] or kv[s])
    assert got == want
    assert offs[0] == 0 and offs[-1] == len(want)
    # LPT: every CTA within one item's cost of the least loaded one
    assert cost.max() - cost.min() <= 5 * 8 + 2
    with pytest.raises(jfa.JFAError):
        jfa.jfa_worklist_build(qo, ko, 2, True, 3, 3)
