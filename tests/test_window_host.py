"""Sliding-window work lists (host only): every pass of the planner visits exactly the
tiles that hold at least one allowed (query, key) pair of the band i' - W <= j <= i',
i' = i + kv_len - q_len, checked by brute force over the pairs."""
import numpy as np
import pytest

from jagged_sequence_attention_gb300 import _build
from jagged_sequence_attention_gb300 import workloads as wl

T = 128


@pytest.fixture(scope="module")
def jfa():
    _build.build()
    from jagged_sequence_attention_gb300 import jfa as m
    m.lib()
    return m


def allowed(q_len, kv_len, W):
    i = np.arange(q_len)[:, None]
    j = np.arange(kv_len)[None, :]
    ip = i + (kv_len - q_len)
    return (j <= ip) & (j >= ip - W)


def key_tiles_of_query_tile(a, t):
    rows = a[t * T:(t + 1) * T]
    cols = np.nonzero(rows.any(axis=0))[0]
    return sorted(set((cols // T).tolist()))


def query_tiles_of_key_tile(a, kt):
    cols = a[:, kt * T:(kt + 1) * T]
    rows = np.nonzero(cols.any(axis=1))[0]
    return sorted(set((rows // T).tolist()))


CASES = [([300, 1000, 129, 5, 640], [300, 1000, 129, 5, 640]),
         ([200, 64, 900], [500, 64, 700])]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("W", [0, 1, 63, 127, 128, 300, 5000])
def test_windowed_worklists_visit_exactly_the_band(jfa, case, W):
    q, kv = CASES[case]
    H = 2
    qo, ko = wl.offsets(q), wl.offsets(kv)
    got = {p: {(int(i[0]), int(i[1]), int(i[2])): int(i[3]) for i in jfa.jfa_worklist_build(qo, ko, H, True, p, 7,
                                                                                               window=W)[0]}
           for p in (0, 1, 2)}
    for b in range(len(q)):
        a = allowed(q[b], kv[b], W)
        nqt, nkt = (q[b] + T - 1) // T, (kv[b] + T - 1) // T
        for h in range(H):
            for t in range(nqt):
                tiles = key_tiles_of_query_tile(a, t)
                # contiguous band of key tiles; the dQ pass visits exactly those
                assert tiles == list(range(tiles[0], tiles[-1] + 1)) if tiles else True
                assert got[2][(b, h, t)] == len(tiles), (b, t, W)
            for p_ in range((q[b] + 2 * T - 1) // (2 * T)):
                ta = key_tiles_of_query_tile(a, 2 * p_)
                tb = key_tiles_of_query_tile(a, 2 * p_ + 1) if (2 * p_ + 1) * T < q[b] else []
                union = sorted(set(ta) | set(tb))
                assert union == list(range(union[0], union[-1] + 1)) if union else True
                assert got[0][(b, h, p_)] == len(union), (b, p_, W)
            for kt in range(nkt):
                tiles = query_tiles_of_key_tile(a, kt)
                assert tiles == list(range(tiles[0], tiles[-1] + 1)) if tiles else True
                assert got[1][(b, h, kt)] == len(tiles), (b, kt, W)


def test_window_needs_causal_and_a_valid_size(jfa):
    qo = ko = wl.offsets([10, 20])
    for causal, W in ((False, 5), (True, -2)):
        with pytest.raises(jfa.JFAError) as e:
            jfa.jfa_worklist_size(qo, ko, 2, causal, 0, window=W)
        assert e.value.status == jfa.JFA_ERR_INVALID_ARG
    assert jfa.jfa_worklist_size(qo, ko, 2, True, 0, window=0) == 2 * 2


def test_window_reduces_partition_cost(jfa):
    w = wl.WORKLOADS["long_causal"]
    q, kv = wl.lengths(w)
    _, full = jfa.jfa_partition_sequences(wl.offsets(q), wl.offsets(kv), w.H, True, 4)
    _, band = jfa.jfa_partition_sequences(wl.offsets(q), wl.offsets(kv), w.H, True, 4, window=2048)
    assert band.sum() * 4 < full.sum()
