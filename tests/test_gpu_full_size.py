"""Full-size backward parity: complete outputs of benchmark-size launches against the
oracle (aihot GEM article, "Jagged Sequence Flash Attention": the efficient backward
pass on jagged tensors; "Generalized Dot-Product Attention (GDPA)" for the GDPA batches).

The sampled full-size tests elsewhere compare suffix rows only, so the dK/dV they check
belong to keys that few query tiles see.  Here every row and every key of one head of
the longest sequence of the long causal workload is compared, including the first key
tiles, which all of the sequence's query tiles visit, and the full shared key/value
batch, where up to 64 query sets add into each user's dK/dV.  Both run once with O in
fp32, under the plain bounds, and once with O in bf16, the launch the benchmark times,
under the bound that allows for O's own final rounding.

The long sequence is one (sequence, head) problem, and the oracle parallelises over
those, so parity.causal_head_oracle splits its rows into blocks, one sub-problem each;
the split is exact (see there, and its CPU test in test_oracle_row_blocks.py)."""
import numpy as np
import pytest
import torch

import parity
from jagged_sequence_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def long_causal():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return wl.make("long_causal", device="cuda")


def _metrics(got, ref, o_bf16):
    m = {"O_max_abs": parity.max_abs(got["O"], ref["O"]), "O_rel_frob": parity.rel_frob(got["O"], ref["O"]),
         "O_bf16": o_bf16, "O_max_abs_beyond_rounding": parity.beyond_rounding(got["O"], ref["O"])}
    fin = np.isfinite(ref["lse"])
    m["lse_nonfinite_match"] = bool(np.array_equal(fin, np.isfinite(got["lse"])))
    m["lse_max_abs"] = parity.max_abs(got["lse"][fin], ref["lse"][fin])
    for k in ("dQ", "dK", "dV"):
        m[f"{k}_rel_frob"] = parity.rel_frob(got[k], ref[k])
    return m


@pytest.mark.parametrize("h", [3])
def test_long_causal_longest_sequence_one_head_in_full(long_causal, h):
    batch = long_causal
    b = int(np.argmax(batch.q_lens))
    q0, q1 = int(batch.q_off[b]), int(batch.q_off[b + 1])
    L = q1 - q0
    assert L > 30000 and int(batch.kv_off[b + 1]) - int(batch.kv_off[b]) == L
    runs = {}
    for o_dtype in (torch.float32, torch.bfloat16):
        g = parity.run_gpu(batch, out_dtype=o_dtype)  # the whole batch, as the benchmark launches it
        assert g["status"] == 0
        runs[o_dtype] = {k: parity.np64(g[k][q0:q1, h]) for k in ("O", "lse", "dQ", "dK", "dV")}
        for k in ("O", "dQ", "dK", "dV"):
            assert torch.isfinite(g[k]).all(), k
        del g
        torch.cuda.empty_cache()
    x = lambda t: parity.np64(t[q0:q1, h])  # noqa: E731
    ref = parity.causal_head_oracle(x(batch.Q), x(batch.K), x(batch.V), x(batch.dO),
                                    parity.np64(batch.bias[h:h + 1]), batch.scale)
    for o_dtype, got in runs.items():
        m = _metrics(got, ref, o_dtype == torch.bfloat16)
        print("long_causal", b, L, h, o_dtype, m)
        parity.assert_within(m)
    # the first key tile: every query tile of the sequence adds into its dK/dV
    for o_dtype, got in runs.items():
        for k in ("dK", "dV"):
            err = parity.rel_frob(got[k][:128], ref[k][:128])
            assert err <= parity.BWD_REL_FROB, (o_dtype, k, err)


def test_ikbo_cross_full_batch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    batch = wl.make("ikbo_cross", device="cuda")
    ref = parity.run_oracle(batch)  # the broadcast definition over all 1024 query sets
    for o_dtype in (torch.float32, torch.bfloat16):
        g = parity.run_gpu(batch, out_dtype=o_dtype)
        assert g["status"] == 0
        m = parity.compare(g, ref)
        print("ikbo_cross", o_dtype, m)
        parity.assert_within(m)


def test_cross_full_batch():
    """The whole cross-attention workload (512 query sets of up to 64 rows over key/value
    histories of up to 16K rows) against the oracle, every output compared: the short-query
    forward with two key tiles per score tile and the short-query backward, as the benchmark
    launches them (bf16 O) and with fp32 O."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import jfa
    batch = wl.make("cross", device="cuda")
    ref = parity.run_oracle(batch)
    for o_dtype in (torch.float32, torch.bfloat16):
        g = parity.run_gpu(batch, out_dtype=o_dtype)
        assert g["status"] == 0
        info = jfa.jfa_plan_info(g["plan"])
        assert info["fwd_short"] == 64 and info["bwd_short"] == 64
        m = parity.compare(g, ref)
        print("cross", o_dtype, m)
        parity.assert_within(m)


def _full_batch(name, expect):
    """A named workload's whole batch against the oracle, every output of every sequence
    and head compared, once with O in fp32 (plain bounds) and once with O in bf16 (the
    launch the benchmark times; the bound allows for O's own rounding).  `expect`: plan
    facts that pin the kernels the benchmark runs on this workload."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import jfa
    batch = wl.make(name, device="cuda")
    softmax = batch.mode == "softmax"
    ref = parity.run_oracle(batch)
    for o_dtype in (torch.float32, torch.bfloat16):
        g = parity.run_gpu(batch, out_dtype=o_dtype)
        assert g["status"] == 0
        info = jfa.jfa_plan_info(g["plan"])
        for k, v in expect.items():
            assert info[k] == v, (k, info[k], v)
        m = parity.compare(g, ref, softmax=softmax)
        print(name, o_dtype, m)
        parity.assert_within(m, softmax=softmax)


def test_causal_bias_full_batch():
    """256 causal sequences of 32 to 2,048 tokens with the relative-position bias, 8 heads:
    the query-tile forward and the fused backward (every key tile's part of dQ added into
    the fp32 accumulator)."""
    _full_batch("causal_bias", {"bwd_fused": 1, "bwd_short": 0, "fwd_short": 0})


@pytest.mark.parametrize("name", ["gdpa_gelu", "gdpa_silu"])
def test_gdpa_full_batch(name):
    """1,024 query sets of 1 to 128 rows over 64 to 4,096 keys, 4 heads, no normalisation:
    the transposed short-query forward and the short-query backward."""
    _full_batch(name, {"bwd_short": 128, "fwd_short": 128})


def test_long_causal_shortest_sequence_all_heads_in_full(long_causal):
    """The shortest sequence of the long causal workload, every head, every row and key,
    from the benchmark's whole-batch launch (bf16 O, and fp32 O)."""
    batch = long_causal
    b = int(np.argmin(batch.q_lens))
    q0, q1 = int(batch.q_off[b]), int(batch.q_off[b + 1])
    assert (int(batch.kv_off[b]), int(batch.kv_off[b + 1])) == (q0, q1)  # self-attention: same rows
    runs = {}
    for o_dtype in (torch.float32, torch.bfloat16):
        g = parity.run_gpu(batch, out_dtype=o_dtype)
        assert g["status"] == 0
        runs[o_dtype] = {k: g[k][q0:q1] for k in ("O", "lse", "dQ", "dK", "dV")}
        del g
        torch.cuda.empty_cache()
    ref = parity.run_oracle(wl.subset(batch, [b]))
    for o_dtype, got in runs.items():
        m = parity.compare(got, ref)
        print("long_causal shortest", b, q1 - q0, o_dtype, m)
        parity.assert_within(m)
