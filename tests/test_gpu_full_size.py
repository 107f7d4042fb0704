"""Full-size backward parity: complete outputs of benchmark-size launches against the
oracle (aihot GEM article, "Jagged Sequence Flash Attention": the efficient backward
pass on jagged tensors).

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
