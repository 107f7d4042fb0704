"""Dense per-pair bias ([H, sum q_len * kv_len], JFA_BIAS_DENSE) on the GPU, through the
C-ABI, against the CPU oracle.  Forward, backward and the bias's own gradient (dS at
every allowed pair, exactly 0 at masked ones).

Cases:
- causal self-attention over lengths at and around the tile size;
- non-causal q_len != kv_len (rows whose keys run past the tile edges);
- a sliding window;
- both GDPA activations;
- the fp32 CUDA-core path;
- the 64-wide head;
- a bf16 output;
- short queries against long keys, the shape this bias is meant for.

A dense bias expanded from the bucket table must give the table's results."""
import numpy as np
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()


def check(batch, out_dtype=torch.float32):
    from jagged_sequence_attention_gb300 import jfa
    out = jfa.attention(batch, with_backward=True, out_dtype=out_dtype, bias_grad=True)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(out["plan"]) == 0
    assert jfa.jfa_plan_info(out["plan"])["pairs"] == batch.dense.shape[1]
    r = parity.run_oracle(batch, True, bias_grads=True)
    m = parity.compare(out, r, softmax=batch.mode == "softmax", with_backward=True)
    g = parity.np64(out["dbias"])
    m["ddense_rel_frob"] = parity.rel_frob(g, r["dbias"])
    # masked pairs: exactly zero
    m["ddense_masked_nonzero"] = int(np.count_nonzero(g[r["dbias"] == 0]))
    print(batch.name, m)
    parity.assert_within(m, softmax=batch.mode == "softmax")
    assert m["ddense_rel_frob"] <= parity.BWD_REL_FROB, m
    return out, r


LENS = [1, 37, 127, 128, 129, 255, 256, 257, 700]


@pytest.mark.parametrize("mode", ["softmax", "gelu_tanh", "silu"])
def test_causal(mode):
    out, r = check(wl.make_custom(LENS, LENS, H=2, D=128, mode=mode, causal=True, dense_bias=True,
                                  value_std=1.0 if mode == "softmax" else 0.5, device="cuda", seed=41))
    # the gradient above the diagonal (masked pairs) is exactly zero
    g = out["dbias"].cpu().numpy()
    po = wl.pair_offsets(wl.offsets(LENS), wl.offsets(LENS))
    for b, L in enumerate(LENS):
        blk = g[:, po[b]:po[b + 1]].reshape(2, L, L)
        assert np.all(np.triu(blk, k=1) == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_asymmetric(causal):
    q, kv = [200, 64, 500, 5, 300, 1], [300, 64, 400, 1, 129, 40]
    check(wl.make_custom(q, kv, H=3, D=128, causal=causal, dense_bias=True, device="cuda", seed=42))


def test_window():
    check(wl.make_custom(LENS, LENS, H=2, D=128, causal=True, dense_bias=True, device="cuda", seed=43, window=150))


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 32), (torch.float32, 64)])
def test_other_head_dims_and_fp32(dtype, D):
    check(wl.make_custom([7, 130, 64, 300], [7, 130, 90, 300], H=2, D=D, dtype=dtype, causal=True,
                         dense_bias=True, device="cuda", seed=44))


def test_fp32_non_causal_gdpa():
    check(wl.make_custom([7, 130, 64], [40, 130, 9], H=2, D=32, dtype=torch.float32, mode="silu", causal=False,
                         dense_bias=True, value_std=0.5, device="cuda", seed=45))


def test_bf16_output():
    check(wl.make_custom(LENS, LENS, H=2, D=128, causal=True, dense_bias=True, device="cuda", seed=46),
          out_dtype=torch.bfloat16)


def test_short_queries_long_keys():
    g = np.random.default_rng(47)
    q = g.integers(1, 65, size=24).tolist()
    kv = g.integers(100, 2000, size=24).tolist()
    check(wl.make_custom(q, kv, H=4, D=64, causal=False, dense_bias=True, device="cuda", seed=47))


def test_dense_expanded_from_the_table_matches_the_table():
    from jagged_sequence_attention_gb300 import jfa
    q, kv = [300, 77, 129], [300, 90, 129]
    b = wl.make_custom(q, kv, H=2, D=128, causal=True, bias=True, device="cuda", seed=48)
    blocks = []
    for a, c in zip(q, kv):
        r = (np.arange(a)[:, None] + (c - a)) - np.arange(c)[None, :]
        r = np.abs(r)
        bucket = np.minimum(31, np.floor(np.log2((1.0 + r) ** 2)).astype(np.int64))
        blocks.append(b.bias.cpu().numpy()[:, bucket].reshape(2, a * c))
    dense_np = np.concatenate(blocks, axis=1)
    # numpy's fancy indexing may leave the expansion in column order: the library takes
    # row-major arrays only, and the binding refuses any other layout
    with pytest.raises(jfa.JFAError):
        jfa._ptr(torch.from_numpy(np.asfortranarray(dense_np)))
    dense = torch.from_numpy(np.ascontiguousarray(dense_np)).float().cuda()
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, b.mode, b.causal)
    O1, lse1 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, out_dtype=torch.float32)
    O2, lse2 = jfa.jfa_fwd(plan, b.Q, b.K, b.V, None, b.scale, out_dtype=torch.float32, dense_bias=dense)
    g1 = jfa.jfa_bwd_ex(plan, b.Q, b.K, b.V, O1, b.dO, lse1, b.bias, b.scale)
    g2 = jfa.jfa_bwd_ex(plan, b.Q, b.K, b.V, O2, b.dO, lse2, None, b.scale, dense_bias=dense)
    torch.cuda.synchronize()
    assert jfa.jfa_plan_device_status(plan) == 0
    d = (O1 - O2).abs().amax(dim=(1, 2))
    bad = torch.nonzero(d > 1e-2).flatten().tolist()
    print("O diff", float(d.max()), "rows", len(bad), bad[:8], bad[-4:], "lse diff", float((lse1 - lse2).abs().max()))
    # the two paths round differently (chunk-constant bias and a max bound, against an
    # exact per-element max); each is within the forward tolerance of the oracle, so
    # they are within twice that of each other
    assert float(d.max()) <= 2 * parity.FWD_MAX_ABS
    assert float((lse1 - lse2).abs().max()) <= 2 * parity.LSE_MAX_ABS
    for x, y in zip(g1[:3], g2[:3]):
        assert float((x.float() - y.float()).norm() / y.float().norm()) <= 2 * parity.BWD_REL_FROB
    # the table's gradient is the bucket-wise sum of the dense gradient
    dt = np.zeros((2, 32))
    po = wl.pair_offsets(b.q_off, b.kv_off)
    gd = g2[3].double().cpu().numpy()
    for s, (a, c) in enumerate(zip(q, kv)):
        r = np.abs((np.arange(a)[:, None] + (c - a)) - np.arange(c)[None, :])
        bucket = np.minimum(31, np.floor(np.log2((1.0 + r) ** 2)).astype(np.int64)).reshape(-1)
        for h in range(2):
            np.add.at(dt[h], bucket, gd[h, po[s]:po[s + 1]])
    d1 = g1[3].double().cpu().numpy()
    assert np.linalg.norm(dt - d1) <= 2 * parity.BWD_REL_FROB * np.linalg.norm(d1)


def test_argument_errors():
    from jagged_sequence_attention_gb300 import jfa
    b = wl.make_custom([10, 20], [10, 20], H=2, D=128, causal=True, bias=True, dense_bias=True, device="cuda",
                       seed=49)
    plan = jfa.jfa_plan_create(b.q_off, b.kv_off, b.H, b.D, b.mode, b.causal)
    with pytest.raises(jfa.JFAError):        # one bias kind at a time
        jfa.jfa_fwd(plan, b.Q, b.K, b.V, b.bias, b.scale, dense_bias=b.dense)
    st = jfa.lib().jfa_fwd(plan.handle, jfa.DTYPES[b.Q.dtype], jfa._ptr(b.Q), jfa._ptr(b.K), jfa._ptr(b.V),
                           jfa.JFA_BIAS_DENSE, None, b.scale, jfa._ptr(b.Q), jfa.DTYPES[b.Q.dtype],
                           jfa._ptr(torch.empty(30, 2, device="cuda")), None)
    assert st == jfa.JFA_ERR_INVALID_ARG      # a dense bias needs its array
    assert jfa.jfa_bwd_ex_workspace_size(plan, b.Q.dtype, dense=True) == jfa.jfa_bwd_workspace_size(plan, b.Q.dtype)
