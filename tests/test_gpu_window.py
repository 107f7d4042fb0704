"""Sliding-window parity of the CUDA path (through the C-ABI) against the CPU oracle:
query i attends to keys i' - W .. i', i' = i + kv_len - q_len (causal), and the kernels
skip every tile outside the band.  Windows below, at and above the 128-row tile size,
lengths at tile boundaries, q > kv and q < kv, every mode, both output types, both head
dims of the tensor-core path and the fp32 CUDA-core path; a long sequence is checked on
sampled rows."""
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


def check_full(batch, out_dtype=torch.float32):
    g = parity.run_gpu(batch, True, out_dtype=out_dtype)
    assert g["status"] == 0, g["status"]
    r = parity.run_oracle(batch, True)
    m = parity.compare(g, r, softmax=batch.mode == "softmax", with_backward=True)
    print(batch.name, batch.window, m)
    parity.assert_within(m, softmax=batch.mode == "softmax")
    return g, r


LENS = [1, 37, 127, 128, 129, 255, 256, 257, 700, 1100]


@pytest.mark.parametrize("W", [1, 100, 127, 128, 129, 300, 1000, 5000])
def test_window_softmax_bias(W):
    check_full(wl.make_custom(LENS, LENS, H=2, D=128, causal=True, bias=True, device="cuda", seed=21, window=W))


def test_window_zero_single_key():
    """W = 0 leaves one key per row: O = V at the aligned key, dV sums dO, and dQ, dK are
    exactly zero (ds = p (dp - p dp) with p = 1).  Relative errors of dQ, dK are undefined
    against zero, so they are bounded absolutely: what remains is the rounding of dP - Delta
    (a bf16 x bf16 -> fp32 product against the fp32 row term), about |dp| 2^-17."""
    b = wl.make_custom(LENS, LENS, H=2, D=128, causal=True, bias=True, device="cuda", seed=21, window=0)
    g = parity.run_gpu(b, True, out_dtype=torch.float32)
    assert g["status"] == 0
    r = parity.run_oracle(b, True)
    assert np.all(r["dQ"] == 0) and np.all(r["dK"] == 0)
    m = parity.compare(g, r, softmax=True, with_backward=True)
    for k in ("dQ_rel_frob", "dK_rel_frob"):
        m.pop(k)
    parity.assert_within(m)
    for k in ("dQ", "dK"):
        assert float(g[k].abs().max()) <= 2e-3, (k, float(g[k].abs().max()))


@pytest.mark.parametrize("W", [63, 300])
def test_window_asymmetric_lengths(W):
    # q > kv leaves rows that see no key; q < kv shifts every row's band
    q, kv = [200, 64, 900, 5, 300], [500, 64, 700, 1, 129]
    check_full(wl.make_custom(q, kv, H=3, D=128, causal=True, bias=True, device="cuda", seed=22, window=W))


@pytest.mark.parametrize("mode", ["gelu_tanh", "silu"])
def test_window_gdpa(mode):
    check_full(wl.make_custom(LENS, LENS, H=2, D=128, mode=mode, causal=True, bias=True, value_std=0.5,
                              device="cuda", seed=23, window=200))


def test_window_bf16_output():
    check_full(wl.make_custom(LENS, LENS, H=2, D=128, causal=True, bias=True, device="cuda", seed=24, window=150),
               out_dtype=torch.bfloat16)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 32), (torch.float32, 64)])
def test_window_other_head_dims(dtype, D):
    check_full(wl.make_custom([7, 130, 64, 300], [7, 130, 64, 300], H=2, D=D, dtype=dtype, causal=True, bias=True,
                              device="cuda", seed=25, window=90))


def test_window_long_sequence_sampled():
    # 12k tokens: most tiles are interior band tiles; checked on suffix sub-problems
    b = wl.make_custom([12000, 3000], [12000, 3000], H=4, D=128, causal=True, bias=True, device="cuda", seed=26,
                       window=1500)
    g = parity.run_gpu(b, out_dtype=torch.bfloat16)
    assert g["status"] == 0
    samples = [(0, 0, 11800), (0, 3, 9000), (1, 1, 2000)]
    m = parity.sampled_parity(b, g, samples)
    print(m)
    parity.assert_within(m)
