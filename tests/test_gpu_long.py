"""A 100,003-token sequence on the GPU (through the C-ABI) against the CPU oracle, on
sampled suffix rows.

This exercises:
- relative positions past the bucket cap (bucket 31 from r = 46,340);
- TMA coordinates and row offsets near 10^5 x H x D;
- the planner on a single sequence far longer than the benchmark's longest.

The oracle computes the last ~100 query rows of each sampled head exactly, with all of
their keys, and the dK, dV of the keys that only those rows see."""
import pytest
import torch

from jagged_sequence_attention_gb300 import workloads as wl

import parity

pytestmark = pytest.mark.gpu

L = 100_003


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from jagged_sequence_attention_gb300 import _build
    _build.build()


@pytest.mark.parametrize("window", [None, 3000])
def test_one_very_long_sequence(window):
    b = wl.make_custom([L, 77], [L, 77], H=2, D=128, causal=True, bias=True, device="cuda", seed=93, window=window)
    g = parity.run_gpu(b, out_dtype=torch.bfloat16)
    assert g["status"] == 0
    m = parity.sampled_parity(b, g, [(0, 0, L - 100), (0, 1, L - 37), (1, 0, 0), (1, 1, 40)])
    print(window, m)
    parity.assert_within(m)
