"""CPU check of the row-block split that the full-size GPU test uses to run the oracle
on one long causal sequence in parallel: the blocks reproduce the oracle on the whole
sequence (outputs and all three gradients) to fp64 rounding."""
import numpy as np

import oracle
import parity
from jagged_sequence_attention_gb300 import workloads as wl


def test_row_block_split_is_exact():
    """The split above reproduces the oracle on the whole sequence (small case, CPU)."""
    rng = np.random.default_rng(3)
    L, D = 300, 16
    Q, K, V, dO = (rng.standard_normal((L, D)) for _ in range(4))
    bias = rng.standard_normal((1, 32)) * 0.1
    got = parity.causal_head_oracle(Q, K, V, dO, bias, 0.25, n_blocks=7)
    off = wl.offsets([L])
    O, LSE = oracle.fwd(off, off, Q[:, None], K[:, None], V[:, None], causal=True, bias=bias, scale=0.25)
    dQ, dK, dV = oracle.bwd(off, off, Q[:, None], K[:, None], V[:, None], dO[:, None], causal=True, bias=bias,
                            scale=0.25)
    for name, ref in (("O", O[:, 0]), ("lse", LSE[:, 0]), ("dQ", dQ[:, 0]), ("dK", dK[:, 0]), ("dV", dV[:, 0])):
        assert np.allclose(got[name], ref, rtol=0, atol=1e-12), name
