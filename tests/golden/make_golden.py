"""Writes tests/golden/oracle_small.json: the oracle's outputs on a few tiny seeded batches.

The pages print no worked numerical example of jagged attention, so no fixture here holds
the pages' own numbers.  These values come from the oracle alone (this script imports only
`oracle` and the seeded input generator).  They guard the oracle against silent change:
a later edit of its arithmetic must either reproduce them or regenerate them, in a commit
that names the passage that justifies it.  The oracle is pinned against independent
references in tests/test_oracle*.py.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from jagged_sequence_attention_gb300 import workloads as wl  # noqa: E402

CASES = [
    # name, q_lens, kv_lens, H, D, mode, causal, window, bias, dense
    ("softmax_causal_bias", [3, 1, 5], [3, 2, 5], 2, 4, "softmax", True, None, True, False),
    ("softmax_cross", [2, 4], [5, 3], 1, 4, "softmax", False, None, False, False),
    ("gelu_window", [6, 2], [6, 4], 2, 4, "gelu_tanh", True, 2, True, False),
    ("silu_dense", [3, 2], [4, 2], 1, 4, "silu", False, None, False, True),
]


def case_inputs(q, kv, H, D, bias, dense, seed):
    g = torch.Generator().manual_seed(seed)
    qo, ko = wl.offsets(q), wl.offsets(kv)
    Q = torch.randn(int(qo[-1]), H, D, generator=g, dtype=torch.float64) * 0.8
    K = torch.randn(int(ko[-1]), H, D, generator=g, dtype=torch.float64) * 0.8
    V = torch.randn(int(ko[-1]), H, D, generator=g, dtype=torch.float64)
    dO = torch.randn(int(qo[-1]), H, D, generator=g, dtype=torch.float64)
    b = torch.randn(H, 32, generator=g, dtype=torch.float64) * 0.5 if bias else None
    P = sum(a * c for a, c in zip(q, kv))
    dn = torch.randn(H, P, generator=g, dtype=torch.float64) * 0.5 if dense else None
    return qo, ko, Q, K, V, dO, b, dn


def run_case(name, q, kv, H, D, mode, causal, window, bias, dense, seed):
    qo, ko, Q, K, V, dO, b, dn = case_inputs(q, kv, H, D, bias, dense, seed)
    kw = dict(mode=mode, causal=causal, window=window, scale=0.5, bias=None if b is None else b.numpy(),
              dense_bias=None if dn is None else dn.numpy())
    O, lse = oracle.fwd(qo, ko, Q.numpy(), K.numpy(), V.numpy(), **kw)
    dQ, dK, dV, dtab, ddense = oracle.bwd(qo, ko, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), bias_grads=True, **kw)
    return {"O": O, "lse": lse, "dQ": dQ, "dK": dK, "dV": dV, "dbias": dtab, "ddense": ddense}


def main():
    out = {}
    for i, c in enumerate(CASES):
        res = run_case(*c, seed=500 + i)
        out[c[0]] = {k: np.where(np.isfinite(v), v, 0.0).tolist() if v is not None else None for k, v in res.items()}
        out[c[0]]["lse_finite"] = np.isfinite(res["lse"]).tolist()
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json"), "w") as f:
        json.dump(out, f)


if __name__ == "__main__":
    main()
