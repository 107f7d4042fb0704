"""The benchmark's JSON line, checked on the CPU.

- The reference arm (the oracle, on the host cores) runs anywhere and prints one JSON line:
  the metric, its value, the run's configuration, the CPU-baseline description and an
  end-to-end object with no host/device copies.
- Our arm needs the CUDA path. Without a GPU it must fail loudly, with a non-zero exit and
  no JSON line, rather than fall back to anything on the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["data"] == "synthetic" and d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_under_two_ranks_prints_once():
    """Launched as two ranks, rank 0 alone runs the oracle and prints; the other rank exits 0."""
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29541", os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_our_arm_fails_loudly_without_a_gpu():
    r = run_bench("--workload", "tiny", "--steps", "1", "--warmup", "3", timeout=300)
    assert r.returncode != 0
    assert not any(ln.strip().startswith("{") for ln in r.stdout.splitlines())


def test_sample_errors_apply_the_parity_tolerances():
    """The bench line's error report on the oracle's sample uses the parity tests' bounds."""
    import numpy as np
    import bench
    rng = np.random.default_rng(0)
    ref = {k: rng.standard_normal((50, 2, 8)) for k in ("O", "dQ", "dK", "dV")}
    ref["lse"] = rng.standard_normal((50, 2))
    got = {k: v.copy() for k, v in ref.items()}
    e = bench.sample_errors(got, ref, True)
    assert e["within_tolerance"] and e["O_max_abs"] == 0.0 and e["dK_rel_frob"] == 0.0
    got["dQ"] = ref["dQ"] * 2.0  # a dQ counted twice
    assert not bench.sample_errors(got, ref, True)["within_tolerance"]
    got = {k: v.copy() for k, v in ref.items()}
    got["O"] = ref["O"] + 0.05  # beyond the forward's max-abs bound
    assert not bench.sample_errors(got, ref, True)["within_tolerance"]


def test_oracle_sample_is_the_same_problem():
    """The bench's oracle sample (its CPU baseline and parity check) keeps every property of
    the workload: on a sliding-window batch it must compute windowed attention."""
    import dataclasses
    import numpy as np
    import bench
    from jagged_sequence_attention_gb300 import workloads as wl
    b = wl.make_custom([40, 90, 70], [40, 90, 70], H=2, D=32, dtype=torch.float32, causal=True, bias=True,
                       window=16, device="cpu", seed=21)
    cpu, seqs = bench.oracle_sample(b, 1.0)
    assert cpu.window == 16 and cpu.causal and cpu.bias is not None
    got = {}
    bench.run_oracle_once(cpu, got)
    plain = {}
    bench.run_oracle_once(dataclasses.replace(cpu, window=None), plain)
    sub = wl.subset(b, seqs)
    ref = {}
    bench.run_oracle_once(sub, ref)
    assert np.array_equal(got["O"], ref["O"]) and np.array_equal(got["dQ"], ref["dQ"])
    assert not np.allclose(got["O"], plain["O"])  # the window changes the result
