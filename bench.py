#!/usr/bin/env python
"""Benchmark: jagged attention forward+backward TFLOP/s (unpadded FLOPs) on GB300.

One step = one forward and one backward pass over one seeded synthetic jagged batch
(the hot path end to end: planner output reused, forward kernel, backward
preprocess, backward main kernel, dQ convert).  Default workload: the long-sequence
causal self-attention batch (64 sequences, lengths U{4096..32768}, 8 heads,
head_dim 128, bf16, relative-position bias) -- the configuration the >=50%-of-peak
target names.  Every input tensor (~2.5 GB each) is larger than the 129 MB L2, so no
flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle instead, on a
bounded sample of the same workload.  Under torchrun each rank runs its own batch
(seeded per rank; weak scaling) with no collective in the data path.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from jagged_sequence_attention_gb300 import workloads as wl  # noqa: E402

METRIC = "jagged attention fwd+bwd TFLOPS (unpadded) and % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"


# ----------------------------------------------------------------------------- FLOPs / bytes


def allowed_pairs(q_lens, kv_lens, causal, window=None):
    q = np.asarray(q_lens, dtype=np.int64)
    kv = np.asarray(kv_lens, dtype=np.int64)
    if not causal:
        return int(np.sum(q * kv))
    tot = 0
    for a, b in zip(q.tolist(), kv.tolist()):
        # row i sees keys [max(0, i' - W), min(b - 1, i')], i' = i + b - a
        ip = np.arange(a, dtype=np.int64) + (b - a)
        hi = np.minimum(ip, b - 1)
        lo = np.zeros_like(ip) if window is None else np.maximum(ip - window, 0)
        tot += int(np.clip(hi - lo + 1, 0, None).sum())
    return tot


def flops_of(batch):
    pairs = allowed_pairs(batch.q_lens, batch.kv_lens, batch.causal, batch.window)
    fwd = 4.0 * batch.D * batch.H * pairs
    return fwd, 2.5 * fwd


def algorithmic_bytes(batch, elem=2, fused=False):
    """Compulsory HBM bytes of one launch of each tensor-core kernel: every input it
    reads and every output it writes, once.  A one-kernel backward (fused or
    short-query) reads Q, dO, K, V and writes dK, dV and dQ (the fused form's fp32 dQ
    accumulator is implementation traffic, not algorithmic)."""
    Tq, Tkv, H, D = int(batch.q_off[-1]), int(batch.kv_off[-1]), batch.H, batch.D
    # softmax row terms: the forward writes lse, the backward reads lse and Delta (GDPA has none)
    sm = batch.mode == "softmax"
    lse_b, rows_b = (4 * H * Tq, 8 * H * Tq) if sm else (0, 0)
    if fused:
        return {
            "fwd": elem * H * D * (2 * Tq + 2 * Tkv) + lse_b,          # Q,K,V -> O; lse
            "bwd_main": elem * H * D * (3 * Tq + 4 * Tkv) + rows_b,    # Q,dO,K,V -> dQ,dK,dV; lse,Delta
        }
    return {
        "fwd": elem * H * D * (2 * Tq + 2 * Tkv) + lse_b,              # Q,K,V -> O; lse
        "bwd_main": elem * H * D * (2 * Tq + 4 * Tkv) + rows_b,        # Q,dO,K,V -> dK,dV; lse,Delta
        "bwd_dq": elem * H * D * (3 * Tq + 2 * Tkv) + rows_b,          # Q,dO,K,V -> dQ; lse,Delta
    }


def kernel_flops(fwd_flop, fused=False):
    """Algorithmic FLOPs per launch of each tensor-core kernel.  The backward's five
    products (S, dP, dV, dK, dQ; 2.5x the forward's two) all run in a one-kernel backward
    (fused or short-query); on the two-pass backward they split as: dK/dV kernel S, dP, dV, dK (2x), dQ
    kernel the dQ product (0.5x), whose recomputed S and dP are not algorithmic work and
    are not counted."""
    if fused:
        return {"fwd": fwd_flop, "bwd_main": 2.5 * fwd_flop}
    return {"fwd": fwd_flop, "bwd_main": 2.0 * fwd_flop, "bwd_dq": 0.5 * fwd_flop}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# The source file of each tensor-core kernel; its digest also covers the shared headers.
KERNEL_SOURCE = {
    "jfa_fwd_kernel": "fwd.cu", "jfa_fwd_short_kernel": "fwd_short.cu", "jfa_fwd_pack_kernel": "fwd_pack.cu",
    "jfa_bwd_dkdv_kernel": "bwd.cu", "jfa_bwd_dq_kernel": "bwd_dq.cu", "jfa_bwd_fused_kernel": "bwd_fused.cu",
    "jfa_bwd_short_kernel": "bwd_short.cu",
}


def kernel_digest(kernel):
    """Digest of the sources a kernel is built from: its own .cu file and every header in
    csrc (a measurement stays valid while these are unchanged)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "jagged_sequence_attention_gb300", "csrc")
    names = [KERNEL_SOURCE[kernel]] + sorted(n for n in os.listdir(csrc) if n.endswith((".h", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/{workload}")
    if not e or kernel not in KERNEL_SOURCE or e.get("kernel_digest") != kernel_digest(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- reference (oracle)


def lengths_text(lens):
    """The sample's query lengths: listed when few, else their count, range and total."""
    lens = sorted(int(x) for x in lens)
    if len(lens) <= 8:
        return f"lengths {lens}"
    return f"lengths {lens[0]}..{lens[-1]}, {sum(lens)} tokens"


def oracle_sample(batch, target_seconds=15.0):
    """The shortest sequences of the batch (all heads), as a CPU batch: a bounded sample
    of the same workload for the oracle."""
    order = np.argsort(batch.q_lens * batch.kv_lens)
    # planning figure: the oracle's measured rate on the GPU machine's host cores, about 28 GFLOP/s
    # of fp64 work (a 4,269-token causal sequence, all 8 heads, forward and backward: 130 GFLOP
    # in 4.6 s)
    budget = 28e9 * target_seconds
    seqs, tot = [], 0.0
    for b in order:
        f = 3.5 * 4.0 * batch.D * batch.H * allowed_pairs([batch.q_lens[b]], [batch.kv_lens[b]], batch.causal,
                                                          batch.window)
        if seqs and tot + f > budget:
            break
        seqs.append(int(b))
        tot += f
    sub = wl.subset(batch, seqs)
    # the same problem (window and all) with its tensors on the host
    cpu = dataclasses.replace(sub, Q=sub.Q.cpu(), K=sub.K.cpu(), V=sub.V.cpu(), dO=sub.dO.cpu(),
                              bias=None if sub.bias is None else sub.bias.cpu(),
                              dense=None if sub.dense is None else sub.dense.cpu())
    return cpu, seqs


def run_oracle_once(cpu_batch, results=None):
    """Times one forward + backward of the oracle on a CPU batch; with a dict `results`, also
    leaves the outputs there (O, lse, dQ, dK, dV as fp64 arrays)."""
    import oracle
    f64 = lambda t: t.detach().to(torch.float32).numpy().astype(np.float64)  # noqa: E731
    b = None if cpu_batch.bias is None else f64(cpu_batch.bias)
    t0 = time.perf_counter()
    O, lse = oracle.fwd(cpu_batch.q_off, cpu_batch.kv_off, f64(cpu_batch.Q), f64(cpu_batch.K), f64(cpu_batch.V),
                        mode=cpu_batch.mode, causal=cpu_batch.causal, bias=b, scale=cpu_batch.scale,
                        window=cpu_batch.window)
    dQ, dK, dV = oracle.bwd(cpu_batch.q_off, cpu_batch.kv_off, f64(cpu_batch.Q), f64(cpu_batch.K), f64(cpu_batch.V),
                            f64(cpu_batch.dO), mode=cpu_batch.mode, causal=cpu_batch.causal, bias=b,
                            scale=cpu_batch.scale, window=cpu_batch.window)
    el = time.perf_counter() - t0
    if results is not None:
        results.update(O=O, lse=lse, dQ=dQ, dK=dK, dV=dV)
    return el


def sample_errors(got, ref, softmax):
    """Errors of the benchmarked launch's outputs on the oracle's sample (the tolerances of the
    parity tests: forward max-abs <= 1e-2 beyond a bf16 output's own rounding and relative
    Frobenius <= 5e-3; dQ, dK, dV relative Frobenius <= 1e-2)."""
    rel = lambda a, r: float(np.linalg.norm(a - r) / max(np.linalg.norm(r), 1e-30))  # noqa: E731
    e = {"O_max_abs": float(np.abs(got["O"] - ref["O"]).max()),
         "O_max_abs_beyond_rounding": float((np.abs(got["O"] - ref["O"]) - np.abs(ref["O"]) * 2.0 ** -8).max()),
         "O_rel_frob": rel(got["O"], ref["O"])}
    for k in ("dQ", "dK", "dV"):
        e[f"{k}_rel_frob"] = rel(got[k], ref[k])
    if softmax:
        fin = np.isfinite(ref["lse"])
        e["lse_max_abs"] = float(np.abs(got["lse"][fin] - ref["lse"][fin]).max()) if fin.any() else 0.0
    e["within_tolerance"] = bool(e["O_max_abs_beyond_rounding"] <= 1e-2 and e["O_rel_frob"] <= 5e-3 and
                                 max(e["dQ_rel_frob"], e["dK_rel_frob"], e["dV_rel_frob"]) <= 1e-2)
    return e


def oracle_cores(cpu_batch):
    import oracle
    return int(min(oracle.max_threads(), cpu_batch.B * cpu_batch.H))


# ----------------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_causal", choices=sorted(wl.WORKLOADS))
    # Pipelined end-to-end steps: the first step's input copy and the last step's result copy
    # have no neighbouring step to overlap, so they add (fill + drain) / steps to every step.
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--broadcast", action="store_true",
                    help="shared key/value workloads: run the plain path on an explicit broadcast copy of each "
                         "query set's user rows (the copies the in-kernel broadcast avoids; copy not timed)")
    ap.add_argument("--deterministic", action="store_true",
                    help="plans in deterministic mode (jfa_plan_set_deterministic): the two-pass bf16 backward, "
                         "the same bits on every run, whatever form the planner would choose")
    ap.add_argument("--partition", action="store_true",
                    help="strong scaling: one batch, its sequences split across the ranks by the LPT partition "
                         "(default: weak scaling, each rank its own batch of the workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    w = wl.WORKLOADS[args.workload]
    cfg = {"workload": args.workload, "description": w.description, "B": w.B, "H": w.H, "D": w.D,
           "mode": w.mode, "causal": w.causal, "bias": w.bias, "window": w.window, "seed": wl.seed_of(w),
           "users": w.users, "broadcast": bool(args.broadcast and w.users), "deterministic": bool(args.deterministic),
           "l2": "inputs larger than L2 (no flush needed)",
           "parallelism": f"dp{world} (" + ("LPT partition of one batch" if args.partition else "independent batches") + ")"}

    if args.impl == "reference":
        if rank != 0:
            if dist:
                dist.barrier()
            return
        batch = wl.broadcast(wl.make(args.workload, device="cpu"))
        # each timed step is one run of the sample: keep all K steps within about 2.5 minutes
        cpu, seqs = oracle_sample(batch, min(args.cpu_seconds, 150.0 / max(1, args.steps)))
        fl_f, fl_b = flops_of(cpu)
        # the oracle's one warm-up effect is loading its library: one tiny call does that
        run_oracle_once(wl.subset(cpu, [0], [0]))
        times = [run_oracle_once(cpu) for _ in range(args.steps)]
        t = sum(times) / len(times)
        v = (fl_f + fl_b) / t / 1e12
        sample = (f"{len(seqs)} shortest sequences of the workload ({lengths_text(batch.q_lens[seqs])}), "
                  f"all {cpu.H} heads, forward+backward in fp64")
        cfg.update({"tokens": int(batch.q_off[-1]), "sample_tokens": int(cpu.q_off[-1])})
        line = {"metric": METRIC, "value": v, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle_cores(cpu), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        if dist:
            dist.barrier()
        return

    from jagged_sequence_attention_gb300 import _build
    from jagged_sequence_attention_gb300 import jfa
    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.partition:
        # every rank draws the same batch and keeps its LPT share of the sequences
        batch = jfa.shard(wl.make(args.workload, device=dev), rank, world)
    else:
        batch = wl.make(args.workload, device=dev, seed=wl.seed_of(w) + 7919 * rank)
    if args.broadcast:
        batch = wl.broadcast(batch)
    fl_f, fl_b = flops_of(batch)
    job_flop = fl_f + fl_b  # summed over ranks below: the work all ranks processed
    cfg.update({"tokens": int(batch.q_off[-1]), "kv_tokens": int(batch.kv_off[-1]),
                "unpadded_fwd_flop": fl_f, "unpadded_bwd_flop": fl_b})

    stream = torch.cuda.current_stream()
    plan = jfa.plan_for(batch, deterministic=args.deterministic)
    # The backward form jfa_bwd runs on bf16 inputs: short-query (no bias, every query set
    # in one tile), else fused (no dense bias, no bias gradient), else two-pass.
    info = jfa.jfa_plan_info(plan)
    bf16 = batch.Q.dtype == torch.bfloat16
    short_q = bf16 and info["bwd_short"] > 0 and batch.bias is None
    fused = bf16 and not short_q and info["bwd_fused"] == 1
    # one backward kernel forms dQ, dK and dV: short-query, fused, and the fp32 path
    one_kernel_bwd = fused or short_q or not bf16
    kbytes = algorithmic_bytes(batch, elem=2 if bf16 else 4, fused=one_kernel_bwd)
    cfg["backward"] = ("fp32 CUDA-core kernel (dQ by atomics) + dQ conversion" if not bf16 else
                       "short-query dQ/dK/dV kernel" if short_q else
                       "fused dK/dV/dQ kernel" if fused else "dK/dV kernel + dQ kernel")
    cfg["forward"] = {"jfa_fwd_kernel": "query-tile kernel", "jfa_fwd_short_kernel": "short-query GDPA kernel",
                      "jfa_fwd_pack_kernel": "short-query softmax kernel (two key tiles per score tile)",
                      "jfa_fwd_f32_kernel": "fp32 CUDA-core kernel"}[
        "jfa_fwd_f32_kernel" if not bf16 else
        ("jfa_fwd_pack_kernel" if batch.mode == "softmax" else "jfa_fwd_short_kernel")
        if (info["fwd_short"] > 0 and batch.bias is None) else "jfa_fwd_kernel"]
    O = torch.empty_like(batch.Q)
    lse = torch.empty((batch.Q.shape[0], batch.H), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(batch.Q), torch.empty_like(batch.K), torch.empty_like(batch.V)
    ws = torch.empty(jfa.jfa_bwd_workspace_size(plan, batch.Q.dtype), dtype=torch.uint8, device=dev)

    def step():
        jfa.jfa_fwd(plan, batch.Q, batch.K, batch.V, batch.bias, batch.scale, O=O, lse=lse)
        jfa.jfa_bwd(plan, batch.Q, batch.K, batch.V, O, batch.dO, lse, batch.bias, batch.scale, dQ=dQ, dK=dK,
                    dV=dV, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = jfa.jfa_plan_device_status(plan)
    if status != 0:
        raise RuntimeError(f"device status after warm-up: {jfa.jfa_status_string(status)}")

    jfa.jfa_plan_set_timing(plan, True)
    jfa.jfa_plan_kernel_times(plan)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else torch.cuda.current_device())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    kt = jfa.jfa_plan_kernel_times(plan)
    jfa.jfa_plan_set_timing(plan, False)
    status = jfa.jfa_plan_device_status(plan)
    if status != 0:
        raise RuntimeError(f"device status after timing: {jfa.jfa_status_string(status)}")
    # The timed launch's outputs for the oracle's sample (the shortest sequences, all heads),
    # kept for the error report beside the CPU baseline (plain batches).
    sampled_rows = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and batch.kv_map is None:
        _, sample_seqs = oracle_sample(batch, args.cpu_seconds)
        qi = np.concatenate([np.arange(batch.q_off[b], batch.q_off[b + 1]) for b in sample_seqs])
        ki = np.concatenate([np.arange(batch.kv_off[b], batch.kv_off[b + 1]) for b in sample_seqs])
        sel = lambda t, idx: t[torch.as_tensor(idx, device=t.device)].float().cpu().numpy().astype(np.float64)  # noqa: E731
        sampled_rows = {"O": sel(O, qi), "lse": sel(lse, qi), "dQ": sel(dQ, qi), "dK": sel(dK, ki), "dV": sel(dV, ki)}
    if dist:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        jf = torch.tensor([job_flop], dtype=torch.float64, device=dev)
        dist.all_reduce(jf, op=dist.ReduceOp.SUM)
        job_flop = float(jf.item())
    ms_step = ms / args.steps
    value = job_flop / (ms_step / 1e3) / 1e12
    peaks = load_peaks()

    # dominant kernel: the largest share of device time among the tensor-core kernels
    per = {k: (v[0] / v[1] if v[1] else 0.0, v[1], v[0]) for k, v in kt.items()}
    kflop = kernel_flops(fl_f, one_kernel_bwd)
    fwd_short = bf16 and info["fwd_short"] > 0 and batch.bias is None
    fwd_kernel = ("jfa_fwd_f32_kernel" if not bf16 else
                  ("jfa_fwd_pack_kernel" if batch.mode == "softmax" else "jfa_fwd_short_kernel") if fwd_short else
                  "jfa_fwd_kernel")
    kname_of = {"fwd": fwd_kernel, "bwd_main": "jfa_bwd_f32_kernel" if not bf16 else ("jfa_bwd_short_kernel" if short_q else
                                                      "jfa_bwd_fused_kernel" if fused else "jfa_bwd_dkdv_kernel")}
    if bf16 and not (fused or short_q):
        kname_of["bwd_dq"] = "jfa_bwd_dq_kernel"
    dom = max(kname_of, key=lambda k: per[k][2])
    dom_ms = per[dom][0]
    achieved = kflop[dom] / (dom_ms / 1e3) / 1e12 if dom_ms > 0 else 0.0
    kname = kname_of[dom]
    # The roof that binds the dominant kernel: the one its algorithmic rate comes closer to
    # (tensor FLOP/s on the long sequences, HBM bytes/s on the short-query shapes).
    gbs = kbytes[dom] / (dom_ms / 1e3) / 1e9 if dom_ms > 0 else 0.0
    frac_t = achieved / peaks["bf16_tflops_sustained"]
    frac_b = gbs / peaks["hbm_gbs"]
    if frac_b > frac_t:
        roofline = {"bound": "hbm", "kernel": kname, "achieved": gbs, "peak": peaks["hbm_gbs"],
                    "peak_kind": f"HBM copy, {peaks['source']}", "unit": "GB/s", "frac": frac_b,
                    "tensor_frac": frac_t}
    else:
        roofline = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peaks["bf16_tflops_sustained"],
                    "peak_kind": f"bf16 dense, sustained, {peaks['source']}", "unit": "TFLOP/s", "frac": frac_t,
                    "hbm_frac": frac_b}
    roofline.update({"traffic": measured_traffic(kname, args.workload),
                     "algorithmic_bytes_per_launch": kbytes[dom], "flop_per_launch": kflop[dom]})
    kernels = {k: {"ms_per_launch": v[0], "launches": v[1], "share": v[2] / max(1e-9, sum(x[2] for x in per.values())),
                   **({"tflops": kflop[k] / (v[0] / 1e3) / 1e12,
                       "gbs": kbytes[k] / (v[0] / 1e3) / 1e9} if k in kflop and v[0] > 0 else {})}
               for k, v in per.items()}
    launches = int(sum(v[1] for v in per.values()))

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "strong" if args.partition else "weak",
            "vs_baseline": None, "dtype": "f32" if batch.Q.dtype == torch.float32 else "bf16", "data": "synthetic",
            "config": cfg,
            "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "pct_of_bf16_peak_sustained": 100.0 * value / world / peaks["bf16_tflops_sustained"],
            "fwd_tflops": fl_f / (kt["fwd"][0] / max(1, kt["fwd"][1]) / 1e3) / 1e12 if kt["fwd"][1] else None,
            # backward alone: every backward launch of a step (row terms, dK/dV, dQ, fp32 convert)
            "bwd_tflops": (fl_b / (sum(per[k][0] for k in ("bwd_pre", "bwd_main", "bwd_dq", "bwd_post")) / 1e3) / 1e12
                           if per["bwd_main"][1] else None),
            "roofline": roofline, "kernels": kernels, "gpu_launches": launches, "clocks": clocks}

    # ---------------------------------------------------------------- end to end through the API
    if not args.no_e2e:
        # Every step: pinned host -> device copies of its inputs (Q, K, V, dO, bias), a new plan
        # from the host offsets, jfa_fwd, jfa_bwd, and device -> host copies of all its results
        # (O, lse, dQ, dK, dV).  Steps are pipelined as a training loop prefetches its next
        # batch: two device buffer sets, inputs copied in on one stream and results copied out
        # on another while the kernels of the neighbouring step run.  All copies are inside the
        # timed region.  The same loop run serially (one step at a time) is reported beside it.
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        hQ, hK, hV, hdO = pin(batch.Q), pin(batch.K), pin(batch.V), pin(batch.dO)
        hbias = None if batch.bias is None else pin(batch.bias)
        hO, hdQ = torch.empty_like(hQ).pin_memory(), torch.empty_like(hQ).pin_memory()
        hdK, hdV = torch.empty_like(hK).pin_memory(), torch.empty_like(hV).pin_memory()
        hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        q_off, kv_off = batch.q_off.copy(), batch.kv_off.copy()
        sets = []
        for k in range(2):
            sets.append({
                "Q": batch.Q if k == 0 else torch.empty_like(batch.Q),
                "K": batch.K if k == 0 else torch.empty_like(batch.K),
                "V": batch.V if k == 0 else torch.empty_like(batch.V),
                "dO": batch.dO if k == 0 else torch.empty_like(batch.dO),
                "bias": None if batch.bias is None else (batch.bias if k == 0 else torch.empty_like(batch.bias)),
                "O": O if k == 0 else torch.empty_like(O), "lse": lse if k == 0 else torch.empty_like(lse),
                "dQ": dQ if k == 0 else torch.empty_like(dQ), "dK": dK if k == 0 else torch.empty_like(dK),
                "dV": dV if k == 0 else torch.empty_like(dV), "ws": ws if k == 0 else torch.empty_like(ws),
                "freed": torch.cuda.Event()})
            sets[k]["freed"].record(stream)
        # plan creation synchronises the stream it is given (the work-list upload): its own
        s_in, s_out, s_plan = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV, hdO)) + (
            0 if hbias is None else hbias.numel() * 4) + q_off.nbytes + kv_off.nbytes
        d2h = sum(t.numel() * t.element_size() for t in (hO, hdQ, hdK, hdV, hlse))

        def e2e_step(i, plans):
            b = sets[i % 2]
            with torch.cuda.stream(s_in):
                s_in.wait_event(b["freed"])  # the set's previous step has copied its results out
                for name, h in (("Q", hQ), ("K", hK), ("V", hV), ("bias", hbias)):
                    if h is not None:
                        b[name].copy_(h, non_blocking=True)
                ev_qkv = torch.cuda.Event()
                ev_qkv.record(s_in)
                b["dO"].copy_(hdO, non_blocking=True)
                ev_do = torch.cuda.Event()
                ev_do.record(s_in)
            p2 = jfa.plan_for(wl.Batch(batch.name, q_off, kv_off, b["Q"], b["K"], b["V"], b["dO"], b["bias"],
                                       batch.scale, batch.mode, batch.causal, batch.H, batch.D,
                                       window=batch.window, kv_map=batch.kv_map), stream=s_plan,
                              deterministic=args.deterministic)
            plans.append(p2)
            stream.wait_event(ev_qkv)
            jfa.jfa_fwd(p2, b["Q"], b["K"], b["V"], b["bias"], batch.scale, O=b["O"], lse=b["lse"], stream=stream)
            ev_fwd = torch.cuda.Event()
            ev_fwd.record(stream)
            stream.wait_event(ev_do)
            jfa.jfa_bwd(p2, b["Q"], b["K"], b["V"], b["O"], b["dO"], b["lse"], b["bias"], batch.scale, dQ=b["dQ"],
                        dK=b["dK"], dV=b["dV"], workspace=b["ws"], stream=stream)
            ev_bwd = torch.cuda.Event()
            ev_bwd.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fwd)
                hO.copy_(b["O"], non_blocking=True)
                hlse.copy_(b["lse"], non_blocking=True)
                s_out.wait_event(ev_bwd)
                hdQ.copy_(b["dQ"], non_blocking=True)
                hdK.copy_(b["dK"], non_blocking=True)
                hdV.copy_(b["dV"], non_blocking=True)
                b["freed"].record(s_out)

        def timed(n_steps, serial):
            plans = []
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            for i in range(n_steps):
                e2e_step(i, plans)
                if serial:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()
            el = (time.perf_counter() - t0) / n_steps
            for p2 in plans:  # freeing device memory synchronises the device: after the timed loop
                jfa.jfa_plan_destroy(p2)
            if dist:
                t = torch.tensor([el], dtype=torch.float64, device=dev)
                dist.all_reduce(t, op=dist.ReduceOp.MAX)
                el = float(t.item())
            return el

        timed(2, False)  # warm-up of both buffer sets and streams
        el = timed(args.e2e_steps, False)
        el_serial = timed(max(1, args.e2e_steps // 2), True)
        line["e2e"] = {"value": job_flop / el / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                       "d2h_bytes_per_step": int(d2h), "ms_per_step": el * 1e3, "steps": args.e2e_steps,
                       "serial_value": job_flop / el_serial / 1e12, "serial_ms_per_step": el_serial * 1e3,
                       "includes": "every step: pinned H2D of Q,K,V,dO,bias; jfa_plan_create from host offsets; "
                                   "jfa_fwd; jfa_bwd; D2H of O,lse,dQ,dK,dV. Steps pipelined on two device buffer "
                                   "sets (copies of one step overlap the kernels of its neighbours; the "
                                   "first step's copy-in and the last step's copy-out, which nothing "
                                   "overlaps, are inside the timed region); serial_*: the same steps one "
                                   "at a time"}

    # ---------------------------------------------------------------- CPU baseline (oracle)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, seqs = oracle_sample(wl.broadcast(batch), args.cpu_seconds)
        cf, cb = flops_of(cpu)
        run_oracle_once(wl.subset(cpu, [0], [0]))
        ref = {}
        t = run_oracle_once(cpu, ref)
        line["cpu_baseline"] = {"value": (cf + cb) / t / 1e12, "unit": UNIT, "cores": oracle_cores(cpu),
                                "kind": "oracle", "seconds": t,
                                "sample": f"{len(seqs)} shortest sequences ({lengths_text(batch.q_lens[seqs])}), "
                                          f"all {cpu.H} heads, fwd+bwd fp64"}
        if sampled_rows is not None:
            # the benchmarked launch's own outputs for the same sequences, against the oracle
            line["parity_sample"] = {"sample": line["cpu_baseline"]["sample"],
                                     **sample_errors(sampled_rows, ref, batch.mode == "softmax")}

    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
