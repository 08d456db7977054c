#!/usr/bin/env python3
"""Benchmark of the Muon optimizer step on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5]
    python bench.py --impl reference ...      (the CPU oracle as the reference arm)

A step is one pass of the whole optimizer over the workload.  The default
(headline) workload is c5, the full mixed step: one muon_step_batched call
over 6144 fine-grained-MoE expert matrices (16 layers x 128 experts x gate,
up 1408x2048 and down 2048x1408, fp32 gradients) -- momentum, normalisation,
five Newton-Schulz iterations on the tensor cores and the final update --
followed by one adamw_step_batched call over the embedding and the LM head
(2 x 163840 x 7168 fp32).  Both calls are inside the timed region.

value: Newton-Schulz TFLOP/s over the whole step time (Muon + AdamW),
counting the algorithmic flops (symmetry exploited) 3 m'^2 n' + m'^3 per
matrix per iteration, summed over all ranks; ms_per_step is that whole
step.  The line also carries the Muon and AdamW parts on their own
("muon_ms_per_step", "adamw"), the per-kernel breakdown ("stages"), the
roofline of the dominant kernel, and one sub-record per other workload
("per_workload": c1 one 256x512 matrix, c2 a dense 24-layer decoder, c3 a
fine-grained MoE with 1568 matrices, c4 a 7168 / 18432 layer).
Under torchrun every rank runs its own replica of the workload (weak
scaling, no collective on the data path).  The headline workload's inputs
(about 250 GB) are far larger than L2 (129 MB); a workload whose W, G and M
fit in 4 x L2 (c1) has L2 flushed between timed steps instead (a 512 MB
write outside the per-step events).

e2e: the same step through the public API with the data in host memory:
every step copies every input of the step (W, G, M; p, g, m, v) from pinned
host buffers to the device and every result (W, M; p, m, v) back, in
pieces pipelined over three streams (copy in / step / copy out).  The GPU
box's host memory (about 200 GB) cannot hold the headline workload's 250 GB
of state, so the pinned host buffers are a ring of two slots per kind of
piece, filled once with the first piece's synthetic data and re-sent for
every piece: the bytes moved are the real ones, the host-side values are
shared between pieces.

graph_replay: the Muon step captured once as a CUDA graph
(muon_step_graph_create) and replayed, each replay timed on its own and
alternating with eager steps (no per-launch timing events), whose median is
reported beside it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "Muon optimizer-step ms & NS TFLOP/s (frac of BF16 peak); AdamW HBM GB/s"
UNIT = "TFLOP/s"
L2_BYTES = 129 << 20  # GB300 L2
ADAMW_BYTES_PER_PARAM = 28  # read p, g, m, v (16 B), write p, m, v (12 B)
HEADLINE = "c5"
SUB_WORKLOADS = ("c1", "c2", "c3", "c4")
KINDS = ("momentum_norm", "norm_finalize", "x0_rescale", "ns_syrk", "ns_poly", "ns_update",
         "final_update", "adamw", "grad_guard", "desc_upload", "stats")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--budget-gb", type=float, default=16.0, help="NS workspace budget")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-adamw", action="store_true",
                    help="leave the workload's AdamW buffers out of the step (profiling only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-guard", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-per-workload", action="store_true", help="skip the c1-c4 sub-records")
    ap.add_argument("--subset", type=int, default=0,
                    help="profiling only: keep the first N matrices of the workload")
    ap.add_argument("--adamw-params", type=int, default=0,
                    help="profiling only: N parameters per AdamW buffer instead of the full embedding size")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# flop and byte accounting
# --------------------------------------------------------------------------

def ns_stage_flops(mp: int, np_: int):
    """Algorithmic flops of one NS iteration on one matrix, per stage."""
    return {"ns_syrk": mp * (mp + 1) * np_,      # upper triangle of X X^T
            "ns_poly": mp * mp * (mp + 1),       # upper triangle of A A
            "ns_update": 2 * mp * mp * np_}      # B X


def _ceil(a: int, b: int) -> int:
    return (a + b - 1) // b


def ns_stage_issued_flops(mp: int, np_: int):
    """Flops the tensor cores are issued for one NS iteration on one matrix,
    per stage: the kernels' tile enumeration, counting computed halves of
    diagonal tiles, rows and columns padded past the matrix and K rounded
    up to 64.  Mirrors the tile choices of the library's NS launch code:
    128x256 single-CTA tiles or 256x256 CTA-pair tiles (every stage on pairs
    when m' > 512 and 256-row pair tiles waste at most 1/8 of the rows),
    the last column tile rounded to 16 (single), 32 (pairs) or 128 (pairs on
    64-aligned shapes)."""
    pad = _ceil(mp, 256) * 256 - mp
    pairs = mp > 512 and pad * 8 <= mp
    chunked = mp % 64 == 0 and np_ % 64 == 0

    def col_widths(n, pair):
        q = (128 if chunked else 32) if pair else 16
        out = []
        for j in range(_ceil(n, 256)):
            rem = n - 256 * j
            out.append(256 if rem >= 256 else _ceil(rem, q) * q)
        return out

    def triangle(k):
        if pairs:  # pairs: tiles (I, J >= I) of 256 x n_J
            w = col_widths(mp, True)
            return sum(256 * w[j] * k for i in range(len(w)) for j in range(i, len(w)))
        w = col_widths(mp, False)
        total = 0
        for ti in range(_ceil(mp, 128)):
            for tj in range(ti // 2, len(w)):
                lo = 128 if (ti % 2 == 1 and tj == ti // 2) else 0
                total += 128 * (w[tj] - lo) * k
        return total

    k_x, k_g = _ceil(np_, 64) * 64, _ceil(mp, 64) * 64
    if pairs:
        upd = _ceil(mp, 256) * 256 * sum(col_widths(np_, True)) * k_g
    else:
        upd = _ceil(mp, 128) * 128 * sum(col_widths(np_, False)) * k_g
    return {"ns_syrk": 2 * triangle(k_x), "ns_poly": 2 * triangle(k_g), "ns_update": 2 * upd}


def workload_flops(w: workloads.Workload, steps: int):
    """(algorithmic flops per stage, dense-equivalent flops, issued flops per
    stage) of `steps` NS iterations on every matrix of the workload."""
    per = {"ns_syrk": 0, "ns_poly": 0, "ns_update": 0}
    issued = dict(per)
    dense = 0
    for s in w.matrices:
        mp, np_ = min(s.rows, s.cols), max(s.rows, s.cols)
        for k, v in ns_stage_flops(mp, np_).items():
            per[k] += steps * v
        for k, v in ns_stage_issued_flops(mp, np_).items():
            issued[k] += steps * v
        dense += steps * (4 * mp * mp * np_ + 2 * mp ** 3)
    return per, dense, issued


def elementwise_bytes(w: workloads.Workload):
    """Algorithmic HBM bytes per step of the element-wise Muon stages."""
    out = {"momentum_norm": 0, "final_update": 0}
    for s in w.matrices:
        n = s.rows * s.cols
        g = 2 if s.g_dtype.itemsize == 2 else 4
        out["momentum_norm"] += n * (g + 4 + 4 + 2)    # read G, M; write M, X0 = bf16(u)
        out["final_update"] += n * (4 + 2 + 4)         # read W, O; write W
    return out


def input_bytes(w: workloads.Workload) -> int:
    """Bytes of W, G and M over every matrix of the workload."""
    return sum(s.rows * s.cols * (4 + s.g_dtype.itemsize + 4) for s in w.matrices)


def l2_note(w: workloads.Workload) -> str:
    b = input_bytes(w)
    if b < 4 * L2_BYTES:
        return f"inputs {b / 2**20:.1f} MB fit in L2: L2 flushed by a 512 MB write before each timed step"
    return f"inputs {b / 2**30:.1f} GB exceed the 129 MB L2; no flush needed"


def workload_config(w: workloads.Workload, steps_ns: int, world: int) -> dict:
    """The config object of the JSON line (the same for both arms)."""
    stage_flops, dense_flops, _ = workload_flops(w, steps_ns)
    step = "muon_step_batched" + (" + adamw_step_batched" if w.adamw_shapes else "")
    return {"workload": f"{w.name}: {w.description}", "step": step, "matrices": len(w.matrices),
            "muon_params": w.muon_params, "adamw_params": w.adamw_params, "ns_steps": steps_ns,
            "ns_flops_per_step_algorithmic": sum(stage_flops.values()),
            "ns_flops_per_step_dense_equivalent": dense_flops,
            "l2": l2_note(w),
            "parallelism": "replicas" if world > 1 else "single"}


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step: int, steps: int, world: int, ms_total_max: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of the workload
    (weak scaling), timed by the slowest rank."""
    return flops_per_step * steps * world / (ms_total_max / 1e3) / 1e12


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu captures
    (profiles/ncu_traffic.json, one record per workload), scaled to the full
    workload's launch; None when no record covers the workload or the
    kernel source changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            doc = json.load(f)
        for rec in doc.get("records", [doc]):
            if rec.get("workload") != workload or kernel not in rec.get("captured_bytes", {}):
                continue
            with open(os.path.join(ROOT, rec["source_file"]), "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()
            if sha != rec["source_sha256"]:
                return None
            b = rec["captured_bytes"][kernel]
            return (b["read"] + b["write"]) * rec["scale_to_full_launch"]
    except Exception:
        return None
    return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sms, maxes, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.NAMES, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "samples": len(sms),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# the CPU oracle (baseline and reference arm)
# --------------------------------------------------------------------------

# Dense fp64 flops of oracle work per sample.  The oracle runs at about 0.11
# TFLOP/s (dense) on 16 host cores: the reference arm's per-step sample is
# about 2 s, the cpu_baseline sample about 13 s.
REFERENCE_STEP_FLOPS = 2.6e11
CPU_BASELINE_FLOPS = 1.5e12
ADAMW_SAMPLE = 1 << 26  # AdamW elements the CPU baseline times (64 M)


def oracle_sample(w: workloads.Workload, budget_flops: float):
    """A bounded sample of the workload for the CPU oracle: matrices of its
    most common shape, drawn from the workload's distributions, as many as
    fit `budget_flops` (at least one), with as many of the 5 NS iterations
    as fit when one matrix alone exceeds it (the oracle multiplies full, not
    triangular, matrices)."""
    import collections
    shapes = collections.Counter((s.rows, s.cols) for s in w.matrices)
    (rows, cols), count = shapes.most_common(1)[0]
    mp, np_ = min(rows, cols), max(rows, cols)
    dense_per_iter = 4 * mp * mp * np_ + 2 * mp ** 3
    full = workloads.MUON_HPARAMS["ns_steps"]
    steps = max(1, min(full, int(budget_flops // dense_per_iter)))
    n_mats = max(1, min(count, int(budget_flops // (dense_per_iter * full)))) if steps == full else 1
    idx = [i for i, s in enumerate(w.matrices) if (s.rows, s.cols) == (rows, cols)][:n_mats]
    t = workloads.make_muon(w, device="cpu", indices=idx)
    mats = [(t.W[k].numpy(), t.G[k].float().numpy(), t.M[k].numpy()) for k in range(len(idx))]
    flops = sum(ns_stage_flops(mp, np_).values()) * steps * len(idx)
    desc = f"{len(idx)} matri{'x' if len(idx) == 1 else 'ces'} {rows}x{cols}, {steps} of {full} NS iterations"
    return mats, flops, desc, steps


def time_oracle(w: workloads.Workload, budget_flops: float, repeats: int = 1):
    """Wall times of `repeats` oracle steps over one bounded sample."""
    import oracle
    mats, flops, desc, steps = oracle_sample(w, budget_flops)
    cfg = oracle.MuonConfig(**dict(workloads.MUON_HPARAMS, ns_steps=steps))
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        for W, G, M in mats:
            oracle.muon_step_matrix(W, G, M, cfg)
        times.append(time.perf_counter() - t0)
    return times, flops, desc, oracle.num_threads(), steps, len(mats)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


_C1_ONE_THREAD = """
import sys, time
sys.path.insert(0, {root!r})
import oracle, workloads
w = workloads.get("c1")
t = workloads.make_muon(w)
cfg = oracle.MuonConfig(**workloads.MUON_HPARAMS)
args = (t.W[0].numpy(), t.G[0].float().numpy(), t.M[0].numpy())
oracle.muon_step_matrix(*args, cfg)
t0 = time.perf_counter()
oracle.muon_step_matrix(*args, cfg)
print(1e3 * (time.perf_counter() - t0), oracle.num_threads())
"""


def single_thread_c1_ms():
    """One whole oracle step on the 256x512 matrix with one OpenMP thread,
    in a child process (fork + exec; nothing of this process's CUDA state
    is inherited).  Returns (ms, threads) or (None, None)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", _C1_ONE_THREAD.format(root=ROOT)], env=env,
                           capture_output=True, text=True, timeout=300)
        ms, threads = r.stdout.split()[-2:]
        return float(ms), int(threads)
    except Exception:
        return None, None


def time_oracle_adamw(n: int):
    """Seconds per element of the oracle's AdamW on an n-element sample."""
    import oracle
    a = workloads.make_adamw(n, seed=0)
    cfg = oracle.AdamwConfig(**workloads.ADAMW_HPARAMS)
    args = [x.numpy() for x in (a.p, a.g, a.m, a.v)]
    t0 = time.perf_counter()
    oracle.adamw_step(*args, cfg, t=workloads.ADAMW_STEP)
    return (time.perf_counter() - t0) / n


def cpu_baseline(w: workloads.Workload) -> dict:
    """The oracle as it stands, timed on this host on a bounded sample of
    the workload, with the whole step extrapolated from it: each distinct
    (m', n') costs the sampled matrix's time scaled by its dense flops,
    AdamW its sampled per-element time times the buffers' elements."""
    import collections
    times, flops, desc, cores, steps, n_mats = time_oracle(w, CPU_BASELINE_FLOPS)
    shapes = collections.Counter((min(m.rows, m.cols), max(m.rows, m.cols)) for m in w.matrices)
    rows, cols = collections.Counter((m.rows, m.cols) for m in w.matrices).most_common(1)[0][0]
    mp0, np0 = min(rows, cols), max(rows, cols)
    full = workloads.MUON_HPARAMS["ns_steps"]
    per_matrix_s = times[0] / n_mats * full / steps
    dense = lambda mp, np_: 4 * mp * mp * np_ + 2 * mp ** 3  # noqa: E731
    muon_s = sum(c * per_matrix_s * dense(mp, np_) / dense(mp0, np0) for (mp, np_), c in shapes.items())
    adamw_s = 0.0
    adamw_desc = None
    if w.adamw_params:
        per_el = time_oracle_adamw(ADAMW_SAMPLE)
        adamw_s = per_el * w.adamw_params
        adamw_desc = f"AdamW on {ADAMW_SAMPLE} elements, {per_el * 1e9:.2f} ns per element"
    c1_ms, c1_threads = single_thread_c1_ms()
    return {"value": flops / times[0] / 1e12, "unit": UNIT, "cores": cores, "threads": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{desc}, of {len(w.matrices)} matrices (full Muon step otherwise), {times[0]:.1f} s"
                      + (f"; {adamw_desc}" if adamw_desc else ""),
            "extrapolated_step_ms": {"muon": 1e3 * muon_s, "adamw": 1e3 * adamw_s,
                                     "total": 1e3 * (muon_s + adamw_s),
                                     "label": "extrapolated from the sample by dense flops per (m', n') "
                                              "and by AdamW elements; not a measured full step"},
            "single_thread_c1_ms": c1_ms, "single_thread_c1_threads": c1_threads}


def run_reference(args, rank):
    if rank != 0:
        return
    w = workloads.get(args.workload)
    time_oracle(workloads.get("c1"), REFERENCE_STEP_FLOPS)  # build + warm the library
    for _ in range(args.warmup):
        time_oracle(w, REFERENCE_STEP_FLOPS)
    times, flops, desc, cores, _, _ = time_oracle(w, REFERENCE_STEP_FLOPS, repeats=args.steps)
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = f"{desc}, of {len(w.matrices)} matrices, per step (full Muon step otherwise)"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, workloads.MUON_HPARAMS["ns_steps"], args.gpus),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

class WorkloadStep:
    """A workload's tensors on the device and one step over them: one
    muon_step_batched call over every matrix, then (when the workload has
    AdamW buffers) one adamw_step_batched call over all of them."""

    def __init__(self, m, w: workloads.Workload, dev, budget: int, with_adamw: bool = True,
                 adamw_params: int = 0):
        self.m, self.w, self.budget = m, w, budget
        self.hp = m.MuonHparams(**workloads.MUON_HPARAMS)
        self.ahp = m.AdamwHparams(**workloads.ADAMW_HPARAMS)
        self.tens = workloads.make_muon(w, device=dev)
        self.batch = m.MuonBatch(self.tens.W, self.tens.G, self.tens.M, budget_bytes=budget)
        self.adamw = []
        if with_adamw and w.adamw_shapes:
            sizes = [adamw_params or r * c for r, c in w.adamw_shapes]
            self.adamw = [workloads.make_adamw(n, seed=w.seed + i, device=dev) for i, n in enumerate(sizes)]
        self.quads = [(b.p, b.g, b.m, b.v) for b in self.adamw]
        self.adamw_params = sum(b.p.numel() for b in self.adamw)

    def muon(self, stream, hp=None):
        self.batch.step(hp or self.hp, stream)

    def adamw_step(self, stream):
        if self.quads:
            self.m.adamw_step_batched(self.quads, self.ahp, workloads.ADAMW_STEP, stream)


def measure(m, ws: WorkloadStep, steps: int, warmup: int, peaks: dict, dev, local_rank: int,
            barrier, max_over_ranks, world: int, subset: bool = False) -> dict:
    """Times `steps` steps (after `warmup` untimed ones) with CUDA events on
    the launching stream around the Muon and the AdamW call of every step,
    per-launch kernel timing on, clocks sampled; returns the step time, the
    per-kernel breakdown and the dominant kernel's roofline."""
    import torch
    w = ws.w
    stream = torch.cuda.current_stream()
    steps_ns = ws.hp.ns_steps
    stage_flops, dense_flops, issued_flops = workload_flops(w, steps_ns)
    step_flops = sum(stage_flops.values())
    ew_bytes = elementwise_bytes(w)
    for _ in range(warmup):
        ws.muon(stream)
        ws.adamw_step(stream)
    torch.cuda.synchronize()
    if m.muon_query_status(ws.batch.workspace) != 0:
        raise RuntimeError("device status set during warm-up")
    flush = None
    if input_bytes(w) < 4 * L2_BYTES:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    clocks = ClockSampler(local_rank)
    m.muon_set_timing(True)
    launches0 = m.muon_launch_count()
    marks = []
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(steps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        ws.muon(stream)
        ev[1].record(stream)
        ws.adamw_step(stream)
        ev[2].record(stream)
        marks.append(ev)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    launches = m.muon_launch_count() - launches0
    kernel_times = m.muon_timing_read()
    m.muon_set_timing(False)
    status = m.muon_query_status(ws.batch.workspace)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    muon_ms = sum(a.elapsed_time(b) for a, b, _ in marks)
    adamw_ms = sum(b.elapsed_time(c) for _, b, c in marks)
    timed_without_launch_events = False
    if (muon_ms + adamw_ms) / steps < 5.0:
        # a launch-bound step: the two timing events around each of its
        # launches lengthen it, so its time comes from a second pass of the
        # same steps without them (the breakdown above keeps them)
        marks = []
        barrier()
        torch.cuda.synchronize()
        for _ in range(steps):
            if flush is not None:
                with torch.cuda.stream(stream):
                    flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            ws.muon(stream)
            ev[1].record(stream)
            ws.adamw_step(stream)
            ev[2].record(stream)
            marks.append(ev)
        torch.cuda.synchronize()
        barrier()
        muon_ms = sum(a.elapsed_time(b) for a, b, _ in marks)
        adamw_ms = sum(b.elapsed_time(c) for _, b, c in marks)
        timed_without_launch_events = True
    ms_total = max_over_ranks(muon_ms + adamw_ms)
    ms_step = ms_total / steps

    stages = {}
    for k in KINDS:
        ms_k, n_k = kernel_times.get(k, (0.0, 0))
        if n_k:
            stages[k] = {"ms_per_step": ms_k / steps, "launches_per_step": n_k / steps}
    ns_kinds = [k for k in ("ns_syrk", "ns_poly", "ns_update") if k in stages]
    for k in ns_kinds:
        s = stages[k]
        s["tflops"] = stage_flops[k] / (s["ms_per_step"] / 1e3) / 1e12
        s["tflops_issued"] = issued_flops[k] / (s["ms_per_step"] / 1e3) / 1e12
    for k in ("momentum_norm", "final_update"):
        if k in stages:
            stages[k]["gbs"] = ew_bytes[k] / (stages[k]["ms_per_step"] / 1e3) / 1e9
    if "adamw" in stages:
        stages["adamw"]["gbs"] = ADAMW_BYTES_PER_PARAM * ws.adamw_params / (stages["adamw"]["ms_per_step"] / 1e3) / 1e9
    dominant = max(stages, key=lambda k: stages[k]["ms_per_step"])
    d = stages[dominant]
    ms_launch = d["ms_per_step"] / d["launches_per_step"]
    if dominant in ns_kinds:
        per_launch = stage_flops[dominant] / d["launches_per_step"]
        achieved = per_launch / (ms_launch / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        roofline = {"bound": "tensor", "kernel": dominant, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_kind": f"bf16 sustained, {peaks['source']}",
                    "algorithmic_per_launch": per_launch, "ms_per_launch": ms_launch,
                    "traffic": None if subset else ncu_traffic(dominant, w.name),
                    "traffic_unit": "bytes per launch (DRAM read + write, ncu)"}
    else:
        per_launch = (ADAMW_BYTES_PER_PARAM * ws.adamw_params if dominant == "adamw"
                      else ew_bytes.get(dominant, 0)) / d["launches_per_step"]
        achieved = per_launch / (ms_launch / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_kind": f"HBM copy, {peaks['source']}",
                    "algorithmic_per_launch": per_launch, "ms_per_launch": ms_launch, "traffic": None}
    ns_ms = sum(stages[k]["ms_per_step"] for k in ns_kinds)
    out = {"ms_total": ms_total, "ms_per_step": ms_step, "muon_ms_per_step": max_over_ranks(muon_ms) / steps,
           "adamw_ms_per_step": max_over_ranks(adamw_ms) / steps if ws.quads else None,
           "value": aggregate_tflops(step_flops, steps, world, ms_total), "step_flops": step_flops,
           "stages": stages, "roofline": roofline, "launches": launches, "clocks": clk,
           "l2_flushed": flush is not None,
           "step_time": ("second pass without per-launch timing events (launch-bound step)"
                         if timed_without_launch_events else "same pass as the per-kernel breakdown")}
    if ns_ms > 0:
        issued_total = sum(issued_flops.values())
        sus = peaks["bf16_tflops_sustained"]
        out["ns"] = {"ms_per_step": ns_ms,
                     "tflops_algorithmic": step_flops / (ns_ms / 1e3) / 1e12,
                     "tflops_issued": issued_total / (ns_ms / 1e3) / 1e12,
                     "tflops_dense_equivalent": dense_flops / (ns_ms / 1e3) / 1e12,
                     "frac_of_peak_algorithmic": step_flops / (ns_ms / 1e3) / 1e12 / sus,
                     "frac_of_peak_issued": issued_total / (ns_ms / 1e3) / 1e12 / sus,
                     "frac_of_peak_dense_equivalent": dense_flops / (ns_ms / 1e3) / 1e12 / sus}
    return out


def run_guarded(m, ws: WorkloadStep, n: int) -> dict:
    """The Muon step with the call-wide gradient guard on (skip on a
    non-finite gradient, clip by the global norm): an extra read of every
    gradient."""
    import torch
    stream = torch.cuda.current_stream()
    w = ws.w
    ghp = m.MuonHparams(**dict(workloads.MUON_HPARAMS, skip_nonfinite=True, max_grad_norm=1e9))
    for _ in range(2):
        ws.muon(stream, ghp)
    torch.cuda.synchronize()
    m.muon_set_timing(True)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(n):
        ws.muon(stream, ghp)
    g1.record(stream)
    torch.cuda.synchronize()
    gk = m.muon_timing_read()["grad_guard"]
    m.muon_set_timing(False)
    if m.muon_query_status(ws.batch.workspace) != 0:
        raise RuntimeError("device status set in the guarded run")
    g_bytes = sum(s.rows * s.cols * (2 if s.g_dtype.itemsize == 2 else 4) for s in w.matrices)
    guard_ms = gk[0] / n
    return {"muon_ms_per_step": g0.elapsed_time(g1) / n, "guard_kernels_ms_per_step": guard_ms,
            "guard_gbs": g_bytes / (guard_ms / 1e3) / 1e9, "guard_bytes_per_step": g_bytes, "steps": n,
            "settings": "skip_nonfinite=1, max_grad_norm=1e9"}


def run_graph(m, ws: WorkloadStep, n: int, world: int, max_over_ranks, dev) -> dict:
    """The Muon step captured once as a CUDA graph and replayed, alternating
    with eager calls so both see the same clocks."""
    import torch
    stream = torch.cuda.current_stream()
    flush = None
    if input_bytes(ws.w) < 4 * L2_BYTES:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    step_flops = sum(workload_flops(ws.w, ws.hp.ns_steps)[0].values())
    g = ws.batch.capture(ws.hp)
    for _ in range(2):
        g.launch(stream)
    torch.cuda.synchronize()
    ev = {"graph": [], "eager": []}
    gl0 = m.muon_launch_count()
    for _ in range(n):
        for kind in ("eager", "graph"):
            if flush is not None:
                with torch.cuda.stream(stream):
                    flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if kind == "graph":
                g.launch(stream)
            else:
                ws.muon(stream)
            b.record(stream)
            ev[kind].append((a, b))
    torch.cuda.synchronize()
    n_launch = (m.muon_launch_count() - gl0) / (2 * n)
    g.destroy()
    if m.muon_query_status(ws.batch.workspace) != 0:
        raise RuntimeError("device status set in the graph replays")
    g_times = [a.elapsed_time(b) for a, b in ev["graph"]]
    e_times = [a.elapsed_time(b) for a, b in ev["eager"]]
    g_ms = max_over_ranks(sum(g_times)) / n
    return {"muon_ms_per_step": g_ms, "value": aggregate_tflops(step_flops, n, world, g_ms * n),
            "median_ms": statistics.median(g_times), "eager_median_ms": statistics.median(e_times),
            "steps": n, "launches_per_step": n_launch,
            "timed": "per call, CUDA events around each graph launch and each eager Muon step, alternating"
                     + ("; L2 flushed before each" if flush is not None else "")}


E2E_SLOT_BYTES = 2 << 30


def e2e_pieces(ws: WorkloadStep, slot_bytes: int):
    """The step cut into pieces whose inputs fit one staging slot: runs of
    consecutive matrices (their W, G, M in; W, M out) and chunks of the AdamW
    buffers (p, g, m, v in; p, m, v out).  Each piece: (kind, inputs,
    outputs, matrix range or AdamW quad)."""
    w = ws.w
    Wf, Gf, Mf = ws.tens.storage
    offs = [0]
    for s in w.matrices:
        offs.append(offs[-1] + s.rows * s.cols)
    per_el = Wf.element_size() + Gf.element_size() + Mf.element_size()
    pieces = []
    a = 0
    while a < len(w.matrices):
        b = a + 1
        while b < len(w.matrices) and (offs[b + 1] - offs[a]) * per_el <= slot_bytes:
            b += 1
        lo, hi = offs[a], offs[b]
        pieces.append(("muon", [Wf[lo:hi], Gf[lo:hi], Mf[lo:hi]], [Wf[lo:hi], Mf[lo:hi]], (a, b)))
        a = b
    chunk = max(4, (slot_bytes // (4 * 4)) // 4 * 4)   # 16 B in per element, float4-aligned starts
    for buf in ws.adamw:
        n = buf.p.numel()
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            quad = tuple(x[lo:hi] for x in (buf.p, buf.g, buf.m, buf.v))
            pieces.append(("adamw", list(quad), [quad[0], quad[2], quad[3]], quad))
    return pieces


class StagingRing:
    """Two pinned host slots per kind of piece and direction.  A slot holds
    one region per tensor role (W, G, M or p, g, m, v), each sized for the
    largest piece of that kind; a piece copies from / to the first elements
    of each region."""

    def __init__(self, pieces, kind: str, direction: int):
        import torch
        mine = [p for p in pieces if p[0] == kind]
        roles = len(mine[0][direction]) if mine else 0
        self.caps = [-(-max(p[direction][r].numel() * p[direction][r].element_size() for p in mine) // 256) * 256
                     for r in range(roles)]
        self.dtypes = [mine[0][direction][r].dtype for r in range(roles)] if mine else []
        total = sum(self.caps)
        self.slots = [torch.empty(total, dtype=torch.uint8, pin_memory=True) for _ in range(2)] if mine else []
        self.bytes = 2 * total

    def views(self, slot: int, tensors):
        out, off = [], 0
        for cap, dt, t in zip(self.caps, self.dtypes, tensors):
            nbytes = t.numel() * t.element_size()
            out.append(self.slots[slot][off:off + nbytes].view(dt))
            off += cap
        return out


E2E_COPY_STREAMS = 2  # per direction: the host link carries more both ways with two (343 vs 312 GB/s)


def run_e2e(m, ws: WorkloadStep, step_flops: int, world: int, barrier, max_over_ranks, n_steps: int,
            slot_bytes: int = E2E_SLOT_BYTES) -> dict:
    """The step from host buffers and back through the public API, pipelined:
    piece g+1's host->device copy, piece g's step and piece g-1's
    device->host copy run concurrently, the copies of successive pieces
    alternating over E2E_COPY_STREAMS streams per direction."""
    import torch
    stream = torch.cuda.current_stream()
    pieces = e2e_pieces(ws, slot_bytes)
    rings = {(k, d): StagingRing(pieces, k, d) for k in ("muon", "adamw") for d in (1, 2)}
    # fill each input slot once with the synthetic data of the largest piece of its kind
    for kind in ("muon", "adamw"):
        mine = [p for p in pieces if p[0] == kind]
        if not mine:
            continue
        big = max(mine, key=lambda p: sum(t.numel() for t in p[1]))
        for slot in range(2):
            for v, t in zip(rings[(kind, 1)].views(slot, big[1]), big[1]):
                v.copy_(t)
    ops = []
    for kind, ins, outs, what in pieces:
        if kind == "muon":
            a, b = what
            batch = m.MuonBatch(ws.tens.W[a:b], ws.tens.G[a:b], ws.tens.M[a:b], workspace=ws.batch.workspace)
            ops.append(lambda st, batch=batch: batch.step(ws.hp, st))
        else:
            ops.append(lambda st, quad=what: m.adamw_step_batched([quad], ws.ahp, workloads.ADAMW_STEP, st))
    s_ins = [torch.cuda.Stream() for _ in range(E2E_COPY_STREAMS)]
    s_outs = [torch.cuda.Stream() for _ in range(E2E_COPY_STREAMS)]
    n = len(pieces)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    ev_out = [None] * n
    counters = {"muon": 0, "adamw": 0}

    def one_step():
        counters["muon"] = counters["adamw"] = 0
        for g, (kind, ins, outs, _) in enumerate(pieces):
            slot = counters[kind] % 2
            counters[kind] += 1
            s_in, s_out = s_ins[g % E2E_COPY_STREAMS], s_outs[g % E2E_COPY_STREAMS]
            with torch.cuda.stream(s_in):
                if ev_out[g] is not None:
                    s_in.wait_event(ev_out[g])
                for dst, src in zip(ins, rings[(kind, 1)].views(slot, ins)):
                    dst.copy_(src, non_blocking=True)
                ev_in[g].record(s_in)
            stream.wait_event(ev_in[g])
            ops[g](stream)
            ev_comp[g].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[g])
                for dst, src in zip(rings[(kind, 2)].views(slot, outs), outs):
                    dst.copy_(src, non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_out)
                ev_out[g] = e

    one_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st in s_ins:
        st.wait_event(e0)
    for _ in range(n_steps):
        one_step()
    for st in s_outs:
        stream.wait_stream(st)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / n_steps
    status = m.muon_query_status(ws.batch.workspace)
    if status != 0:
        raise RuntimeError(f"device status {status} in the end-to-end run")
    h2d = sum(t.numel() * t.element_size() for p in pieces for t in p[1])
    d2h = sum(t.numel() * t.element_size() for p in pieces for t in p[2])
    n_muon = sum(1 for p in pieces if p[0] == "muon")
    return {"value": step_flops * world / (e2e_ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_steps,
            "pipeline": f"{n_muon} Muon pieces (runs of matrices) and {n - n_muon} AdamW chunks per step; "
                        f"copy in / step / copy out, {E2E_COPY_STREAMS} copy streams per direction",
            "host_buffers": f"pinned staging ring, 2 slots per kind and direction, "
                            f"{sum(r.bytes for r in rings.values()) / 2**30:.1f} GiB; input slots hold the "
                            "first (largest) piece's synthetic data, re-sent for every piece",
            "host_link_gbs": (h2d + d2h) / (e2e_ms / 1e3) / 1e9}


def sub_record(m, name: str, args, peaks, dev, local_rank, barrier, max_over_ranks, world) -> dict:
    """One other workload, measured like the headline (Muon only: c1-c4
    have no AdamW buffers)."""
    import torch
    w = workloads.get(name)
    ws = WorkloadStep(m, w, dev, int(args.budget_gb * 2 ** 30))
    r = measure(m, ws, args.steps, args.warmup, peaks, dev, local_rank, barrier, max_over_ranks, world)
    rec = {"workload": f"{w.name}: {w.description}", "matrices": len(w.matrices), "value": r["value"],
           "unit": UNIT, "ms_per_step": r["ms_per_step"], "steps": args.steps, "ns": r.get("ns"),
           "stages": r["stages"], "roofline": r["roofline"], "gpu_launches": r["launches"],
           "clocks": r["clocks"], "l2_flushed": r["l2_flushed"], "step_time": r["step_time"]}
    if name == "c1" and not args.no_graph:
        rec["graph_replay"] = run_graph(m, ws, max(3, min(args.steps, 20)), world, max_over_ranks, dev)
    del ws
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, local_rank):
    import gc

    import torch
    import torch.distributed as dist
    import optimizer_muon_step_gb300 as m

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    m.load_library()
    peaks = measured_peaks()
    w = workloads.get(args.workload)
    if args.subset:
        w.matrices = w.matrices[:args.subset]
        w.description += f" (first {args.subset} matrices only, profiling subset)"

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, world, dev)

    ws = WorkloadStep(m, w, dev, int(args.budget_gb * 2 ** 30), with_adamw=not args.no_adamw,
                      adamw_params=args.adamw_params)
    head = measure(m, ws, args.steps, args.warmup, peaks, dev, local_rank, barrier, max_over_ranks, world,
                   subset=bool(args.subset))
    big = head["ms_per_step"] > 50
    adamw = None
    if ws.quads:
        a_ms = head["adamw_ms_per_step"]
        gbs = ADAMW_BYTES_PER_PARAM * ws.adamw_params / (a_ms / 1e3) / 1e9
        k = head["stages"]["adamw"]
        adamw = {"workload": ("embedding + LM head, " + " + ".join(f"{r}x{c}" for r, c in w.adamw_shapes)
                              if not args.adamw_params else
                              f"{len(ws.adamw)} x {args.adamw_params} fp32 parameters (profiling size)")
                 + f" fp32, t={workloads.ADAMW_STEP}, one adamw_step_batched call",
                 "params": ws.adamw_params, "ms_per_step": a_ms, "gbs": gbs,
                 "frac_of_hbm": gbs / peaks["hbm_gbs"], "frac_of_nominal_8tbs": gbs / 8000.0,
                 "kernel_ms_per_step": k["ms_per_step"], "kernel_gbs": k["gbs"],
                 "bytes_per_param": ADAMW_BYTES_PER_PARAM}
    guard = None if args.no_guard else run_guarded(m, ws, 3 if big else max(3, min(args.steps, 10)))
    graph = None if args.no_graph else run_graph(m, ws, 3 if big else max(3, min(args.steps, 20)), world,
                                                 max_over_ranks, dev)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(m, ws, head["step_flops"], world, barrier, max_over_ranks,
                      3 if big else max(3, min(args.steps, 10)))
    del ws
    gc.collect()
    torch.cuda.empty_cache()

    per_workload = None
    if not args.no_per_workload and not args.subset:
        per_workload = {}
        for name in SUB_WORKLOADS:
            if name != w.name:
                per_workload[name] = sub_record(m, name, args, peaks, dev, local_rank, barrier,
                                                max_over_ranks, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(w, workloads.MUON_HPARAMS["ns_steps"], world),
                "muon_ms_per_step": head["muon_ms_per_step"], "adamw": adamw,
                "roofline": head["roofline"], "ns": head.get("ns"), "stages": head["stages"],
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": head["launches"], "clocks": head["clocks"],
                "guarded_step": guard, "graph_replay": graph, "per_workload": per_workload}
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
