#!/usr/bin/env python3
"""Benchmark of the Muon optimizer step on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2]
    python bench.py --impl reference ...      (the CPU oracle as the reference arm)

A step is one call of muon_step_batched over every hidden matrix of the
workload (default c2: dense 24-layer decoder, hidden 2048, FFN 5632, 168
matrices, bf16 gradients): momentum, normalisation, five Newton-Schulz
iterations on the tensor cores and the final update.  The AdamW step (the
last row of the hot path) is timed in the same run on the full-size
embedding + LM-head buffers of the mixed workload (2 x 163840 x 7168 fp32)
and reported under "adamw".

value: Newton-Schulz TFLOP/s over the whole step time, counting the
algorithmic flops (symmetry exploited) 3 m'^2 n' + m'^3 per matrix per
iteration, summed over all ranks; ms_per_step is the Muon step time.
Under torchrun every rank runs its own replica of the workload (weak
scaling, no collective on the data path).  The default workload's inputs
total > 12 GB, far larger than L2 (129 MB); a workload whose W, G and M fit
in 4 x L2 has L2 flushed between timed steps instead (a 512 MB write outside
the per-step events).

graph_replay: the same step captured once as a CUDA graph
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
KINDS = ("momentum_norm", "norm_finalize", "x0_rescale", "ns_syrk", "ns_poly", "ns_update",
         "final_update", "adamw", "grad_guard", "desc_upload", "stats")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c2", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--budget-gb", type=float, default=16.0, help="NS workspace budget")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-adamw", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-guard", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--subset", type=int, default=0,
                    help="profiling only: keep the first N matrices of the workload")
    ap.add_argument("--adamw-params", type=int, default=0,
                    help="profiling only: N parameters per AdamW buffer instead of the full embedding size")
    return ap.parse_args()


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
    when 256-row pair tiles waste at most 1/8 of the rows),
    the last column tile rounded to 16 (single), 32 (pairs) or 128 (pairs on
    64-aligned shapes)."""
    pad = _ceil(mp, 256) * 256 - mp
    chunked = mp % 64 == 0 and np_ % 64 == 0

    def col_widths(n, pair):
        q = (128 if chunked else 32) if pair else 16
        out = []
        for j in range(_ceil(n, 256)):
            rem = n - 256 * j
            out.append(256 if rem >= 256 else _ceil(rem, q) * q)
        return out

    def triangle(k):
        if pad * 8 <= mp:  # pairs: tiles (I, J >= I) of 256 x n_J
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
    if pad * 8 <= mp:
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
    return {"workload": f"{w.name}: {w.description}", "matrices": len(w.matrices),
            "muon_params": w.muon_params, "ns_steps": steps_ns,
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
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (profiles/ncu_traffic.json), scaled to the full workload; None when the
    kernel source changed since the capture or the workload differs."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)
        with open(os.path.join(ROOT, rec["source_file"]), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if sha != rec["source_sha256"] or workload != rec["workload"]:
            return None
        b = rec["captured_bytes"][kernel]
        return (b["read"] + b["write"]) * rec["scale_to_full_launch"]
    except Exception:
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
    return times, flops, desc, oracle.num_threads()


def run_reference(args, rank):
    if rank != 0:
        return
    w = workloads.get(args.workload)
    time_oracle(workloads.get("c1"), REFERENCE_STEP_FLOPS)  # build + warm the library
    for _ in range(args.warmup):
        time_oracle(w, REFERENCE_STEP_FLOPS)
    times, flops, desc, cores = time_oracle(w, REFERENCE_STEP_FLOPS, repeats=args.steps)
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

def layer_groups(w: workloads.Workload, n_groups: int):
    """Contiguous runs of matrices of about equal size (matrix boundaries)."""
    sizes = [s.rows * s.cols for s in w.matrices]
    total = sum(sizes)
    groups, start, acc = [], 0, 0
    for i, n in enumerate(sizes):
        acc += n
        if acc >= total * (len(groups) + 1) / n_groups or i == len(sizes) - 1:
            groups.append((start, i + 1))
            start = i + 1
    return groups


def run_e2e(m, w, tens, hp, stream, step_flops, world, barrier, max_over_ranks, n_steps, budget):
    """Muon step from pinned host buffers and back, pipelined over layer
    groups: group g+1's host->device copy, group g's step and group g-1's
    device->host copy run concurrently on three streams.  Every step copies
    all inputs (W, G, M) in and all results (W, M) out."""
    import torch
    Wf, Gf, Mf = tens.storage
    host = [t.cpu().pin_memory() for t in tens.storage]
    groups = layer_groups(w, 8)
    offs = [0]
    for s in w.matrices:
        offs.append(offs[-1] + s.rows * s.cols)
    ws_bytes = max(m.muon_workspace_size([(s.rows, s.cols) for s in w.matrices[a:b]], budget)
                   for a, b in groups)
    ws = m.allocate_workspace(ws_bytes)
    batches = [m.MuonBatch(tens.W[a:b], tens.G[a:b], tens.M[a:b], workspace=ws) for a, b in groups]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in groups]
    ev_comp = [torch.cuda.Event() for _ in groups]
    ev_out = [None for _ in groups]

    def one_step():
        for g, (a, b) in enumerate(groups):
            lo, hi = offs[a], offs[b]
            with torch.cuda.stream(s_in):
                if ev_out[g] is not None:
                    s_in.wait_event(ev_out[g])
                Wf[lo:hi].copy_(host[0][lo:hi], non_blocking=True)
                Gf[lo:hi].copy_(host[1][lo:hi], non_blocking=True)
                Mf[lo:hi].copy_(host[2][lo:hi], non_blocking=True)
                ev_in[g].record(s_in)
            stream.wait_event(ev_in[g])
            batches[g].step(hp, stream)
            ev_comp[g].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[g])
                host[0][lo:hi].copy_(Wf[lo:hi], non_blocking=True)
                host[2][lo:hi].copy_(Mf[lo:hi], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_out)
                ev_out[g] = e

    one_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(n_steps):
        one_step()
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / n_steps
    status = m.muon_query_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} in the end-to-end run")
    h2d = sum(t.numel() * t.element_size() for t in tens.storage)
    d2h = Wf.numel() * Wf.element_size() + Mf.numel() * Mf.element_size()
    return {"value": step_flops * world / (e2e_ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_steps,
            "pipeline": f"{len(groups)} layer groups, copy in / step / copy out on 3 streams",
            "host_to_device_gbs": (h2d + d2h) / (e2e_ms / 1e3) / 1e9}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import optimizer_muon_step_gb300 as m

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    m.load_library()
    peaks = measured_peaks()
    w = workloads.get(args.workload)
    if args.subset:
        w.matrices = w.matrices[:args.subset]
        w.description += f" (first {args.subset} matrices only, profiling subset)"
    hp = m.MuonHparams(**workloads.MUON_HPARAMS)
    steps_ns = hp.ns_steps
    tens = workloads.make_muon(w, device=dev)
    batch = m.MuonBatch(tens.W, tens.G, tens.M, budget_bytes=int(args.budget_gb * 2 ** 30))
    stage_flops, dense_flops, issued_flops = workload_flops(w, steps_ns)
    step_flops = sum(stage_flops.values())
    ew_bytes = elementwise_bytes(w)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, world, dev)

    for _ in range(args.warmup):
        batch.step(hp, stream)
    torch.cuda.synchronize()
    if m.muon_query_status(batch.workspace) != 0:
        raise RuntimeError("device status set during warm-up")
    in_bytes = sum(t.numel() * t.element_size() for t in tens.storage)
    assert in_bytes == input_bytes(w)
    flush = None
    if in_bytes < 4 * L2_BYTES:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    # ---- device-timed region ----
    clocks = ClockSampler(local_rank)
    m.muon_set_timing(True)
    launches0 = m.muon_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    if flush is None:
        ev0.record(stream)
        for _ in range(args.steps):
            batch.step(hp, stream)
        ev1.record(stream)
    else:
        step_events = []
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            batch.step(hp, stream)
            b.record(stream)
            step_events.append((a, b))
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    launches = m.muon_launch_count() - launches0
    kernel_times = m.muon_timing_read()
    m.muon_set_timing(False)
    status = m.muon_query_status(batch.workspace)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    if flush is None:
        ms_total = max_over_ranks(ev0.elapsed_time(ev1))
    else:
        ms_total = max_over_ranks(sum(a.elapsed_time(b) for a, b in step_events))
    ms_step = ms_total / args.steps
    value = aggregate_tflops(step_flops, args.steps, world, ms_total)

    # ---- per-kernel roofline (live, same timed region) ----
    stages = {}
    for k in KINDS:
        ms_k, n_k = kernel_times.get(k, (0.0, 0))
        if n_k:
            stages[k] = {"ms_per_step": ms_k / args.steps, "launches_per_step": n_k / args.steps}
    ns_kinds = [k for k in ("ns_syrk", "ns_poly", "ns_update") if k in stages]
    dominant = max(stages, key=lambda k: stages[k]["ms_per_step"])
    for k in ns_kinds:
        s = stages[k]
        s["tflops"] = stage_flops[k] / (s["ms_per_step"] / 1e3) / 1e12
        s["tflops_issued"] = issued_flops[k] / (s["ms_per_step"] / 1e3) / 1e12
    for k in ("momentum_norm", "final_update"):
        if k in stages:
            stages[k]["gbs"] = ew_bytes[k] / (stages[k]["ms_per_step"] / 1e3) / 1e9
    d = stages[dominant]
    if dominant in ns_kinds:
        per_launch = stage_flops[dominant] / d["launches_per_step"]
        ms_launch = d["ms_per_step"] / d["launches_per_step"]
        achieved = per_launch / (ms_launch / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        roofline = {"bound": "tensor", "kernel": dominant, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_kind": f"bf16 sustained, {peaks['source']}",
                    "algorithmic_per_launch": per_launch, "ms_per_launch": ms_launch,
                    "traffic": None if args.subset else ncu_traffic(dominant, w.name),
                    "traffic_unit": "bytes per launch (DRAM read + write, ncu)"}
    else:
        per_launch = ew_bytes[dominant] / d["launches_per_step"]
        ms_launch = d["ms_per_step"] / d["launches_per_step"]
        achieved = per_launch / (ms_launch / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_kind": f"HBM copy, {peaks['source']}",
                    "algorithmic_per_launch": per_launch, "ms_per_launch": ms_launch, "traffic": None}
    ns_ms = sum(stages[k]["ms_per_step"] for k in ns_kinds)
    issued_total = sum(issued_flops.values())
    ns_summary = {"ms_per_step": ns_ms,
                  "tflops_algorithmic": step_flops / (ns_ms / 1e3) / 1e12,
                  "tflops_issued": issued_total / (ns_ms / 1e3) / 1e12,
                  "frac_of_peak_issued": issued_total / (ns_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
                  "tflops_dense_equivalent": dense_flops / (ns_ms / 1e3) / 1e12,
                  "frac_of_peak_algorithmic": step_flops / (ns_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
                  "frac_of_peak_dense_equivalent": dense_flops / (ns_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"]}

    # ---- the step with the call-wide gradient guard on (skip on non-finite,
    # clip by the global norm): an extra read of every gradient ----
    guard = None
    if not args.no_guard:
        ghp = m.MuonHparams(**dict(workloads.MUON_HPARAMS, skip_nonfinite=True, max_grad_norm=1e9))
        for _ in range(2):
            batch.step(ghp, stream)
        torch.cuda.synchronize()
        m.muon_set_timing(True)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        n_guard = max(3, min(args.steps, 10))
        for _ in range(n_guard):
            batch.step(ghp, stream)
        g1.record(stream)
        torch.cuda.synchronize()
        gk = m.muon_timing_read()["grad_guard"]
        m.muon_set_timing(False)
        if m.muon_query_status(batch.workspace) != 0:
            raise RuntimeError("device status set in the guarded run")
        g_bytes = sum(s.rows * s.cols * (2 if s.g_dtype.itemsize == 2 else 4) for s in w.matrices)
        guard_ms = gk[0] / n_guard
        guard = {"ms_per_step": g0.elapsed_time(g1) / n_guard, "guard_kernels_ms_per_step": guard_ms,
                 "guard_gbs": g_bytes / (guard_ms / 1e3) / 1e9, "guard_bytes_per_step": g_bytes,
                 "settings": "skip_nonfinite=1, max_grad_norm=1e9"}

    # ---- the same step replayed from a captured CUDA graph, alternating
    # with eager calls so both see the same clocks ----
    graph = None
    if not args.no_graph:
        g = batch.capture(hp)
        for _ in range(2):
            g.launch(stream)
        torch.cuda.synchronize()
        n_graph = max(3, min(args.steps, 20))
        ev = {"graph": [], "eager": []}
        gl0 = m.muon_launch_count()
        for _ in range(n_graph):
            for kind in ("eager", "graph"):
                if flush is not None:
                    with torch.cuda.stream(stream):
                        flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                if kind == "graph":
                    g.launch(stream)
                else:
                    batch.step(hp, stream)
                b.record(stream)
                ev[kind].append((a, b))
        torch.cuda.synchronize()
        n_launch = (m.muon_launch_count() - gl0) / (2 * n_graph)
        g.destroy()
        if m.muon_query_status(batch.workspace) != 0:
            raise RuntimeError("device status set in the graph replays")
        g_times = [a.elapsed_time(b) for a, b in ev["graph"]]
        e_times = [a.elapsed_time(b) for a, b in ev["eager"]]
        g_ms = max_over_ranks(sum(g_times)) / n_graph
        graph = {"ms_per_step": g_ms, "value": aggregate_tflops(step_flops, n_graph, world, g_ms * n_graph),
                 "median_ms": statistics.median(g_times), "eager_median_ms": statistics.median(e_times),
                 "steps": n_graph, "launches_per_step": n_launch,
                 "timed": "per call, CUDA events around each graph launch and each eager step, alternating"
                          + ("; L2 flushed before each" if flush is not None else "")}

    # ---- end to end through the public API, host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(m, w, tens, hp, stream, step_flops, world, barrier, max_over_ranks,
                      max(3, min(args.steps, 10)), int(args.budget_gb * 2 ** 30))

    # ---- AdamW on the mixed workload's embedding + LM head ----
    adamw = None
    if not args.no_adamw:
        c5 = workloads.get("c5")
        ahp = m.AdamwHparams(**workloads.ADAMW_HPARAMS)
        sizes = [args.adamw_params or r * c for r, c in c5.adamw_shapes]
        bufs = [workloads.make_adamw(n, seed=c5.seed + i, device=dev) for i, n in enumerate(sizes)]
        n_params = sum(b.p.numel() for b in bufs)
        for _ in range(args.warmup):
            for b in bufs:
                m.adamw_step(b.p, b.g, b.m, b.v, ahp, workloads.ADAMW_STEP, stream)
        torch.cuda.synchronize()
        m.muon_set_timing(True)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(args.steps):
            for b in bufs:
                m.adamw_step(b.p, b.g, b.m, b.v, ahp, workloads.ADAMW_STEP, stream)
        a1.record(stream)
        torch.cuda.synchronize()
        at = m.muon_timing_read()["adamw"]
        m.muon_set_timing(False)
        a_ms = a0.elapsed_time(a1) / args.steps
        gbs = ADAMW_BYTES_PER_PARAM * n_params / (a_ms / 1e3) / 1e9
        k_ms = at[0] / at[1]
        k_gbs = ADAMW_BYTES_PER_PARAM * (n_params / len(bufs)) / (k_ms / 1e3) / 1e9
        a_desc = ("c5 AdamW: embedding + LM head, 2 x 163840x7168 fp32, t=100" if not args.adamw_params else
                  f"AdamW on 2 x {args.adamw_params} fp32 parameters (profiling size), t=100")
        adamw = {"workload": a_desc,
                 "params": n_params, "ms_per_step": a_ms, "gbs": gbs,
                 "frac_of_hbm": gbs / peaks["hbm_gbs"], "frac_of_nominal_8tbs": gbs / 8000.0,
                 "kernel_ms_per_launch": k_ms, "kernel_gbs": k_gbs,
                 "bytes_per_param": ADAMW_BYTES_PER_PARAM}
        del bufs

    # ---- CPU oracle baseline (rank 0, one GPU only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times, flops, desc, cores = time_oracle(w, CPU_BASELINE_FLOPS, repeats=1)
        cpu = {"value": flops / times[0] / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{desc}, of {len(w.matrices)} matrices (full Muon step otherwise), "
                         f"{times[0]:.1f} s"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(w, steps_ns, world),
                "roofline": roofline, "ns": ns_summary, "stages": stages, "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": launches, "clocks": clk, "adamw": adamw, "guarded_step": guard,
                "graph_replay": graph}
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
