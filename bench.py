#!/usr/bin/env python3
"""Benchmark of the sm_103a fp16 GEMM (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline] [--cpu-threads T]

A step is one C = A*B of the workload (default: the MoE-flattened
131072 x 2048 x 7168 case of the C500 review, fp16 inputs, fp32 accumulation,
fp16 output) on inputs already resident in device memory.  L2 is flushed
before every timed step (a 512 MiB buffer written, then a second 512 MiB
buffer read, so the step finds neither its inputs nor dirty lines in L2) and
each step is bracketed by its own CUDA events on the launching stream, the
flush outside them.  `value` is
TFLOP/s of useful 2MNK work over all ranks.  `back_to_back` repeats the timing
with the steps run back to back (one replay of a CUDA graph of K calls, two
events around it, no flush): the warm figure of a serving loop.  `e2e` repeats the measurement
through the torch-level API with every step's inputs copied in from pinned host
memory and its result copied out inside the timed region, pipelined as a
serving loop runs it (two device slots; the copy-in of step i+1 and the
copy-out of step i-1 overlap the compute of step i on their own streams).  `roofline` rates the GEMM kernel against the
measured peak of this machine; `cpu_baseline` times the CPU oracle on a bounded
slab of output rows.

Multi-GPU: the GEMM does not need to be sharded to be measured; with torchrun
each rank runs an independent replica of the workload on its own GPU (weak
scaling, no collective on the data path) and rank 0 reports the aggregate.

--impl reference times the CPU oracle itself, as it stands, on bounded slabs of
the same workload (rank 0 only).
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

METRIC = "fp16 GEMM TFLOP/s (fp32 acc) and % of GB300 roofline; HBM GB/s at small M"

# The pages' own measurement of a bench workload (the only one they give): the
# C500 review's TileLang GEMM on the MoE-flattened shape, 117.25 TFLOPS.  Other
# hardware: `vs_baseline` against it is context, not a target.
PAGES_NUMBERS = {
    "moe_131072x2048x7168": (117.25, "TFLOP/s", "TileLang GEMM on a MetaX C500, the C500 review's final "
                             "version (other hardware: context, not a target)"),
}


def vs_pages(workload: str, value: float, unit: str):
    """(value / the pages' number for this workload, its description), or
    (None, None) when the pages give none in this unit."""
    ref = PAGES_NUMBERS.get(workload)
    if ref is None or ref[1] != unit:
        return None, None
    return round(value / ref[0], 3), f"{ref[0]} {ref[1]}: {ref[2]}"
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = ("flushed before every step (a 512 MiB buffer written, then another 512 MiB buffer read: "
           "no input lines and no dirty lines left in L2)")


class L2Flush:
    """Evicts L2 between timed steps: writing a buffer four times the L2's
    129 MB pushes every line of the previous step out; reading a second one
    then replaces the written (dirty) lines with clean ones, so the next step
    does not pay for writing the flush buffer back to HBM."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.out)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def kernel_source_hash() -> str:
    """First 16 hex digits of sha256 over the kernel sources (ptx, kernel, host,
    operand copy), with comments and blank space removed: a change of comment
    does not change the code the counters were taken on."""
    import hashlib
    import re

    csrc = os.path.join(ROOT, "dense_tiled_gemm_fp16_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("ptx.cuh", "gemm_kernel.cuh", "gemm_f16.cu", "repack.cuh"):
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    or None when there is none or it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", f"gemm_f16_persistent__{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "tflops": float(d["bf16_tflops"]),
                "tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and parts[1] != self.uuid:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def timed_steps(torch, dev, stream, steps, flush, step, graph_step, barrier):
    """Device time of `steps` steps on `stream` (ms), bracketed by a barrier
    and a synchronize on both sides; returns (total ms, wall seconds, timing note).

    With an L2 flush buffer every step is bracketed by its own CUDA events and
    the flush runs between them, outside.  Without one the steps run back to
    back: they are captured once as a CUDA graph of `steps` calls (graph_step(s)
    enqueues one step on stream s) and timed by two events around its replay,
    as a serving loop would run them."""
    if flush is None:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(steps):
                graph_step(cap)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return e0.elapsed_time(e1), time.perf_counter() - t0, "CUDA graph of the steps, events around its replay"
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    wall = time.perf_counter() - t0
    return sum(a.elapsed_time(b) for a, b in zip(starts, ends)), wall, "per-step CUDA events, L2 flushed between"


def max_over_ranks(pg, x: float, device) -> float:
    """x reduced with MAX over every rank of the process group (x itself when
    there is no group): the slowest rank's time is the job's time."""
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, steps: int, world: int, total_ms: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest
    rank's time (the replicas each process `units_per_step` per step)."""
    return units_per_step * steps * world / (total_ms * 1e-3)


def oracle_slab(w, rows: int, threads: int, fused=None):
    """(callable, FLOPs): the CPU oracle on the first `rows` output rows of the
    one-GEMM workload `w`; `fused` = (up projection operand or None, act) runs
    the fused output stage's oracle instead."""
    import numpy as np

    import oracle

    k = np.arange(w.K, dtype=np.int64)
    A_rows = np.ascontiguousarray(w.A.values_at(np.arange(rows)[:, None], k[None, :]))
    Bv = w.B.host_view()
    flops = 2.0 * rows * w.N * w.K
    if fused is None:
        return (lambda: oracle.gemm(A_rows, Bv, threads=threads)), flops
    up, act = fused
    if up is None:
        return (lambda: oracle.gemm_fused(A_rows, Bv, act=act, threads=threads)), flops
    Uv = up.host_view()
    return (lambda: oracle.gemm_fused(A_rows, Bv, Uv, act=act, threads=threads)), 2 * flops


def cpu_oracle_rate(w, target_s: float, threads: int, fused=None):
    """Time the CPU oracle on a slab of output rows (repeated when the whole
    problem takes less than the target); returns (TFLOP/s, rows, seconds, reps).
    The whole problem's time follows by linear extrapolation over the rows."""
    def slab(rows, reps=1):
        run, flops = oracle_slab(w, rows, threads, fused)
        t = time.perf_counter()
        for _ in range(reps):
            run()
        return time.perf_counter() - t, flops * reps

    rows = 1
    dt, _ = slab(rows)
    while dt < 0.5 and rows < w.M:
        rows = min(w.M, rows * 4)
        dt, _ = slab(rows)
    rate = rows / dt                              # rows per second
    rows = int(max(1, min(w.M, rate * target_s)))
    reps = max(1, min(100, int(target_s * rate / rows))) if rows == w.M else 1
    dt, flops = slab(rows, reps)
    return flops / dt / 1e12, rows, dt, reps


def back_to_back(torch, dev, stream, steps, step, graph_step, barrier, pg, flops, nbytes, world):
    """The warm figure: the same steps run back to back without a flush, as
    one replay of a CUDA graph of `steps` calls timed by two events."""
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    local_ms, _, note = timed_steps(torch, dev, stream, steps, None, step, graph_step, barrier)
    total_ms = max_over_ranks(pg, local_ms, dev)
    ms = total_ms / steps
    return {"value": round(whole_job_rate(flops, steps, world, total_ms) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 5), "hbm_gbs_min_traffic": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "timing": note + ", no flush (L2 warm)"}


# Timed regions at least this long (device time) run tensor-bound kernels
# under the power limit: their roofline is the sustained GEMM peak.  (On
# these boxes 20 MoE-shape steps, ~45 ms, ran at the maximum clock; 200
# steps, ~450 ms, showed sw_power_cap.)
SUSTAINED_AFTER_MS = 200.0


def roofline(bnd, flops, nbytes, ms_per_step, peaks, workload, busy_ms=0.0):
    """The dominant kernel against the measured peak.  Tensor-bound shapes in
    TFLOP/s: against the bf16 burst peak when the timed region is short (the
    kernel timed alone, one call per step), against the sustained peak when it
    lasts SUSTAINED_AFTER_MS or more (`busy_ms`, the steps' device time: the
    power limit then sets the clock, as in the sustained measurement); the
    fractions of both are given.  HBM-bound shapes in GB/s of algorithmic
    bytes against the copy bandwidth."""
    if bnd == "tensor":
        achieved = flops / (ms_per_step * 1e-3) / 1e12
        sustained = busy_ms >= SUSTAINED_AFTER_MS
        peak = peaks["tflops_sustained"] if sustained else peaks["tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "peak_kind": "sustained" if sustained else "burst",
                "frac_of_burst": round(achieved / peaks["tflops"], 4),
                "frac_of_sustained": round(achieved / peaks["tflops_sustained"], 4),
                "peak_burst": peaks["tflops"], "peak_sustained": peaks["tflops_sustained"],
                "timed_region_ms": round(busy_ms, 1)}
    else:
        achieved = nbytes / (ms_per_step * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": "copy bandwidth"}
    roof["traffic"] = profiled_traffic(workload)
    roof["peak_source"] = (f"{peaks['source']} (MEASURED_PEAKS.json: bf16 burst and sustained GEMM, "
                           "copy bandwidth)")
    roof["kernel"] = "gemm_f16_persistent"
    return roof


# Workloads small enough that a single-thread oracle run is also reported.
SINGLE_THREAD_CPU = ("tail_130x70x65_b_rowmajor", "tail_130x70x65_b_transposed", "decode_m16_n16384_k8192")


def cpu_baseline(w, seconds, threads, fused=None, label="oracle", name=None):
    """The CPU oracle, as it stands, on a slab of output rows with `threads`
    threads; the whole workload's time is extrapolated linearly over its rows.
    For the small workloads a single-thread run is reported beside it."""
    rate, r, dt, reps = cpu_oracle_rate(w, seconds, threads, fused)
    full_flops = 2.0 * w.M * w.N * w.K * (2 if fused is not None and fused[0] is not None else 1)
    out = {"value": round(rate, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{label}: {r} of {w.M} output rows x all {w.N} columns, K={w.K}"
                     f"{f', {reps} times' if reps > 1 else ''} ({dt:.1f} s)",
           "full_workload_s": round(full_flops / (rate * 1e12), 3),
           "full_workload_s_kind": "measured" if r == w.M else "extrapolated from the slab"}
    if (name or w.name) in SINGLE_THREAD_CPU and threads != 1:
        rate1, r1, dt1, reps1 = cpu_oracle_rate(w, min(seconds, 5.0), 1, fused)
        out["single_thread"] = {
            "value": round(rate1, 6), "unit": "TFLOP/s", "cores": 1,
            "sample": f"{r1} of {w.M} output rows{f', {reps1} times' if reps1 > 1 else ''} ({dt1:.1f} s)",
            "full_workload_s": round(full_flops / (rate1 * 1e12), 4)}
    return out


# -------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    import dense_tiled_gemm_fp16_gb300 as g
    from dense_tiled_gemm_fp16_gb300 import ledger
    from synth import workloads

    rank, world, local = dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()

    w = workloads.BY_NAME[args.workload]
    if isinstance(w, workloads.MultiWorkload):
        return run_ours_multi(args, w, dev, barrier, pg, rank, world)
    M, N, K = w.M, w.N, w.K
    flops = ledger.flops(M, N, K)
    nbytes = ledger.min_bytes(M, N, K)
    peaks = load_peaks()
    bnd = ledger.bound(M, N, K, peaks["tflops"], peaks["hbm_gbs"])

    A = w.A.device_view(dev)
    B = w.B.device_view(dev)
    C = torch.empty((M, N), dtype=torch.float16, device=dev)
    # L2 is flushed before every timed step, so no step finds the previous
    # step's inputs (or the flush's dirty lines) in L2.
    flush = L2Flush(torch, dev)
    l2_note = L2_NOTE
    stream = torch.cuda.current_stream(dev)
    plan = g.plan_for(A, B, C)
    # The C-ABI call with its arguments marshalled once (device pointers and
    # element strides of the resident operands).
    call_args = (A.data_ptr(), A.stride(0), A.stride(1), B.data_ptr(), B.stride(0), B.stride(1),
                 C.data_ptr(), C.stride(0), M, N, K)
    handle = stream.cuda_stream

    def step():
        g.gemm_f16(*call_args, stream=handle)

    def graph_step(s):
        g.gemm_f16(*call_args, stream=s.cuda_stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    assert g.gemm_f16_device_status() == 0

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    clocks = ClockSampler(str(uuid) if uuid else None)
    clocks.start()
    time.sleep(0.3)

    local_ms, wall, timing = timed_steps(torch, dev, stream, args.steps, flush, step, graph_step, barrier)
    clk = clocks.stop()
    l2_note += "; " + timing

    total_ms = max_over_ranks(pg, local_ms, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(flops, args.steps, world, total_ms) / 1e12
    b2b = back_to_back(torch, dev, stream, args.steps, step, graph_step, barrier, pg, flops, nbytes, world)

    # ---- end to end: pinned host inputs in, result out, inside the timed region
    if args.no_e2e:
        e2e_ms = float("nan")
    else:
        e2e_ms = run_e2e(args, w, dev, stream, C, barrier, pg)
    status = g.gemm_f16_device_status()
    result = None
    if rank == 0:
        result = report(args, w, plan, peaks, bnd, flops, nbytes, ms_per_step, value, wall, clk, e2e_ms,
                        world, status, A, B, l2_note)
        result["back_to_back"] = b2b
    if pg is not None:
        pg.destroy_process_group()
    return result


def run_ours_multi(args, w, dev, barrier, pg, rank, world):
    """Batched or grouped workload: one gemm_f16_batched / gemm_f16_grouped call
    per step over resident operands, timed like the one-GEMM workloads."""
    import numpy as np
    import torch

    import dense_tiled_gemm_fp16_gb300 as g

    M, N, K, n = w.M, w.N, w.K, w.count
    flops = w.flops
    fused = w.B_up is not None or w.act != "none"
    nB = 2 if w.B_up is not None else 1   # projections read per problem
    if w.kind == "batched":
        nbytes = 2.0 * n * (M * K + nB * K * N + M * N)
    else:
        nbytes = 2.0 * (M * K + nB * n * K * N + M * N)
    peaks = load_peaks()
    bnd = "tensor" if flops / nbytes * peaks["hbm_gbs"] * 1e9 > peaks["tflops"] * 1e12 else "hbm"
    A = w.A.device_view(dev)
    B = w.B.device_view(dev)
    U = w.B_up.device_view(dev) if w.B_up is not None else None
    C = torch.empty((w.c_rows, N), dtype=torch.float16, device=dev)
    in_bytes = 2 * (w.A.numel + w.B.numel + (w.B_up.numel if w.B_up is not None else 0))
    flush = L2Flush(torch, dev)
    l2_note = L2_NOTE
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    act = g.ACTIVATIONS[w.act]
    up = U.data_ptr() if U is not None else 0
    if w.kind == "batched" and not fused:
        call = (A.data_ptr(), M * K, K, 1, B.data_ptr(), K * N, N, 1, C.data_ptr(), M * N, N, M, N, K, n)

        def step(h=handle):
            g.gemm_f16_batched(*call, stream=h)
    elif w.kind == "batched":
        call = (A.data_ptr(), M * K, K, 1, B.data_ptr(), K * N, N, 1, up, 0, 0, 0, act, C.data_ptr(), M * N, N,
                M, N, K, n)

        def step(h=handle):
            g.gemm_f16_batched_fused(*call, stream=h)
    elif not fused:
        rows = list(w.group_rows)
        call = (A.data_ptr(), K, 1, B.data_ptr(), K * N, N, 1, C.data_ptr(), N, rows, N, K)

        def step(h=handle):
            g.gemm_f16_grouped(*call, stream=h)
    else:
        rows = list(w.group_rows)
        call = (A.data_ptr(), K, 1, B.data_ptr(), K * N, N, 1, up, 0, 0, 0, act, C.data_ptr(), N, rows, N, K)

        def step(h=handle):
            g.gemm_f16_grouped_fused(*call, stream=h)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    assert g.gemm_f16_device_status() == 0
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    clocks = ClockSampler(str(uuid) if uuid else None)
    clocks.start()
    time.sleep(0.3)
    local_ms, wall, timing = timed_steps(torch, dev, stream, args.steps, flush, step,
                                         lambda s: step(s.cuda_stream), barrier)
    clk = clocks.stop()
    l2_note += "; " + timing
    total_ms = max_over_ranks(pg, local_ms, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(flops, args.steps, world, total_ms) / 1e12
    b2b = back_to_back(torch, dev, stream, args.steps, step, lambda s: step(s.cuda_stream), barrier, pg, flops,
                       nbytes, world)

    e2e = None
    if not args.no_e2e:
        # pinned host operands in and C out inside the timed region, through the
        # torch-level wrappers a user calls
        A_h = torch.from_numpy(np.ascontiguousarray(w.A.host_buffer())).pin_memory()
        B_h = torch.from_numpy(np.ascontiguousarray(w.B.host_buffer())).pin_memory()
        U_h = (torch.from_numpy(np.ascontiguousarray(w.B_up.host_buffer())).pin_memory()
               if w.B_up is not None else None)
        C_h = [torch.empty(tuple(C.shape), dtype=torch.float16).pin_memory() for _ in range(2)]
        A_buf = [torch.empty(w.A.numel, dtype=torch.float16, device=dev) for _ in range(2)]
        B_buf = [torch.empty(w.B.numel, dtype=torch.float16, device=dev) for _ in range(2)]
        U_buf = [torch.empty(w.B_up.numel, dtype=torch.float16, device=dev) if U_h is not None else None
                 for _ in range(2)]
        Cs = [C, torch.empty_like(C)]

        def copy_in(k, s):
            with torch.cuda.stream(s):
                A_buf[k].copy_(A_h, non_blocking=True)
                B_buf[k].copy_(B_h, non_blocking=True)
                if U_h is not None:
                    U_buf[k].copy_(U_h, non_blocking=True)

        def compute(k, s):
            B3 = B_buf[k].view(n, K, N)
            U3 = U_buf[k].view(n, K, N) if U_h is not None else None
            if w.kind == "batched":
                A3, C3 = A_buf[k].view(n, M, K), Cs[k].view(n, M, N)
                if fused:
                    g.fused_mm(A3, B3, act=w.act, b_up=U3, out=C3, stream=s)
                else:
                    g.bmm(A3, B3, out=C3, stream=s)
            elif fused:
                g.grouped_fused_mm(A_buf[k].view(M, K), B3, list(w.group_rows), act=w.act, b_up=U3, out=Cs[k],
                                   stream=s)
            else:
                g.grouped_mm(A_buf[k].view(M, K), B3, list(w.group_rows), out=Cs[k], stream=s)

        def copy_out(k, s):
            with torch.cuda.stream(s):
                C_h[k].copy_(Cs[k], non_blocking=True)

        e2e_ms = pipelined_e2e(dev, stream, max(5, min(args.steps, 10)), args.warmup, copy_in, compute, copy_out,
                               barrier, pg)
        e2e = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(in_bytes),
               "d2h_bytes_per_step": int(2 * C.numel())}
    status = g.gemm_f16_device_status()
    if pg is not None:
        pg.destroy_process_group()
    if rank != 0:
        return None
    roof = roofline(bnd, flops, nbytes, ms_per_step, peaks, w.name, busy_ms=ms_per_step * args.steps)
    cpu = None
    if not args.no_cpu_baseline:
        threads = args.cpu_threads or os.cpu_count() or 1
        first = w.first_problem()
        fused = (w.first_up(), w.act) if (w.B_up is not None or w.act != "none") else None
        cpu = cpu_baseline(first, args.cpu_seconds, threads, fused,
                           ("fused-stage oracle" if fused else "oracle") + ", problem 0", name=w.name)
        # the whole launch's time, extrapolated from problem 0's rate
        cpu["full_workload_s"] = round(flops / (cpu["value"] * 1e12), 3)
        cpu["full_workload_s_kind"] = "extrapolated from problem 0's slab"
    config = {"workload": w.name, "kind": w.kind, "M": M, "N": N, "K": K, "problems": n,
              "fused_stage": ({"act": w.act, "gate_up": w.B_up is not None} if fused else None),
              "distribution": w.A.kind, "l2": l2_note,
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU", "options": args.opt}
    if w.kind == "grouped":
        config["group_rows"] = list(w.group_rows)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64 fill)", "config": config,
        "hbm_gbs_min_traffic": round(nbytes / (ms_per_step * 1e-3) / 1e9, 1),
        "wall_s_timed_region": round(wall, 4), "clocks": clk, "e2e": e2e, "gpu_launches": args.steps,
        "roofline": roof, "cpu_baseline": cpu, "device_status": status, "back_to_back": b2b,
    }


def pipelined_e2e(dev, stream, steps, warmup, copy_in, compute, copy_out, barrier, pg):
    """End-to-end steps as a serving loop runs them: two device slots, the
    host-to-device copy of step i+1 on one copy stream and the device-to-host
    copy of step i-1 on another while step i computes on `stream`.  Every
    step's copies and compute lie inside the timed region, which runs from
    before the first copy-in to after the last copy-out; returns ms per step.

    copy_in(slot, s), compute(slot, s), copy_out(slot, s) enqueue one step's
    work for device slot `slot` on stream `s`."""
    import torch

    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # slot_free[k]: the compute that last read slot k's inputs is done (its
    # inputs may be overwritten); out_free[k]: slot k's result has been copied out
    slot_free = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    for k in range(2):
        slot_free[k].record(stream)
        out_free[k].record(stream)

    def run(n):
        for i in range(n):
            k = i & 1
            h2d.wait_event(slot_free[k])
            copy_in(k, h2d)
            ready = torch.cuda.Event()
            ready.record(h2d)
            stream.wait_event(ready)
            stream.wait_event(out_free[k])
            compute(k, stream)
            slot_free[k].record(stream)
            d2h.wait_event(slot_free[k])
            copy_out(k, d2h)
            out_free[k].record(d2h)

    run(max(1, warmup))
    torch.cuda.synchronize(dev)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    es.record(h2d)
    run(steps)
    ee.record(d2h)
    torch.cuda.synchronize(dev)
    return max_over_ranks(pg, es.elapsed_time(ee) / steps, dev)


def run_e2e(args, w, dev, stream, C, barrier, pg):
    import numpy as np
    import torch

    import dense_tiled_gemm_fp16_gb300 as g

    M, N = w.M, w.N
    A_h = torch.from_numpy(np.ascontiguousarray(w.A.host_buffer())).pin_memory()
    B_h = torch.from_numpy(np.ascontiguousarray(w.B.host_buffer())).pin_memory()
    C_h = [torch.empty((M, N), dtype=torch.float16).pin_memory() for _ in range(2)]
    A_buf = [torch.empty(w.A.numel, dtype=torch.float16, device=dev) for _ in range(2)]
    B_buf = [torch.empty(w.B.numel, dtype=torch.float16, device=dev) for _ in range(2)]
    Cs = [C, torch.empty_like(C)]

    def views(k):
        A_v = A_buf[k].view(*w.A.buf_shape)
        B_v = B_buf[k].view(*w.B.buf_shape)
        return (A_v.t() if w.A.transposed else A_v), (B_v.t() if w.B.transposed else B_v)

    def copy_in(k, s):
        with torch.cuda.stream(s):
            A_buf[k].copy_(A_h, non_blocking=True)
            B_buf[k].copy_(B_h, non_blocking=True)

    def compute(k, s):
        A_v, B_v = views(k)
        g.matmul(A_v, B_v, out=Cs[k], stream=s)

    def copy_out(k, s):
        with torch.cuda.stream(s):
            C_h[k].copy_(Cs[k], non_blocking=True)

    return pipelined_e2e(dev, stream, max(10, min(args.steps, 30)), args.warmup, copy_in, compute, copy_out,
                         barrier, pg)


def report(args, w, plan, peaks, bnd, flops, nbytes, ms_per_step, value, wall, clk, e2e_ms, world,
           status, A, B, l2_note):
    M, N, K = w.M, w.N, w.K
    roof = roofline(bnd, flops, nbytes, ms_per_step, peaks, w.name, busy_ms=ms_per_step * args.steps)
    cpu = None
    if not args.no_cpu_baseline:
        threads = args.cpu_threads or os.cpu_count() or 1
        cpu = cpu_baseline(w, args.cpu_seconds, threads)
    e2e = None
    if e2e_ms == e2e_ms:   # not NaN
        e2e = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": int(2 * (w.A.numel + w.B.numel)),
               "d2h_bytes_per_step": int(2 * M * N)}
    vsb, vsb_ref = vs_pages(w.name, value, "TFLOP/s")
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": vsb,
        "vs_baseline_ref": vsb_ref,
        "dtype": "f16 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64 fill)",
        "config": {"workload": w.name, "M": M, "N": N, "K": K,
                   "A": f"strides {tuple(A.stride())}", "B": f"strides {tuple(B.stride())}",
                   "distribution": w.A.kind, "l2": l2_note,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "options": args.opt,
                   "plan": {k: plan[k] for k in ("swap_ab", "pair", "a_tma", "b_tma", "c_tma", "tile_n",
                                                 "splits", "streamk_tiles", "tail_split", "grid",
                                                 "stages", "repack")}},
        "hbm_gbs_min_traffic": round(nbytes / (ms_per_step * 1e-3) / 1e9, 1),
        "wall_s_timed_region": round(wall, 4),
        "clocks": clk,
        "e2e": e2e,
        # the GEMM kernel, plus the copy of operands TMA cannot address into an
        # aligned buffer (repack bits 0-1) and the copy of C out of one (bit 2)
        "gpu_launches": args.steps * (1 + (1 if plan["repack"] & 3 else 0) + (1 if plan["repack"] & 4 else 0)),
        "roofline": roof,
        "cpu_baseline": cpu,
        "device_status": status,
    }


# -------------------------------------------------------- reference arm
def run_reference(args):
    from synth import workloads

    rank, world, _ = dist_env()
    if rank != 0:
        return None
    w = workloads.BY_NAME[args.workload]
    fused = None
    if isinstance(w, workloads.MultiWorkload):   # the oracle on problem 0, at the same rate unit
        if w.B_up is not None or w.act != "none":
            fused = (w.first_up(), w.act)
        w = w.first_problem()
    threads = args.cpu_threads or os.cpu_count() or 1
    per_step = min(5.0, 150.0 / max(1, args.steps + args.warmup))
    # size one slab, then time warmup + steps slabs of that size
    _, rows, _, _ = cpu_oracle_rate(w, per_step, threads, fused)
    run, flops = oracle_slab(w, rows, threads, fused)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        run()
        times.append(time.perf_counter() - t)
    sec = sum(times) / len(times)
    value = flops / sec / 1e12
    sample = (f"{'fused-stage oracle: ' if fused else ''}{rows} of {w.M} output rows x all {w.N} columns, "
              f"K={w.K} per step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 accumulate of f16 inputs (CPU oracle)",
        "data": "synthetic (seeded SplitMix64 fill)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="moe_131072x2048x7168")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--shape", default=None,
                    help="M,N,K[,at][,bt]: an ad-hoc uniform[-1,1] workload instead of --workload (row-major; "
                         "at / bt make A / B transposed views of row-major buffers)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="threads of the CPU oracle baseline (default: every host core)")
    ap.add_argument("--opt", action="append", default=[],
                    help="library tuning knob NAME=VALUE, NAME an option of the library without its OPT_ prefix "
                         "(force_gather, splits, tile_n, panel, swap, max_ctas, l2_a, two_k_loads, ...)")
    args = ap.parse_args()
    if args.opt and args.impl == "ours":
        import dense_tiled_gemm_fp16_gb300 as g
        for kv in args.opt:
            k, v = kv.split("=")
            g.gemm_f16_set_option(getattr(g, "OPT_" + k.upper()), int(v))
    if args.shape:
        from synth import workloads
        parts = args.shape.split(",")
        M, N, K = (int(x) for x in parts[:3])
        at, bt = "at" in parts[3:], "bt" in parts[3:]
        name = f"rowmajor_{M}x{N}x{K}" + ("_at" if at else "") + ("_bt" if bt else "")
        workloads.BY_NAME[name] = workloads.Workload(
            name, M, N, K, workloads.Operand(M, K, "uniform", 21, transposed=at),
            workloads.Operand(K, N, "uniform", 22, transposed=bt),
            "ad-hoc uniform[-1,1] shape (row-major, or transposed views with at / bt)")
        args.workload = name
    if args.warmup < 3 and args.impl == "ours":
        log("note: fewer than 3 warm-up steps")
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
