#!/usr/bin/env python3
"""Benchmark: RMSNorm (and LayerNorm) forward + backward HBM throughput on GB300.

One step = one forward (rmsnorm_fwd) and one backward (rmsnorm_bwd: fused row
kernel + dgamma column reduction) over the whole workload, inputs resident in
HBM. Default workload: bf16, M = 65536 rows (8 sequences x 8192 tokens),
N = 4096, eps = 1e-6, x ~ 3*N(0,1), gamma = 1 + 0.1*N(0,1), dy ~ 1e-2*N(0,1).
Each tensor is 512 MiB, larger than L2 (129 MB), so no L2 flush is needed
between steps.

value  = algorithmic bytes of all ranks' steps / max-over-ranks time, in GB/s,
         where fwd bytes = 2*M*N*s + N*s + 4*M and bwd bytes = 3*M*N*s + 2*N*s + 4*M.
e2e    = the same metric through the C ABI with host buffers: each step copies
         x, gamma, dy from pinned host memory, runs both passes, and copies
         y, rstd, dx, dgamma back; copies in, kernels and copies out run as a
         pipeline on three streams over two buffer sets, so the two directions
         of the host link overlap. link_gbs / link_ceiling: plain copies of one
         step's bytes in both directions at once, timed in the same run.
roofline = the backward pass (the dominant cost) against the measured HBM copy
         bandwidth in MEASURED_PEAKS.json.
cpu_baseline / --impl reference = the CPU oracle (its C fp32-intermediate
         reference, rows split over every core of the process's affinity mask;
         cpu_baseline also times one thread and the fp64 golden) on a bounded
         row sample of the workload.
--static-rows: the RMSNorm plans without the row pool (every block keeps a fixed
         share of the rows), for comparison.

--double-backward: the step is one RMSNorm double backward (rmsnorm_bwd_bwd:
         fused row kernel + d_gamma column reduction) on the workload, with
         cotangents ddx ~ N(0,1), ddgamma ~ N(0,1); r comes from one untimed
         forward. Algorithmic bytes = 5*M*N*s + 3*N*s + 4*M (read x, dy, ddx,
         gamma, ddgamma, rstd; write d_dy, d_x, d_gamma).
--workload ln_*: the same step for LayerNorm (layernorm_fwd + layernorm_bwd:
         fused row kernel + dgamma/dbeta column reduction); its algorithmic
         bytes add beta and dbeta (N*s each) and the saved mean (4*M each way).

Multi-GPU (torchrun): one process per GPU, each running an independent replica
of the workload (weak scaling); there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
# Nominal HBM3e bandwidth of a GB300 (~8 TB/s); the >= 85 % target is stated
# against this figure, while frac_of_peak uses the measured copy bandwidth.
NOMINAL_HBM_GBS = 8000.0
METRIC = "RMSNorm fwd/bwd HBM GB/s & % of peak, bf16 M=65536 N=4096, 1 GB300"


def metric_for(w) -> str:
    if w.op == "layernorm":
        return f"LayerNorm fwd/bwd HBM GB/s & % of peak, {w.dtype} M={w.M} N={w.N}, 1 GB300"
    from rmsnorm_fwd_bwd_gb300 import inputs
    if w.name != inputs.HEADLINE:
        return f"RMSNorm fwd/bwd HBM GB/s & % of peak, {w.dtype} M={w.M} N={w.N}, 1 GB300"
    return METRIC


# --------------------------------------------------------------------------- #
# the two operations behind one interface
# --------------------------------------------------------------------------- #
class RmsOp:
    """RMSNorm: inputs x, g, dy; outputs y, r (rstd), dx, dg."""
    name = "rmsnorm"
    inputs = ("x", "g", "dy")
    outputs = ("y", "r", "dx", "dg")
    passes = (0, 1)
    kernel = "rmsnorm_bwd (fused row kernel + dgamma reduce)"

    def __init__(self, w):
        self.w = w

    def host_inputs(self):
        from rmsnorm_fwd_bwd_gb300 import inputs
        x, g, dy = inputs.workload_inputs(self.w)
        return {"x": x, "g": g, "dy": dy}

    def workspace_size(self, B):
        return B.rmsnorm_bwd_workspace_size(self.w.M, self.w.N, self.w.dtype)

    def fwd(self, B, b, s):
        w = self.w
        return B.rmsnorm_fwd(b["x"], b["g"], b["y"], b["r"], w.M, w.N, w.eps, w.dtype, int(w.offset), s)

    def bwd(self, B, b, s, wsz):
        w = self.w
        return B.rmsnorm_bwd(b["dy"], b["x"], b["g"], b["r"], b["dx"], b["dg"], w.M, w.N, w.dtype,
                             int(w.offset), b["ws"], wsz, s)

    def oracle_step(self, orc, h, a, rows):
        w = self.w
        x, dy = h["x"][a:a + rows], h["dy"][a:a + rows]
        orc.fwd_reference(x, h["g"], w.dtype, eps=w.eps, offset=w.offset)
        orc.bwd_reference(dy, x, h["g"], w.dtype, eps=w.eps, offset=w.offset)

    def golden_step(self, orc, h, a, rows):
        w = self.w
        x, dy = h["x"][a:a + rows], h["dy"][a:a + rows]
        orc.fwd_golden(x, h["g"], w.dtype, eps=w.eps, offset=w.offset)
        orc.bwd_golden(dy, x, h["g"], w.dtype, eps=w.eps, offset=w.offset)

    def step_bytes(self, rows):
        s, N = self.w.elem_bytes, self.w.N
        return (2 * rows * N * s + N * s + 4 * rows) + (3 * rows * N * s + 2 * N * s + 4 * rows)


class LnOp(RmsOp):
    """LayerNorm: inputs x, g, b, dy; outputs y, m (mean), r (rstd), dx, dg, db."""
    name = "layernorm"
    inputs = ("x", "g", "b", "dy")
    outputs = ("y", "m", "r", "dx", "dg", "db")
    passes = (2, 3)
    kernel = "layernorm_bwd (fused row kernel + dgamma/dbeta reduce)"

    def host_inputs(self):
        from rmsnorm_fwd_bwd_gb300 import inputs
        x, g, b, dy = inputs.workload_inputs(self.w)
        return {"x": x, "g": g, "b": b, "dy": dy}

    def workspace_size(self, B):
        return B.layernorm_bwd_workspace_size(self.w.M, self.w.N, self.w.dtype)

    def fwd(self, B, b, s):
        w = self.w
        return B.layernorm_fwd(b["x"], w.N, b["g"], b["b"], b["y"], w.N, b["m"], b["r"], w.M, w.N, w.eps,
                               w.dtype, s)

    def bwd(self, B, b, s, wsz):
        w = self.w
        return B.layernorm_bwd(b["dy"], w.N, b["x"], w.N, b["g"], b["m"], b["r"], b["dx"], w.N, b["dg"],
                               b["db"], w.M, w.N, w.dtype, b["ws"], wsz, s)

    def oracle_step(self, orc, h, a, rows):
        w = self.w
        x, dy = h["x"][a:a + rows], h["dy"][a:a + rows]
        orc.ln_fwd_reference(x, h["g"], h["b"], w.dtype, eps=w.eps)
        orc.ln_bwd_reference(dy, x, h["g"], w.dtype, eps=w.eps)

    def golden_step(self, orc, h, a, rows):
        w = self.w
        x, dy = h["x"][a:a + rows], h["dy"][a:a + rows]
        orc.ln_fwd_golden(x, h["g"], h["b"], w.dtype, eps=w.eps)
        orc.ln_bwd_golden(dy, x, h["g"], w.dtype, eps=w.eps)

    def step_bytes(self, rows):
        s, N = self.w.elem_bytes, self.w.N
        return (2 * rows * N * s + 2 * N * s + 8 * rows) + (3 * rows * N * s + 3 * N * s + 8 * rows)


def op_for(w):
    return LnOp(w) if w.op == "layernorm" else RmsOp(w)


# --------------------------------------------------------------------------- #
# distributed plumbing (also exercised on CPU with gloo by the tests)
# --------------------------------------------------------------------------- #
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_step_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step_per_rank * steps / max_seconds / 1e9


# --------------------------------------------------------------------------- #
# clocks
# --------------------------------------------------------------------------- #
def clock_log_path(args, rank: int) -> str:
    """Where the raw clock samples of this rank go: --clock-log DIR, else the
    system's temporary directory (the JSON line carries their summary)."""
    import tempfile
    d = args.clock_log or tempfile.gettempdir()
    os.makedirs(d, exist_ok=True)
    return os.path.join(d, f"clocks_rank{rank}.csv")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        self.f = None
        self.gpu = gpu_index
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            if self.f is not None:
                self.f.close()
                self.f = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t_start: float, t_end: float):
        del t_start, t_end
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            lines = f.readlines()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- #
# helpers
# --------------------------------------------------------------------------- #
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest(sources=None) -> str:
    """Digest of the kernel sources: the named files of csrc/ (their names and
    contents), or every file there when sources is None."""
    csrc = os.path.join(ROOT, "rmsnorm_fwd_bwd_gb300", "csrc")
    paths = (sorted(glob.glob(os.path.join(csrc, "*"))) if sources is None
             else [os.path.join(csrc, n) for n in sorted(sources)])
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str, plan=None, path=None):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current
    sources of the kernels it covers (the entry's "sources": the kernels' files and
    the shared headers; every kernel file when absent) and, when the entry records
    one, with the launch plan `plan` (rmsnorm_describe_plan's text)."""
    path = path or os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    try:
        digest = kernel_source_digest(rec.get("sources"))
    except OSError:
        return None
    if rec.get("source_digest") != digest:
        return None
    if "plan" in rec and rec["plan"] != plan:
        return None
    return rec.get("dram_bytes_per_launch")


def host_cores() -> int:
    """Cores in this process's affinity mask."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def run_oracle_rows(step, orc, h, start: int, rows: int, threads: int) -> None:
    """step(orc, h, a, r) over rows [start, start + rows), split into contiguous
    chunks on `threads` threads. The oracle's C calls release the GIL (ctypes),
    so the chunks run in parallel; each chunk's dgamma is its own partial sum
    (combining a few N-vectors is negligible next to the rows)."""
    threads = max(1, min(threads, rows))
    if threads == 1:
        step(orc, h, start, rows)
        return
    from concurrent.futures import ThreadPoolExecutor
    bounds = [(start + rows * i // threads, start + rows * (i + 1) // threads) for i in range(threads)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda ab: step(orc, h, ab[0], ab[1] - ab[0]), bounds))


def oracle_rate(w, h, step, threads: int, budget_s: float):
    """Time `step` (the fp32 reference or the fp64 golden, fwd + bwd) on a row
    sample sized to about budget_s seconds on `threads` threads. Returns (GB/s
    of algorithmic bytes, rows, seconds)."""
    from oracle import oracle as orc
    op = op_for(w)
    orc.build()

    def run(rows):
        t = time.perf_counter()
        run_oracle_rows(step, orc, h, 0, rows, threads)
        return time.perf_counter() - t

    probe = min(64 * threads, w.M)
    t = run(probe)
    rows = int(min(w.M, max(probe, probe * budget_s / max(t, 1e-6))))
    t = run(rows)
    return op.step_bytes(rows) / t / 1e9, rows, t


def cpu_baseline(w, h, budget_s: float):
    """The CPU oracle on this host: the fp32-intermediate reference on every core
    of the affinity mask (the headline figure) and on one thread, and the fp64
    golden on every core, each on a bounded row sample of the workload."""
    op = op_for(w)
    cores = host_cores()
    rate, rows, t = oracle_rate(w, h, op.oracle_step, cores, budget_s / 3)
    rate1, rows1, t1 = oracle_rate(w, h, op.oracle_step, 1, budget_s / 3)
    rateg, rowsg, tg = oracle_rate(w, h, op.golden_step, cores, budget_s / 3)
    return {"value": rate, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} rows of the workload, fwd+bwd fp32-intermediate reference, "
                      f"rows split over {cores} threads, {t:.1f} s",
            "single_thread": {"value": rate1, "unit": "GB/s", "cores": 1,
                              "sample": f"first {rows1} rows, {t1:.1f} s"},
            "golden_fp64": {"value": rateg, "unit": "GB/s", "cores": cores,
                            "sample": f"first {rowsg} rows, fwd+bwd fp64 golden, {tg:.1f} s"}}


# --------------------------------------------------------------------------- #
# the reference arm: the CPU oracle
# --------------------------------------------------------------------------- #
def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import oracle as orc
    op = op_for(w)
    h = op.host_inputs()
    orc.build()
    cores = host_cores()
    total_budget = 60.0
    probe = min(w.M, 64 * cores)
    t0 = time.perf_counter()
    run_oracle_rows(op.oracle_step, orc, h, 0, probe, cores)
    per_row = (time.perf_counter() - t0) / probe
    rows = int(max(1, min(w.M, total_budget / max(args.steps + args.warmup, 1) / max(per_row, 1e-9))))
    starts = [(i * rows) % max(1, w.M - rows + 1) for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        run_oracle_rows(op.oracle_step, orc, h, starts[i], rows, cores)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        run_oracle_rows(op.oracle_step, orc, h, starts[i], rows, cores)
    dt = time.perf_counter() - t0
    value = op.step_bytes(rows) * args.steps / dt / 1e9
    sample = (f"{rows} consecutive rows of the {w.M}x{w.N} workload per step, "
              f"split over {cores} threads")
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_flush(buf):
    """Evict the L2 between timed steps: write a buffer 4x the L2, then read it,
    so the lines left in L2 are clean (no write-back of the flush's own data
    lands inside the next timed kernel). Runs outside the timed events."""
    import torch
    buf.zero_()
    buf.view(torch.int32).sum()


def needs_flush(w) -> bool:
    """Workloads whose tensors are under 256 MB each flush the L2 between timed
    passes; larger ones stream more than the L2 holds anyway."""
    return w.M * w.N * w.elem_bytes < 256e6


def workload_config(w):
    title = "LayerNorm" if w.op == "layernorm" else "RMSNorm"
    return {"workload": f"{title} fwd+bwd {w.dtype} M={w.M} N={w.N} eps={w.eps:g}"
                        + (" offset" if w.offset else ""),
            "name": w.name, "M": w.M, "N": w.N, "io_dtype": w.dtype, "offset": w.offset,
            "l2": "L2 flushed before each pass (512 MB written then read, outside the events)"
            if needs_flush(w) else "inputs larger than L2 (no flush)",
            "parallelism": "replicas"}


def protocol_median_us(fn, stream, flush=None, warmup_calls=20, samples=50, calls=20):
    """The pages' timing protocol for one pass: warm-up calls, then `samples`
    samples of `calls` back-to-back calls each, bracketed by CUDA events on the
    launching stream; returns the median over samples of the per-call time (us).
    With `flush`, the L2 is flushed before each sample, outside the events."""
    import torch
    for _ in range(warmup_calls):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(samples)]
    for a, b in ev:
        if flush is not None:
            l2_flush(flush)
        a.record(stream)
        for _ in range(calls):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) * 1e3 / calls for a, b in ev)


def link_copy_seconds(pairs_in, pairs_out, dev, reps=3):
    """Plain pinned-memory copies of one step's bytes, host to device on one
    stream and device to host on another at the same time (the link is full
    duplex); the best of `reps`. pairs_in: (device dst, host src); pairs_out:
    (host dst, device src)."""
    import torch
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = None
    for _ in range(reps):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        e0.record(cur)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        with torch.cuda.stream(s_in):
            for d, h in pairs_in:
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in pairs_out:
                h.copy_(d, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)
        e1.record(cur)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        best = t if best is None else min(best, t)
    return best


def pipelined_e2e_seconds(steps, sets, houts, copy_in, compute, copy_out, compute_stream, dev):
    """End-to-end timing of `steps` steps through the public API with host
    buffers, as a three-stage pipeline on three streams: step k's host-to-device
    copies (copy_in), its kernels (compute, on compute_stream) and its
    device-to-host copies (copy_out) use buffer set k % 2, so the copies in of
    step k + 1 overlap the kernels and the copies out of step k (the host link
    is full duplex). Events order each stage after the one before it in the
    same step and after the stage of step k - 2 that last used the same set.
    Returns the seconds from the first copy in to the last copy out."""
    import torch
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_k = compute_stream

    def ev():
        return torch.cuda.Event()

    def run(n):
        done_in, done_k, done_out = [], [], []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_k)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for k in range(n):
            b, ho = sets[k % 2], houts[k % 2]
            if k >= 2:
                s_in.wait_event(done_k[k - 2])      # the set's inputs were consumed by step k - 2
            with torch.cuda.stream(s_in):
                copy_in(b, s_in)
            done_in.append(ev())
            done_in[k].record(s_in)
            s_k.wait_event(done_in[k])
            if k >= 2:
                s_k.wait_event(done_out[k - 2])     # the set's outputs were copied out by step k - 2
            compute(b, s_k)
            done_k.append(ev())
            done_k[k].record(s_k)
            s_out.wait_event(done_k[k])
            with torch.cuda.stream(s_out):
                copy_out(b, ho, s_out)
            done_out.append(ev())
            done_out[k].record(s_out)
        s_k.wait_stream(s_in)
        s_k.wait_stream(s_out)
        e1.record(s_k)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    run(2)  # warm-up: both sets touched once
    return run(steps)


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def run_ours(args, w):
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    if args.static_rows:
        assert B.rmsnorm_set_row_pool(False) == B.RMSNORM_OK
    op = op_for(w)
    dt = w.dtype
    M, N = w.M, w.N

    h_np = op.host_inputs()
    # pinned host copies of the inputs (the end-to-end leg copies them in every step)
    host = {k: B.to_device(v.reshape(-1), dt, "cpu").pin_memory() for k, v in h_np.items()}
    wsz = op.workspace_size(B)

    def device_set():
        b = {k: v.to(dev) for k, v in host.items()}
        b["y"] = torch.empty_like(b["x"])
        b["dx"] = torch.empty_like(b["x"])
        b["dg"] = torch.empty_like(b["g"])
        if "db" in op.outputs:
            b["db"] = torch.empty_like(b["g"])
        for k in ("m", "r"):
            if k in op.outputs:
                b[k] = torch.empty(M, dtype=torch.float32, device=dev)
        b["ws"] = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)
        return b

    bufs = device_set()
    flush = None
    if needs_flush(w):
        flush = torch.empty(int(512e6), dtype=torch.uint8, device=dev)

    def fwd():
        st = op.fwd(B, bufs, stream)
        if st:
            raise B.RMSNormError(st, f"{op.name} forward")

    def bwd():
        st = op.bwd(B, bufs, stream, wsz)
        if st:
            raise B.RMSNormError(st, f"{op.name} backward")

    B.rmsnorm_device_error(clear=True)
    for _ in range(args.warmup):
        if flush is not None:
            l2_flush(flush)
        fwd()
        bwd()
    torch.cuda.synchronize()

    K = args.steps
    # events per step: fwd start, fwd end, bwd start, bwd end. Workloads that fit
    # in L2 flush it before each pass, outside the events, so that every pass
    # starts from a clean L2 (the convention of ncu's cache control); the larger
    # ones run back to back (bwd start = fwd end).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local, clock_log_path(args, rank))
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for k in range(K):
        if flush is not None:
            l2_flush(flush)
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        if flush is not None:
            l2_flush(flush)
        ev[k][2].record(stream)
        bwd()
        ev[k][3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # the pages' protocol per pass (after the timed region; not part of `value`)
    proto = None
    if not args.no_protocol:
        proto = {"fwd_us_median": protocol_median_us(fwd, stream, flush),
                 "bwd_us_median": protocol_median_us(bwd, stream, flush)}
    clocks.stop()
    fwd_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    bwd_ms = [ev[k][2].elapsed_time(ev[k][3]) for k in range(K)]
    if flush is None:
        total_ms = ev[0][0].elapsed_time(ev[K - 1][3])
    else:
        total_ms = sum(fwd_ms) + sum(bwd_ms)
    dev_err = B.rmsnorm_device_error(clear=True)

    secs = max_over_ranks(total_ms / 1e3, world, device=dev)
    step_bytes = w.fwd_bytes() + w.bwd_bytes()
    value = aggregate(step_bytes, K, world, secs)

    # end to end through the C ABI with host buffers: every step copies its inputs
    # in from pinned host memory and its results back out, pipelined over two
    # buffer sets (pipelined_e2e_seconds)
    e2e_steps = 0 if args.no_e2e else max(3, min(K, args.e2e_steps))
    out_names = [k for k in op.outputs]
    sets = [bufs, device_set()] if e2e_steps else None
    houts = ([{k: torch.empty(bufs[k].numel(), dtype=bufs[k].dtype).pin_memory() for k in out_names}
              for _ in range(2)] if e2e_steps else None)

    def copy_in(b, s):
        for name in op.inputs:
            b[name].copy_(host[name], non_blocking=True)

    def compute(b, s):
        st = op.fwd(B, b, s) or op.bwd(B, b, s, wsz)
        if st:
            raise B.RMSNormError(st, "end-to-end step")

    def copy_out(b, ho, s):
        for name in out_names:
            ho[name].copy_(b[name].view(-1), non_blocking=True)

    e2e_secs = None
    if e2e_steps:
        barrier(world)
        e2e_secs = max_over_ranks(pipelined_e2e_seconds(e2e_steps, sets, houts, copy_in, compute, copy_out,
                                                        stream, dev), world, device=dev)
    h2d = sum(host[k].numel() * host[k].element_size() for k in op.inputs)
    d2h = sum(bufs[k].numel() * bufs[k].element_size() for k in out_names)
    link_s = None
    if e2e_steps:
        # the host link alone: the same bytes as one step's copies, no kernels
        link_s = link_copy_seconds([(bufs[k], host[k]) for k in op.inputs],
                                   [(houts[0][k], bufs[k].view(-1)) for k in out_names], dev)

    if rank != 0:
        return 0
    peak, peak_kind = measured_peak()
    bwd_avg_ms = statistics.mean(bwd_ms)
    fwd_avg_ms = statistics.mean(fwd_ms)
    bwd_gbs = w.bwd_bytes() / (bwd_avg_ms / 1e3) / 1e9
    fwd_gbs = w.fwd_bytes() / (fwd_avg_ms / 1e3) / 1e9

    def pass_entry(nbytes, times_ms, pass_id):
        mean_ms = statistics.mean(times_ms)
        med_ms = statistics.median(times_ms)
        gbs = nbytes / (mean_ms / 1e3) / 1e9
        return {"us": mean_ms * 1e3, "us_median": med_ms * 1e3, "gbs": gbs,
                "gbs_median": nbytes / (med_ms / 1e3) / 1e9, "frac_of_peak": gbs / peak,
                "frac_of_nominal_peak": gbs / NOMINAL_HBM_GBS, "bytes": nbytes,
                "plan": B.rmsnorm_describe_plan(pass_id, M, N, dt)}

    e2e = None
    if e2e_steps:
        e2e_value = step_bytes * e2e_steps / e2e_secs / 1e9 * world
        ceiling = step_bytes / link_s / 1e9
        e2e = {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "link_gbs": (h2d + d2h) / link_s / 1e9,
               "link_ceiling": ceiling, "frac_of_link_ceiling": e2e_value / world / ceiling,
               "link_note": "link_gbs: one step's h2d and d2h bytes copied at once (pinned, both directions, "
                            "no kernels), best of 3; link_ceiling: the e2e value those copies alone allow"}
    if proto is not None:
        proto.update({"fwd_gbs": w.fwd_bytes() / proto["fwd_us_median"] / 1e3,
                      "bwd_gbs": w.bwd_bytes() / proto["bwd_us_median"] / 1e3,
                      "warmup_calls": 20, "samples": 50, "calls_per_sample": 20,
                      "l2": "flushed before each sample" if flush is not None
                      else "inputs larger than L2"})
    p_fwd, p_bwd = op.passes
    traffic = recorded_traffic(f"{op.name}_bwd {w.name}", plan=B.rmsnorm_describe_plan(p_bwd, M, N, dt))
    line = {
        "metric": metric_for(w), "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": secs * 1e3 / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if dt == "float32" else
        {"bfloat16": "bf16", "float16": "f16"}[dt],
        "data": "synthetic (seeded; see rmsnorm_fwd_bwd_gb300/inputs.py)",
        "config": dict(workload_config(w), **({"bwd_rows": "static (no row pool)"} if args.static_rows else {})),
        "fwd": pass_entry(w.fwd_bytes(), fwd_ms, p_fwd),
        "bwd": pass_entry(w.bwd_bytes(), bwd_ms, p_bwd),
        "roofline": {"bound": "hbm", "kernel": op.kernel,
                     "achieved": bwd_gbs, "peak": peak, "peak_kind": f"{peak_kind} HBM copy",
                     "unit": "GB/s", "frac": bwd_gbs / peak, "traffic": traffic,
                     "algorithmic_bytes": w.bwd_bytes(), "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal_peak": bwd_gbs / NOMINAL_HBM_GBS,
                     "target": ">= 0.85 of the nominal peak (frac_of_nominal_peak); frac is of the measured copy"},
        "protocol": proto,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "device_error_word": dev_err,
        "clocks": clocks.summary(0, 0),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, h_np, args.cpu_budget)
    print(json.dumps(line), flush=True)
    return 0


def run_double_backward(args, w):
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    from rmsnorm_fwd_bwd_gb300 import inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    dt, M, N, s = w.dtype, w.M, w.N, w.elem_bytes
    x_np, g_np, dy_np = inputs.workload_inputs(w)
    ddx_np = inputs.to_storage(inputs.normal(w.seed, 3, (M, N)), dt)
    ddg_np = inputs.to_storage(inputs.normal(w.seed, 4, (N,)), dt)
    host = {k: B.to_device(v.reshape(-1), dt, "cpu").pin_memory()
            for k, v in (("x", x_np), ("g", g_np), ("dy", dy_np), ("ddx", ddx_np), ("ddg", ddg_np))}
    wsz = B.rmsnorm_bwd_bwd_workspace_size(M, N, dt)

    def device_set():
        b = {k: v.to(dev) for k, v in host.items()}
        b["r"] = torch.empty(M, dtype=torch.float32, device=dev)
        b["d_dy"] = torch.empty_like(b["x"])
        b["d_x"] = torch.empty_like(b["x"])
        b["d_g"] = torch.empty_like(b["g"])
        b["ws"] = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)
        y = torch.empty_like(b["x"])
        st = B.rmsnorm_fwd(b["x"], b["g"], y, b["r"], M, N, w.eps, dt, int(w.offset), stream)
        if st:
            raise B.RMSNormError(st, "rmsnorm_fwd")
        return b

    def step(b, strm):
        return B.rmsnorm_bwd_bwd(b["ddx"], N, b["ddg"], b["dy"], N, b["x"], N, b["g"], b["r"], b["d_dy"], N,
                                 b["d_x"], N, b["d_g"], M, N, dt, int(w.offset), b["ws"], wsz, strm)

    bufs = device_set()
    flush = None
    if needs_flush(w):
        flush = torch.empty(int(512e6), dtype=torch.uint8, device=dev)
    B.rmsnorm_device_error(clear=True)
    for _ in range(args.warmup):
        if flush is not None:
            l2_flush(flush)
        st = step(bufs, stream)
        if st:
            raise B.RMSNormError(st, "rmsnorm_bwd_bwd")
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local, clock_log_path(args, rank))
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for k in range(K):
        if flush is not None:
            l2_flush(flush)
        ev[k][0].record(stream)
        step(bufs, stream)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks.stop()
    if flush is None:
        total_ms = ev[0][0].elapsed_time(ev[K - 1][1])
    else:
        total_ms = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(K))
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    dev_err = B.rmsnorm_device_error(clear=True)
    secs = max_over_ranks(total_ms / 1e3, world, device=dev)
    nbytes = 5 * M * N * s + 3 * N * s + 4 * M
    value = aggregate(nbytes, K, world, secs)

    # end to end with host buffers: each step copies ddx, ddgamma, dy, x, gamma and
    # rstd in and d_dy, d_x, d_gamma out, pipelined as in the main bench
    e2e_steps = 0 if args.no_e2e else max(3, min(K, args.e2e_steps))
    sets = [bufs, device_set()] if e2e_steps else None
    r_host = bufs["r"].cpu().pin_memory()
    houts = ([{k: torch.empty(bufs[k].numel(), dtype=bufs[k].dtype).pin_memory() for k in ("d_dy", "d_x", "d_g")}
              for _ in range(2)] if e2e_steps else None)

    def copy_in(b, strm):
        for name in ("ddx", "ddg", "dy", "x", "g"):
            b[name].copy_(host[name], non_blocking=True)
        b["r"].copy_(r_host, non_blocking=True)

    def compute(b, strm):
        st = step(b, strm)
        if st:
            raise B.RMSNormError(st, "end-to-end double backward")

    def copy_out(b, ho, strm):
        for name in ("d_dy", "d_x", "d_g"):
            ho[name].copy_(b[name].view(-1), non_blocking=True)

    e2e_secs = None
    if e2e_steps:
        barrier(world)
        e2e_secs = max_over_ranks(pipelined_e2e_seconds(e2e_steps, sets, houts, copy_in, compute, copy_out,
                                                        stream, dev), world, device=dev)
    h2d = sum(host[k].numel() * host[k].element_size() for k in host) + 4 * M
    d2h = 2 * M * N * s + N * s
    if rank != 0:
        return 0
    peak, peak_kind = measured_peak()
    avg_ms = statistics.mean(step_ms)
    gbs = nbytes / (avg_ms / 1e3) / 1e9
    line = {
        "metric": f"RMSNorm double backward HBM GB/s & % of peak, {dt} M={M} N={N}, 1 GB300",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if dt == "float32" else {"bfloat16": "bf16", "float16": "f16"}[dt],
        "data": "synthetic (seeded; see rmsnorm_fwd_bwd_gb300/inputs.py; cotangents tags 3 and 4)",
        "config": dict(workload_config(w), workload=f"RMSNorm double backward {dt} M={M} N={N} eps={w.eps:g}"
                       + (" offset" if w.offset else "")),
        "dbwd": {"us": avg_ms * 1e3, "gbs": gbs, "frac_of_peak": gbs / peak, "bytes": nbytes,
                 "plan": B.rmsnorm_describe_plan(4, M, N, dt)},
        "roofline": {"bound": "hbm", "kernel": "rmsnorm_bwd_bwd (fused row kernel + d_gamma reduce)",
                     "achieved": gbs, "peak": peak, "peak_kind": f"{peak_kind} HBM copy", "unit": "GB/s",
                     "frac": gbs / peak, "traffic": recorded_traffic(f"rmsnorm_bwd_bwd {w.name}",
                                                                plan=B.rmsnorm_describe_plan(4, M, N, dt)),
                     "algorithmic_bytes": nbytes},
        "e2e": ({"value": nbytes * e2e_steps / e2e_secs / 1e9 * world, "unit": "GB/s",
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}
                if e2e_steps else None),
        "gpu_launches": 2 * K,
        "device_error_word": dev_err,
        "clocks": clocks.summary(0, 0),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the headline)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=24.0,
                    help="seconds of oracle work (three legs: all cores, one thread, fp64 golden)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-protocol", action="store_true",
                    help="skip the per-pass medians of the pages' protocol (20 warm-up calls, 50 samples x 20)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (one device set only; for profiler captures)")
    ap.add_argument("--clock-log", default=None,
                    help="directory for the raw nvidia-smi clock samples (default: the temporary directory)")
    ap.add_argument("--double-backward", action="store_true",
                    help="time the RMSNorm double backward on the workload instead of fwd+bwd")
    ap.add_argument("--rows", type=int, default=None,
                    help="override the row count M (small cases for profiler captures)")
    ap.add_argument("--static-rows", action="store_true",
                    help="RMSNorm forward and backward without the row pool (every block keeps a fixed share of the rows)")
    args = ap.parse_args(argv)
    import dataclasses
    from rmsnorm_fwd_bwd_gb300 import inputs
    w = inputs.WORKLOADS[args.workload or inputs.HEADLINE]
    if args.rows is not None:
        w = dataclasses.replace(w, M=args.rows, name=f"{w.name}@rows={args.rows}")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.double_backward:
        if w.op != "rmsnorm":
            ap.error("--double-backward applies to RMSNorm workloads")
        return run_double_backward(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
