#!/usr/bin/env python
"""Benchmark of libgemv on GB300: achieved HBM GB/s (cold L2) and % of the measured peak.

One step = one GEMV of the largest single-GPU configuration: bf16 y = A.x with A
128256 x 4096 (1.05 GB of weights, the Llama-3 vocabulary projection), one vector,
no bias.  Inputs are resident in HBM; L2 is flushed (a write, then a read, of
twice the L2 size) before every GEMV; each GEMV is timed with CUDA events on the
stream it runs on.

    value      = Q_min of the step / mean step time            (GB/s, whole job)
    Q_min      = M*K*s_A + B*K*s_x + B*M*s_y                   (per GEMV)
    roofline   = the step's kernel: its Q_min / its mean event time, against the
                 measured HBM copy bandwidth; traffic = DRAM bytes read + written
                 per launch from a committed ncu capture of the same kernel source
    e2e        = the same metric through gemv_host (the C-ABI call on host buffers):
                 A and x copied in from pinned host memory and y copied back,
                 inside the timed region, every step
    cpu_baseline = the CPU oracle on the same GEMV, on all host cores and on one
    fp32_step  = the fp32 configurations with bias at M = 16384 over K in
                 {16, 32, 4096}: three GEMVs, timed the same way
    sweep      = every configuration at its full size, timed the same way, plus
                 the int4 and tensor-core workloads, with the vendor library's
                 time for the same product (torch.matmul, i.e. cuBLAS) beside
                 the floating-point ones without bias
    decode_layer = a Llama-3-8B-shaped bf16 layer's four GEMVs, eager and from a
                 CUDA graph, and again with the residual adds and SwiGLU fused
                 into the GEMV epilogues

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs the same workload on its own GPU (replicas: the
GEMV needs no exchange between GPUs); value adds the ranks' bytes over the
slowest rank's time.  ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "GEMV achieved HBM GB/s (cold L2) & % of GB300 peak; µs per y=A·x"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# What the step's kernel is made of: the CUDA-core kernels' source and the launcher of
# its family (comments stripped), and the launch configuration the dispatcher picks
# for the workload.  The DRAM traffic of a committed ncu capture is reported only
# while these are unchanged.
KERNEL_SOURCE = "gemv_kernels.cuh"
LAUNCH_SOURCE = ("gemv_launch.cuh", "cudaError_t launch_rowteam(")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
HEADLINE_DESC = "bf16 GEMV y = A.x, A 128256x4096 row-major (1.05 GB), B = 1, no bias: 1 GEMV per step"
FP32_STEP_DESC = "f32 GEMV + bias at M=16384 over K in {16, 32, 4096}: 3 GEMVs per step"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-configuration sweep")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--sweep-iters", type=int, default=100)
    ap.add_argument("--only", default=None, help="sweep only these comma-separated configs")
    ap.add_argument("--sweep-only", action="store_true",
                    help="only the per-configuration sweep (e.g. under ncu); prints one JSON line")
    ap.add_argument("--sweep-bare", action="store_true",
                    help="sweep without the vendor-library and back-to-back legs (for ncu launch lists)")
    ap.add_argument("--force", default=None,
                    help="with --sweep-only: run every configuration on this kernel family where it "
                         "applies (rows_per_warp, warp_per_row, block_per_row, split_k, batched, "
                         "scalar, stream, xsplit, tc), through the library's test hook; "
                         "family:param passes the hook's parameter (e.g. batched:1 for the row pairs)")
    return ap.parse_args(argv)


def max_over_ranks(v: float, pg=None) -> float:
    """The largest value over all ranks (the slowest rank's time), via the process group."""
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank_step: int, step_ms: float) -> float:
    """Bytes of all ranks' steps over the slowest rank's step time, in GB/s."""
    return world * bytes_per_rank_step / (step_ms * 1e-3) / 1e9


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def code_only(src: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed: what the
    compiler sees, so that an edit to a comment does not change the hash."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_sha(workload: str) -> str:
    """Hash of the step kernel's code and of its launch configuration for `workload`."""
    csrc = os.path.join(ROOT, "decode_linear_layers_gb300", "csrc")
    h = hashlib.sha256()
    with open(os.path.join(csrc, KERNEL_SOURCE), encoding="utf-8") as fh:
        h.update(code_only(fh.read()).encode())
    with open(os.path.join(csrc, LAUNCH_SOURCE[0]), encoding="utf-8") as fh:
        src = fh.read()
    i = src.index(LAUNCH_SOURCE[1])
    j = src.find("\ntemplate", i)
    h.update(code_only(src[i:j if j >= 0 else len(src)]).encode())
    import decode_linear_layers_gb300 as g

    w = W.BY_NAME[workload]
    plan = g.plan_for(w.dtype, w.M, w.K, w.B)
    h.update(json.dumps({k: plan[k] for k in sorted(plan) if k != "kernel_name"}, sort_keys=True).encode())
    return h.hexdigest()[:16]


def read_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it is for this kernel."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    sha = kernel_sha(workload)
    cur = None
    for line in open(TRAFFIC_FILE):
        parts = line.split()
        if len(parts) >= 2 and parts[0] == "kernel_sha":
            cur = parts[1]
        elif len(parts) >= 3 and parts[0] == workload and parts[1] == "traffic_bytes" and cur == sha:
            return int(parts[2].replace(",", ""))
    return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak_tflops():
    """Dense bf16 tensor throughput (burst) measured on this GPU model, else the
    fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        self.marks = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.perf_counter(), [c.strip() for c in line.split(",")]))

    def wait_first(self, timeout=5.0):
        t0 = time.perf_counter()
        while self.proc is not None and not self.rows and time.perf_counter() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for (_, r) in self.rows[-3:]]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(torch, dev) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


# ------------------------------------------------------------------ our arm
def call_gemv(g, w, d, y):
    if w.dtype in ("w8", "w4"):
        getattr(g, f"gemv_{w.dtype}")(d["A"], d["scale"], d["x"], d["bias"], y, w.M, w.K, w.B)
    else:
        getattr(g, f"gemv_{w.dtype}")(d["A"], d["x"], d["bias"], y, w.M, w.K, w.B)


def out_dtype(torch, dtype):
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "w8": torch.bfloat16,
            "w4": torch.bfloat16}[dtype]


def l2_flush(flush):
    """Evict L2: write a buffer twice the L2 size, then read it back, so that L2
    holds clean lines of unrelated data (no dirty lines of the flush itself are left
    to be written back inside the next timed kernel)."""
    flush.zero_()
    flush.sum()


def time_gemvs(torch, g, items, flush, iters, warmup):
    """Per-GEMV CUDA-event times (ms), L2 flushed before each launch."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for (w, d, y) in items:
            l2_flush(flush)
            call_gemv(g, w, d, y)
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in items] for _ in range(iters)]
    for s in range(iters):
        for i, (w, d, y) in enumerate(items):
            l2_flush(flush)
            ev[s][i][0].record(stream)
            call_gemv(g, w, d, y)
            ev[s][i][1].record(stream)
    torch.cuda.synchronize()
    return [[ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(iters)] for i in range(len(items))]


def run_ours(args, rank, world, local_rank):
    import torch
    import decode_linear_layers_gb300 as g

    g.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    def allmax(v: float) -> float:
        return max_over_ranks(v, pg)

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024) or 126 * 1024 * 1024)
    flush = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev)
    peak, peak_kind = measured_peaks()

    if args.sweep_only:
        if args.force:
            kname, _, kparam = args.force.partition(":")
            g.force_kernel(kname, int(kparam or 0))
        try:
            if rank == 0:
                print(json.dumps({"sweep": sweep(args, torch, g, dev, flush, peak)}), flush=True)
        finally:
            g.force_kernel("auto")
        return None

    head = [W.BY_NAME[n] for n in W.HEADLINE]
    host_inputs = [W.make_inputs(w) for w in head]
    items = device_items(torch, dev, head, host_inputs)

    # ---- device-resident timed region (the clock sampler starts before the warm-up,
    # so that starting nvidia-smi does not land in a timed launch)
    sampler = ClockSampler(gpu_id_for(torch, dev)) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    for _ in range(args.warmup):
        for (w, d, y) in items:
            l2_flush(flush)
            call_gemv(g, w, d, y)
    barrier()
    n0 = g.launch_count()
    t0 = time.perf_counter()
    times = time_gemvs(torch, g, items, flush, args.steps, 0)
    barrier()
    t1 = time.perf_counter()
    launches = g.launch_count() - n0
    if sampler:
        sampler.stop()
    per_gemv_ms = [statistics.mean(t) for t in times]
    step_ms = allmax(sum(per_gemv_ms))
    step_bytes = sum(w.qmin_bytes for w in head)
    value = whole_job_gbs(world, step_bytes, step_ms)

    dom = max(range(len(head)), key=lambda i: per_gemv_ms[i])
    wd = head[dom]
    dom_ms = per_gemv_ms[dom]
    achieved = wd.qmin_bytes / (dom_ms * 1e-3) / 1e9
    plans = []
    for (w, d, y) in items:
        call_gemv(g, w, d, y)
        plans.append(g.last_plan())
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": read_traffic(wd.name),
                "kernel": plans[dom]["kernel_name"], "workload": wd.name, "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": wd.qmin_bytes, "mean_us": round(dom_ms * 1e3, 3)}

    # ---- end to end: host buffers, copies inside the timed region
    e2e = None
    if rank == 0 or world > 1:
        e2e = end_to_end(args, torch, g, items, host_inputs, barrier, allmax, world)

    # ---- the fp32 three-GEMV step (rows per warp, warp per row, long rows)
    fp32 = fp32_step(args, torch, g, dev, flush, peak)

    if rank != 0:
        if pg is not None:
            pg.barrier()
        return None

    clocks = sampler.summary(t0, t1) if sampler else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded PCG64: A ~ N(0, 0.02^2), x ~ N(0, 1), rounded to bf16)",
        "config": headline_config(world),
        "per_gemv_us": {w.name: round(t * 1e3, 3) for w, t in zip(head, per_gemv_ms)},
        # the distribution behind each mean: one slow launch moves a mean of 200
        "per_gemv_us_median": {w.name: round(statistics.median(t) * 1e3, 3) for w, t in zip(head, times)},
        "per_gemv_us_max": {w.name: round(max(t) * 1e3, 3) for w, t in zip(head, times)},
        "per_gemv_kernel": {w.name: p["kernel_name"] for w, p in zip(head, plans)},
        "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
        "wall_s_timed_region": round(t1 - t0, 3),
        "fp32_step": fp32,
        "launch_floor_us": round(launch_floor_us(torch, g, dev, flush), 3),
    }

    if not args.no_sweep:
        line["sweep"] = sweep(args, torch, g, dev, flush, peak)
        line["decode_layer"] = decode_layer(args, torch, g, dev, flush, peak)
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(head, host_inputs)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
    return line


def device_items(torch, dev, ws, host_inputs):
    """(workload, device inputs, device y) per workload."""
    items = []
    for w, inp in zip(ws, host_inputs):
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        items.append((w, d, torch.empty((w.B, w.M), dtype=out_dtype(torch, w.dtype), device=dev)))
    return items


def end_to_end(args, torch, g, items, host_inputs, barrier, allmax, world):
    """The step through gemv_host: every input copied in from pinned host memory and
    y copied back to it, inside the timed region (one CUDA-event interval over all
    steps)."""
    pinned = []
    for (w, d, y), inp in zip(items, host_inputs):
        hp = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
        hy = torch.empty((w.B, w.M), dtype=y.dtype).pin_memory()
        pinned.append((hp, hy))
    h2d = sum(sum(v.numel() * v.element_size() for v in hp.values() if v is not None) for hp, _ in pinned)
    d2h = sum(hy.numel() * hy.element_size() for _, hy in pinned)
    steps = max(3, min(args.steps, 50))
    step_bytes = sum(w.qmin_bytes for (w, _, _) in items)

    def e2e_step():
        # the library's host-buffer call: it copies A, scale, x, bias in, runs the
        # GEMV and copies y out (one cudaMemcpyAsync per buffer), all on the stream
        for (w, d, y), (hp, hy) in zip(items, pinned):
            g.gemv_host(w.dtype, hp["A"], hp["scale"], hp["x"], hp["bias"], hy,
                        d["A"], d["scale"], d["x"], d["bias"], y, w.M, w.K, w.B)

    for _ in range(2):
        e2e_step()
    barrier()
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record()
    for _ in range(steps):
        e2e_step()
    e_ev.record()
    torch.cuda.synchronize()
    ms = allmax(s_ev.elapsed_time(e_ev) / steps)
    return {"value": round(whole_job_gbs(world, step_bytes, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "steps": steps}


def fp32_step(args, torch, g, dev, flush, peak):
    """The three fp32 GEMVs with bias at M = 16384 (K = 16, 32, 4096), each timed
    like the headline: Q_min of the three over the sum of their mean times."""
    ws = [W.BY_NAME[n] for n in W.FP32_STEP]
    items = device_items(torch, dev, ws, [W.make_inputs(w) for w in ws])
    times = time_gemvs(torch, g, items, flush, max(20, min(args.steps, 200)), 3)
    means = [statistics.mean(t) for t in times]
    kernels = []
    for (w, d, y) in items:
        call_gemv(g, w, d, y)
        kernels.append(g.last_plan()["kernel_name"])
    nbytes = sum(w.qmin_bytes for w in ws)
    gbs = nbytes / (sum(means) * 1e-3) / 1e9
    return {"workload": FP32_STEP_DESC, "value": round(gbs, 2), "unit": UNIT,
            "ms_per_step": round(sum(means), 5), "frac_of_peak": round(gbs / peak, 4),
            "per_gemv_us": {w.name: round(t * 1e3, 3) for w, t in zip(ws, means)},
            "per_gemv_kernel": {w.name: k for w, k in zip(ws, kernels)}}


def sweep(args, torch, g, dev, flush, peak):
    """Every configuration at full size (and the int4 workloads): µs, GB/s and
    fraction of peak."""
    out = []
    names = [w.name for w in W.CONFIGS + W.W4_CONFIGS + W.TC_CONFIGS]
    if args.only:
        names = [n for n in names if n in args.only.split(",")]
    for n in names:
        w = W.BY_NAME[n]
        inp = W.make_inputs(w)
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        del inp
        y = torch.empty((w.B, w.M), dtype=out_dtype(torch, w.dtype), device=dev)
        t = time_gemvs(torch, g, [(w, d, y)], flush, args.sweep_iters, 3)[0]
        plan = g.last_plan()
        # single event intervals come in steps of about 2 us on GB300, so a median
        # snaps to a step; the mean over the launches is the figure reported
        mean = statistics.mean(t)
        ts = sorted(t)
        gbs = w.qmin_bytes / (mean * 1e-3) / 1e9
        out.append({"config": n, "kernel": plan["kernel_name"], "us_mean": round(mean * 1e3, 3),
                    "us_median": round(statistics.median(t) * 1e3, 3),
                    "us_p10": round(ts[len(ts) // 10] * 1e3, 3), "us_p90": round(ts[(9 * len(ts)) // 10] * 1e3, 3),
                    "qmin_bytes": w.qmin_bytes, "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                    "gflops": round(w.flops / (mean * 1e-3) / 1e9, 1),
                    "roofline_us": round(w.qmin_bytes / (peak * 1e9) * 1e6, 3)})
        if plan["kernel_name"] == "tc":  # a contraction on the tensor cores: its own roofline too
            tp, _ = measured_tensor_peak_tflops()
            out[-1]["frac_of_tensor_peak"] = round(w.flops / (mean * 1e-3) / 1e12 / tp, 4)
        if args.sweep_bare:
            del d, y
            torch.cuda.empty_cache()
            continue
        if w.dtype in ("f32", "f16", "bf16") and not w.bias:
            # context: the vendor library's time for the same product on the same
            # tensors (torch.matmul -> cuBLAS), timed the same way
            out[-1]["torch_linear_us"] = round(library_linear_us(torch, d, y, flush, args.sweep_iters) * 1e3, 3)
        b2b = back_to_back_us(torch, g, w, d, y, flush)
        out[-1]["us_back_to_back"] = round(b2b["us"], 3)
        out[-1]["frac_of_peak_back_to_back"] = round(w.qmin_bytes / (b2b["us"] * 1e-6) / 1e9 / peak, 4)
        out[-1]["back_to_back_copies"] = b2b["copies"]
        del d, y
        torch.cuda.empty_cache()
    return out


def launch_floor_us(torch, g, dev, flush, iters=100):
    """Mean CUDA-event time of the library's least-work launch (fp32, M = 1, K = 0:
    one CTA writes y = 0), timed like every GEMV: the fixed cost of a single launch
    between two events on this GPU, which no kernel design can remove."""
    y = torch.empty((1, 1), dtype=torch.float32, device=dev)
    for _ in range(5):
        g.gemv_f32(None, None, None, y, 1, 0, 1)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    stream = torch.cuda.current_stream()
    for e0, e1 in ev:
        l2_flush(flush)
        e0.record(stream)
        g.gemv_f32(None, None, None, y, 1, 0, 1)
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3


def back_to_back_us(torch, g, w, d, y, flush, rounds=3):
    """Per-GEMV time (us) of the workload launched back to back, as a decode loop
    runs its GEMVs: A rotates over enough device copies that together they exceed
    twice the L2 size (so every launch reads its weights from HBM), x and y stay;
    one CUDA-event interval over 8 passes of the copies, mean over `rounds`."""
    twice_l2 = flush.numel() * flush.element_size()  # the flush buffer is twice the L2 size
    abytes = d["A"].numel() * d["A"].element_size()
    copies = max(1, min(16, -(-twice_l2 // abytes)))
    As = [d["A"]] + [d["A"].clone() for _ in range(copies - 1)]
    n = max(8, 8 * copies)
    dd = dict(d)

    def run():
        for i in range(n):
            dd["A"] = As[i % copies]
            call_gemv(g, w, dd, y)

    run()
    times = []
    for _ in range(rounds):
        l2_flush(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / n)
    del As
    return {"us": statistics.mean(times), "copies": copies}


def library_linear_us(torch, d, y, flush, iters):
    """Mean CUDA-event time (ms) of the vendor library's product y = x A^T (B x M)
    on the same device tensors (torch.matmul into y: cuBLAS), L2 flushed before
    each call."""
    x, A = d["x"], d["A"]
    for _ in range(3):
        l2_flush(flush)
        torch.matmul(x, A.t(), out=y)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    stream = torch.cuda.current_stream()
    for e0, e1 in ev:
        l2_flush(flush)
        e0.record(stream)
        torch.matmul(x, A.t(), out=y)
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)


# A Llama-3-8B-shaped decode layer (bf16, one token): fused QKV, output
# projection, fused gate+up, down projection.
DECODE_LAYER = (("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096), ("down", 4096, 14336))


def decode_layer(args, torch, g, dev, flush, peak, iters=20):
    """The layer's four GEMVs back to back, eager and replayed from a CUDA graph.

    L2 is flushed once before each layer (not between its GEMVs); the weights
    (434 MB) do not fit in L2 anyway."""
    ws = [W.Workload(f"bf16_{n}", "bf16", M, K, 1, False, ("normal", 0.02), ("normal", 1.0), seed=i)
          for i, (n, M, K) in enumerate(DECODE_LAYER)]
    items = []
    for w in ws:
        inp = W.make_inputs(w)
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        items.append((w, d, torch.empty((1, w.M), dtype=torch.bfloat16, device=dev)))
    layer_bytes = sum(w.qmin_bytes for w in ws)

    def run():
        for (w, d, y) in items:
            call_gemv(g, w, d, y)

    def timed(fn):
        out = []
        for i in range(iters + 3):
            l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                out.append(e0.elapsed_time(e1))
        return statistics.mean(out)  # event intervals come in ~2 us steps: the mean, not a median

    eager_ms = timed(run)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    n0 = g.launch_count()
    with torch.cuda.graph(graph):
        run()
    launches = g.launch_count() - n0
    graph_ms = timed(graph.replay)
    iso = time_gemvs(torch, g, items, flush, iters, 3)
    iso_ms = sum(statistics.mean(t) for t in iso)
    fused = decode_layer_fused(torch, g, dev, items, timed)
    # the same layer with plain launches (no programmatic dependent launch)
    g.set_launch_overlap("off")
    try:
        plain_eager_ms = timed(run)
        side2 = torch.cuda.Stream()
        side2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side2):
            run()
        torch.cuda.current_stream().wait_stream(side2)
        graph2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph2):
            run()
        plain_graph_ms = timed(graph2.replay)
        # the weights' first loads issued before each kernel's wait for the one before
        # (valid here: no kernel of the layer writes a weight)
        g.set_launch_overlap("weights")
        side3 = torch.cuda.Stream()
        side3.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side3):
            run()
        torch.cuda.current_stream().wait_stream(side3)
        graph3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph3):
            run()
        weights_graph_ms = timed(graph3.replay)
    finally:
        g.set_launch_overlap("launch")
    return {"layer": "bf16 B=1: " + ", ".join(f"{n} {M}x{K}" for n, M, K in DECODE_LAYER),
            "bytes": layer_bytes, "kernels": launches,
            "eager_us": round(eager_ms * 1e3, 2), "graph_us": round(graph_ms * 1e3, 2),
            "isolated_sum_us": round(iso_ms * 1e3, 2),
            "eager_gbs": round(layer_bytes / (eager_ms * 1e-3) / 1e9, 1),
            "graph_gbs": round(layer_bytes / (graph_ms * 1e-3) / 1e9, 1),
            "graph_frac_of_peak": round(layer_bytes / (graph_ms * 1e-3) / 1e9 / peak, 4),
            "launch_overlap": "programmatic dependent launch (the library's default)",
            "plain_launches": {"eager_us": round(plain_eager_ms * 1e3, 2), "graph_us": round(plain_graph_ms * 1e3, 2)},
            "weights_prefetch": {"graph_us": round(weights_graph_ms * 1e3, 2),
                                 "graph_frac_of_peak": round(layer_bytes / (weights_graph_ms * 1e-3) / 1e9 / peak, 4)},
            "fused": dict(fused, graph_frac_of_peak=round(fused["graph_gbs"] / peak, 4))}


def decode_layer_fused(torch, g, dev, items, timed):
    """The same layer with its elementwise steps in the GEMV epilogues: the output
    and down projections add the residual stream h in place (gemv_ex), and gate_up
    stores silu(gate) * up (gemv_swiglu, I = 14336), which the down projection then
    reads as its x.  Unfused, these steps would be three more kernels."""
    (wq, dq, yq), (wo, do, yo), (wg, dg, _), (wd, dd, yd) = items
    I = wg.M // 2
    h_o = torch.zeros((1, wo.M), dtype=torch.bfloat16, device=dev)
    h_d = torch.zeros((1, wd.M), dtype=torch.bfloat16, device=dev)
    act = torch.empty((1, I), dtype=torch.bfloat16, device=dev)

    def run():
        g.gemv_bf16(dq["A"], dq["x"], None, yq, wq.M, wq.K, 1)
        g.gemv_ex("bf16", do["A"], None, do["x"], None, h_o, h_o, wo.M, wo.K, 1)
        g.gemv_swiglu("bf16", dg["A"], None, dg["x"], None, act, I, wg.K, 1)
        g.gemv_ex("bf16", dd["A"], None, act, None, h_d, h_d, wd.M, wd.K, 1)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    n0 = g.launch_count()
    with torch.cuda.graph(graph):
        run()
    launches = g.launch_count() - n0
    ms = timed(graph.replay)
    # Q_min of the fused layer: the weights, each x once, each y once, residuals read
    nbytes = (wq.qmin_bytes + wo.qmin_bytes + 2 * wo.M + wg.M * wg.K * 2 + wg.K * 2 + I * 2
              + wd.qmin_bytes + 2 * wd.M)
    return {"epilogues": "o, down: + residual in place; gate_up: silu(gate) * up",
            "bytes": nbytes, "kernels": launches, "graph_us": round(ms * 1e3, 2),
            "graph_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def headline_config(world: int) -> dict:
    """The `config` object of both arms' lines (the same workload, the same keys)."""
    w = W.BY_NAME[W.HEADLINE[0]]
    return {"workload": HEADLINE_DESC, "M": w.M, "K": w.K, "B": w.B, "bias": w.bias, "dtype": w.dtype,
            "l2": "flushed before every GEMV (write then read of a 2x L2 buffer)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def oracle_rate(ws, inputs, nthreads, budget_s, max_reps=50, rows=None):
    """GB/s (over Q_min) of the oracle on the workloads, on the first `rows` rows of
    each (all rows if None), repeated until `budget_s` seconds have passed."""
    import oracle

    bits = []
    for w, i in zip(ws, inputs):
        r = w.M if rows is None else min(rows, w.M)
        bias = None if i["bias"] is None else i["bias"][:r]
        scale = None if i["scale"] is None else i["scale"][:r]
        bits.append((w, r, W.storage_bits(i["A"][:r]), W.storage_bits(i["x"]), W.storage_bits(bias),
                     None if scale is None else scale.numpy()))
    reps = 0
    t0 = time.perf_counter()
    while True:
        for (w, r, A, x, b, sc) in bits:
            oracle.gemv(w.dtype, A, x, b, scale=sc, nthreads=nthreads)
        reps += 1
        if time.perf_counter() - t0 >= budget_s or reps >= max_reps:
            break
    dt = (time.perf_counter() - t0) / reps
    nbytes = sum(W.qmin_bytes(w.dtype, r, w.K, w.B) for (w, r, *_rest) in bits)
    return nbytes / dt / 1e9, dt, reps, [r for (_, r, *_rest) in bits]


def cpu_baseline(head, host_inputs, budget_s=10.0):
    """The oracle (as it stands) on the same GEMV: on all host cores (OpenMP over
    rows) over the whole matrix, and on one core over its first rows (a bounded
    sample of the same matrix, about one second per repetition)."""
    cores = host_cores()
    gbs, dt, reps, _ = oracle_rate(head, host_inputs, cores, budget_s)
    # one core: size the row sample from a short probe
    w = head[0]
    probe_rows = min(w.M, 2048)
    g1, d1, _, _ = oracle_rate(head, host_inputs, 1, 0.0, max_reps=1, rows=probe_rows)
    rows = int(max(256, min(w.M, probe_rows * 1.0 / max(d1, 1e-6))))
    g1, d1, reps1, _ = oracle_rate(head, host_inputs, 1, budget_s, rows=rows)
    return {"value": round(gbs, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the full GEMV ({HEADLINE_DESC}), {reps} repetitions, fp64 C, OpenMP over rows",
            "ms_per_step": round(dt * 1e3, 3),
            "single_thread": {"value": round(g1, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                              "sample": f"the first {rows} of the {w.M} rows of the same matrix, {reps1} "
                                        f"repetitions, fp64 C, one thread",
                              "ms_per_repetition": round(d1 * 1e3, 3)}}


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    """The CPU oracle timed on the host cores, on a bounded sample of the step."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    cores = host_cores()
    head = [W.BY_NAME[n] for n in W.HEADLINE]
    full = [W.make_inputs(w) for w in head]
    # a sample: the first `rows` rows of the GEMV (same K, same values), sized so
    # that the whole run ends within about 1.5 minutes
    rows = 4096
    _, one, _, _ = oracle_rate(head, full, cores, 0.0, max_reps=1, rows=rows)
    budget = 90.0 / max(1, args.steps + args.warmup)
    if one > 0:
        rows = int(max(256, min(head[0].M, rows * budget / one)))
    if args.warmup > 0:
        oracle_rate(head, full, cores, 0.0, max_reps=args.warmup, rows=rows)
    value, dt, _, _ = oracle_rate(head, full, cores, float("inf"), max_reps=max(1, args.steps), rows=rows)
    desc = (f"the first {rows} of the {head[0].M} rows of the step's GEMV ({HEADLINE_DESC}), "
            f"fp64 C, OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded PCG64: A ~ N(0, 0.02^2), x ~ N(0, 1), rounded to bf16)",
        "config": headline_config(world),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
