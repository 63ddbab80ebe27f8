#!/usr/bin/env python
"""Throughput benchmark of batched quintic Newton-Schulz on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

A step is one pass of the whole hot path -- norm and 5 x {gram, square,
apply} -- over one batch of the workload (default: 8 bf16 8192 x 6144
matrices, N(0, 0.02), one library call). Inputs are resident in HBM when the
timed region starts and are restored from a pristine copy between steps,
outside the timed events; the batch (768 MiB) is larger than L2, so no
separate flush is needed. Each step is timed with one CUDA-event pair on the
launching stream; `value` is matrices / second over the K timed steps (max
over ranks of the time). The per-kernel breakdown and the roofline figure
come from a second pass of the same K steps with an event pair around every
launch, so the events never sit inside the timed region of `value`. On one
GPU the other workloads follow, each timed alone (`configs`).

Multi-GPU (torchrun, one process per GPU): matrices are independent. By
default one batch is split: every rank runs the matrices the library's host
planner assigns it (largest ns_cost first onto the least-loaded rank) and
`value` is the batch over the slowest rank's time (strong scaling);
`--parallel replicas` gives every rank a whole batch (weak scaling). Either
way no collective touches the data path; only the timing barrier and the
max-reduction of times use the process group.

`--impl reference` times the CPU fp64 oracle on the host cores instead: each
step is one Newton-Schulz step of one matrix of the workload (a bounded
sample), scaled to matrices / second.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


# ------------------------------------------------------------------ helpers

def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--gemm-schedule", choices=["phase", "single"], default="phase",
                   help="tensor-core launches: one per step and phase, or one per call")
    p.add_argument("--matrices", type=int, default=0,
                   help="use only the first K matrices of the workload (profiling captures)")
    p.add_argument("--parallel", choices=["split", "replicas"], default="split",
                   help="N > 1: split one batch over the GPUs by ns_cost, or run a whole batch per GPU")
    p.add_argument("--configs", type=int, default=1,
                   help="1: after the headline, time every other workload on this GPU (N = 1 only)")
    p.add_argument("--config-steps", type=int, default=5)
    return p.parse_args()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    elif torch.cuda.is_available() and args.impl == "ours":
        torch.cuda.set_device(local)
    return world, rank, local, pg


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
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
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def physical_gpu_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        items = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(items) and items[local].isdigit():
            return int(items[local])
    return local


def workload_flops(shapes, steps):
    nominal = executed = apply = 0
    for M, N in shapes:
        m, n = min(M, N), max(M, N)
        nominal += steps * (4 * m * m * n + 2 * m ** 3)
        executed += steps * (3 * m * m * n + m ** 3)
        apply += steps * (2 * m * m * n)
    return nominal, executed, apply


def input_digest(mats):
    """SHA-256 over the inputs' bytes, matrix after matrix (bf16 as its 16-bit
    patterns), so that a run names exactly the data it measured."""
    import torch
    h = hashlib.sha256()
    for t in mats:
        v = t.detach().cpu().contiguous()
        if v.dtype == torch.bfloat16:
            v = v.view(torch.int16)
        h.update(v.numpy().tobytes())
    return h.hexdigest()


def norm_pass_record(ktimes, bytes_per_step, steps, hbm_peak):
    """Achieved HBM bandwidth of the pass over the caller's matrices (the
    Frobenius sums and extents; it reads every input byte once per call) from
    its CUDA-event times, or None when the workload never launched it."""
    ms, launches = ktimes.get("norm_pass", (0.0, 0))
    if not launches or ms <= 0:
        return None
    gbs = bytes_per_step * steps / (ms / 1e3) / 1e9
    return {"kernel": "ns_norm_tiles_kernel (Frobenius sums and extents)", "bound": "hbm",
            "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(gbs / hbm_peak, 4) if hbm_peak else None,
            "bytes_per_step": int(bytes_per_step), "launches": int(launches), "ms_total": round(ms, 4)}


def traffic_record(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` on `workload` from the committed ncu
    summary, if it was captured from the current kernel source (sha256 prefix
    matches) for this workload."""
    src = os.path.join(ROOT, "newton_schulz_quintic_gb300", "csrc", "ns_tc.cu")
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(src, "rb") as fh:
            sha = hashlib.sha256(fh.read()).hexdigest()[:16]
        with open(path) as fh:
            lines = fh.readlines()
    except Exception:
        return None
    for line in lines:
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") == kernel and f.get("source_sha") == sha and f.get("workload") == workload:
            return f
    return None


# ------------------------------------------------------------------ our arm

def rank_share(wl, world: int, rank: int) -> list:
    """Indices of the workload's matrices that `rank` orthogonalizes when one
    batch is split over `world` GPUs: whole matrices, largest ns_cost first onto
    the least-loaded rank, with the 0.3 per-call numel cap (the second page's
    "Changes" items 1-3, through the library's host planner). Every rank
    computes the same plan, so no rank sends another anything."""
    from newton_schulz_quintic_gb300 import api
    if world <= 1:
        return list(range(wl.count))
    assign, _ = api.plan_shards(wl.shapes, world, numel_eps=0.3)
    return [i for i, r in enumerate(assign) if r == rank]


def rank_calls(wl, mine: list, split: bool) -> list:
    """The library calls a rank makes per step, as lists of matrix indices: the
    workload's own calls (e.g. remainder batches 64 + 12) for a replica, one
    call over the rank's share when the batch is split."""
    if not split:
        return [list(range(sl.start, sl.stop)) for sl in wl.call_slices()]
    return [mine] if mine else []


def time_steps(steps, restore, one_step, stream):
    """CUDA-event time of each of `steps` steps (ms); inputs restored before
    each step, outside its events."""
    import torch
    ev = []
    for _ in range(steps):
        restore()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        one_step()
        e.record(stream)
        ev.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def small_f32(wl) -> bool:
    """Whether every matrix of an fp32 workload takes the shared-memory
    resident path (m <= 64), not the tensor cores."""
    return all(min(M, N) <= 64 for M, N in wl.shapes)


def measure_workload(wl, dev, steps, warmup, graph=False):
    """Matrices/s of one workload on this GPU alone (the per-config record):
    direct library calls, and optionally the same calls replayed from a CUDA
    graph (the library's repeat calls allocate and upload nothing, so they
    can be captured) to show the device time without host launch work."""
    import torch
    from newton_schulz_quintic_gb300 import api
    host = wl.matrices()
    pristine = [h.to(dev) for h in host]
    work = [torch.empty_like(p) for p in pristine]
    slices = wl.call_slices()
    stream = torch.cuda.current_stream(dev)

    def restore():
        for w, p in zip(work, pristine):
            w.copy_(p, non_blocking=True)

    def one_step():
        for sl in slices:
            api.orthogonalize_batched(work[sl], steps=wl.steps)

    for _ in range(max(warmup, 1)):
        restore()
        one_step()
    torch.cuda.synchronize()
    times = time_steps(steps, restore, one_step, stream)
    if api.get_status() != 0:
        raise RuntimeError(f"device status word reports a timeout on {wl.name}")
    # the same calls with their arguments marshalled once (api.PreparedBatch)
    prepared = [api.PreparedBatch(work[sl], steps=wl.steps) for sl in slices]

    def one_step_prepared():
        for pb in prepared:
            pb()

    ptimes = time_steps(steps, restore, one_step_prepared, stream)
    # host time of a call (argument marshalling, planning, launches), measured
    # back to back without waiting for the GPU
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(10):
        one_step()
    host_us = (time.perf_counter() - t0) / 10 * 1e6
    torch.cuda.synchronize()
    # per-kernel times: the same steps with an event pair around every launch
    api.set_kernel_timing(True)
    time_steps(steps, restore, one_step, stream)
    kt = api.kernel_times()
    api.set_kernel_timing(False)
    kbytes = sum(M * N for M, N in wl.shapes) * (2 if wl.dtype == "bf16" else 4)
    nominal, executed, _ = workload_flops(wl.shapes, wl.steps)
    peaks, _ = measured_peaks()
    mean = statistics.mean(times)
    rec = {"matrices": wl.count, "calls": [s.stop - s.start for s in slices], "steps": steps,
           "ms_per_step": round(mean, 4), "ms_per_step_median": round(statistics.median(times), 4),
           "value": round(wl.count / (mean / 1e3), 3), "unit": "matrices/s",
           "tflops_executed": round(executed / (mean / 1e3) / 1e12, 2),
           "tflops_nominal": round(nominal / (mean / 1e3) / 1e12, 2)}
    rec["executed_frac"] = {"burst": round(rec["tflops_executed"] / peaks["bf16_tflops"], 4),
                            "sustained": round(rec["tflops_executed"] / peaks["bf16_tflops_sustained"], 4)}
    if wl.dtype == "f32" and not small_f32(wl):
        # large fp32 matrices run on the bf16 tensor cores as six slice products
        # per GEMM: their bf16 tensor work is six times the fp32 flops
        bf16_work = 6 * rec["tflops_executed"]
        rec["executed_frac"] = {"note": "fp32 flops; the bf16 tensor work is 6x (three bf16 slices per tensor, "
                                        "six slice products per GEMM)",
                                "bf16_tensor_tflops": round(bf16_work, 2),
                                "bf16_tensor_burst": round(bf16_work / peaks["bf16_tflops"], 4),
                                "bf16_tensor_sustained": round(bf16_work / peaks["bf16_tflops_sustained"], 4)}
    rec["ms_per_step_prepared"] = round(statistics.mean(ptimes), 4)
    rec["ms_per_step_prepared_median"] = round(statistics.median(ptimes), 4)
    rec["host_us_per_call"] = round(host_us, 1)
    rec["kernels"] = {k: {"ms_per_step": round(v[0] / steps, 4), "launches_per_step": round(v[1] / steps, 2)}
                      for k, v in kt.items() if v[1]}
    rec["norm_pass"] = norm_pass_record(kt, kbytes, steps, peaks.get("hbm_gbs"))
    if graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            one_step()                      # warm the per-stream workspace of the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cap):
                one_step()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        for _ in range(2):
            restore()
            g.replay()
        torch.cuda.synchronize()
        gt = time_steps(steps, restore, g.replay, stream)
        rec["ms_per_step_graph"] = round(statistics.mean(gt), 4)
        rec["ms_per_step_graph_median"] = round(statistics.median(gt), 4)
        rec["value_graph"] = round(wl.count / (statistics.mean(gt) / 1e3), 3)
    del work, pristine
    torch.cuda.synchronize()
    return rec


def run_ours(args, world, rank, local, pg):
    import torch
    from newton_schulz_quintic_gb300 import api, inputs

    api.load_library()
    api.set_gemm_schedule(args.gemm_schedule)
    wl = inputs.WORKLOADS[args.workload or inputs.HEADLINE]
    if args.matrices:
        wl = inputs.subset(wl, args.matrices)
    split = args.parallel == "split" and world > 1
    dev = torch.device("cuda", local)
    mine = rank_share(wl, world, rank) if split else list(range(wl.count))
    calls = rank_calls(wl, mine, split)
    host = {i: wl.matrix(i) for i in mine}
    digest = input_digest([wl.matrix(i) for i in range(wl.count)]) if rank == 0 else None
    pristine = {i: h.to(dev) for i, h in host.items()}
    work = {i: torch.empty_like(p) for i, p in pristine.items()}
    call_mats = [[work[i] for i in c] for c in calls]
    stream = torch.cuda.current_stream(dev)

    def restore():
        for i, w in work.items():
            w.copy_(pristine[i], non_blocking=True)

    def one_step():
        for mats in call_mats:
            api.orthogonalize_batched(mats, steps=wl.steps)

    for _ in range(max(args.warmup, 0)):
        restore()
        one_step()
    torch.cuda.synchronize()
    if api.get_status() != 0:
        raise RuntimeError("device status word reports a timeout during warm-up")

    # timed region: K steps, one CUDA-event pair per step and no other event
    clocks = ClockSampler(physical_gpu_index(local))
    if rank == 0:
        clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    launches0 = api.num_kernel_launches()
    times = time_steps(args.steps, restore, one_step, stream)
    launches = api.num_kernel_launches() - launches0
    if pg:
        pg.barrier()
    clock_rec = clocks.stop() if rank == 0 else None
    if api.get_status() != 0:
        raise RuntimeError("device status word reports a timeout during the timed steps")
    total_ms = sum(times)
    if pg:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total_ms = float(t.item())

    # kernel breakdown: the same K steps again with a CUDA-event pair around
    # every launch of the library (on the stream it launches on)
    api.set_kernel_timing(True)
    itimes = time_steps(args.steps, restore, one_step, stream)
    ktimes = api.kernel_times()
    api.set_kernel_timing(False)

    # end to end through the host entry point: pinned host inputs, H2D copy,
    # compute, D2H copy of the result, all inside the timed region
    e2e_bytes = sum(h.numel() * h.element_size() for h in host.values())
    e2e_s = float("nan")
    if args.e2e_steps > 0:
        pinned = {i: h.clone().pin_memory() for i, h in host.items()}
        pcalls = [[pinned[i] for i in c] for c in calls]
        for mats in pcalls:  # warm the host entry point's staging buffers
            api.orthogonalize_batched_host(mats, steps=wl.steps, device=dev)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            for mats in pcalls:
                api.orthogonalize_batched_host(mats, steps=wl.steps, device=dev)
        e2e_s = time.perf_counter() - t0
    if pg:
        t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_total_bytes = e2e_bytes
    if pg:
        t = torch.tensor([float(e2e_bytes)], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.SUM)
        e2e_total_bytes = int(t.item())

    # the other workloads, each on this GPU alone, after the headline
    configs = None
    if world == 1 and args.configs and not args.matrices:
        del work, pristine, call_mats
        api.release_workspace()
        torch.cuda.empty_cache()
        configs = {}
        for name in inputs.WORKLOADS:
            if name == wl.name:
                continue
            other = inputs.WORKLOADS[name]
            small = sum(M * N for M, N in other.shapes) <= (1 << 22)
            k = args.config_steps if not small else max(args.config_steps, 20)
            # the small workloads and the remainder pair (64 + 12) are also replayed from one graph
            configs[name] = measure_workload(other, dev, k, 3, graph=small or len(other.call_slices()) > 1)
            api.release_workspace()
            torch.cuda.empty_cache()

    if rank != 0:
        return None

    count = wl.count
    ms_per_step = total_ms / args.steps
    matrices_per_rank = [len(mine)] if not split else None
    ws_bytes = max((api.workspace_bytes([tuple(wl.shapes[i]) for i in c], host[c[0]].dtype) for c in calls if c),
                   default=0)
    total_mats = count if split else world * count
    value = total_mats * args.steps / (total_ms / 1e3)
    nominal, executed, apply_flops = workload_flops(wl.shapes, wl.steps)
    if not split:
        nominal, executed = world * nominal, world * executed
    peaks, peak_kind = measured_peaks()
    # dominant kernel: the tensor-core GEMM. Run as one launch per call it does
    # every phase (executed flops: m^2 n gram + m^3 square + 2 m^2 n apply per
    # matrix per step); run per phase, the apply launches (2 m^2 n) are reported.
    _, my_executed, my_apply = workload_flops([wl.shapes[i] for i in mine], wl.steps)
    gms, glaunch = ktimes["gemm"]
    if glaunch:
        kname, kms, klaunch, kflops = "ns_tc_gemm_kernel (all steps and phases of a call)", gms, glaunch, my_executed
    else:
        kname, kms, klaunch, kflops = "ns_tc_gemm_kernel (apply: W' = aW + BW)", *ktimes["apply"], my_apply
    flops_per_launch = kflops * args.steps / max(klaunch, 1)
    achieved = flops_per_launch / (kms / max(klaunch, 1) / 1e3) / 1e12 if klaunch else None
    peak = peaks.get("bf16_tflops_sustained", 1700.0)
    peak_burst = peaks.get("bf16_tflops", 1900.0)
    tr = traffic_record("gemm" if glaunch else "apply", wl.name) if not split else None
    gemm_ms = sum(ktimes[k][0] for k in ("gram", "square", "apply", "gemm"))
    tflops_exec = executed * args.steps / (total_ms / 1e3) / 1e12
    ktotal = max(sum(x[0] for x in ktimes.values()), 1e-9)
    out = {
        "metric": "NS-orthogonalized matrices/s (bf16 tensor-core TFLOP/s and fraction of peak alongside)",
        "value": round(value, 3),
        "unit": "matrices/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "ms_per_step_median": round(statistics.median(times), 4),
        "higher_is_better": True,
        "scaling": "strong" if split else "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,0.02) bf16, per-matrix torch.Generator seeds)",
        "config": {"workload": wl.name, "matrices": count,
                   "shapes": [list(t) for t in sorted({tuple(x) for x in wl.shapes})],
                   "ns_steps": wl.steps, "coeffs": [3.4445, -4.775, 2.0315],
                   "calls": [len(c) for c in calls],
                   "l2": "inputs (%.0f MiB) larger than L2; restored from a pristine copy between steps"
                         % (sum(h.numel() * h.element_size() for h in host.values()) / 2 ** 20),
                   "parallelism": (f"split x{world}: whole matrices by ns_cost, largest first onto the "
                                   "least-loaded GPU; no collective" if split else
                                   f"replicas x{world} (every GPU its own batch, no collective)")},
        "tflops_executed": round(tflops_exec, 2),
        "executed_frac": {"burst": round(tflops_exec / peak_burst, 4),
                          "sustained": round(tflops_exec / peak, 4),
                          "note": "executed = 3 m^2 n + m^3 per matrix and step (upper tiles of the symmetric "
                                  "products), over the whole step including the norm pass"},
        "tflops_nominal_equivalent": round(nominal * args.steps / (total_ms / 1e3) / 1e12, 2),
        "roofline": {
            "kernel": kname,
            "bound": "tensor",
            "achieved": round(achieved, 2) if achieved else None,
            "peak": peak,
            "peak_source": f"{peak_kind} bf16_tflops_sustained (kernel timed inside a long step)",
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4) if achieved else None,
            "peak_burst": peak_burst,
            "frac_of_burst": round(achieved / peak_burst, 4) if achieved else None,
            "traffic": (int(float(tr["bytes_per_launch"])) if tr else None),
            "algorithmic_flops_per_launch": flops_per_launch,
            "timed_in": "a second pass of the same steps with a CUDA-event pair around every launch",
        },
        "norm_pass": norm_pass_record(ktimes, e2e_bytes, args.steps, peaks.get("hbm_gbs")),
        "workspace_bytes": int(ws_bytes),
        "input_sha256": digest,
        "ms_per_step_instrumented": round(statistics.mean(itimes), 4),
        "kernels": {k: {"ms_total": round(v[0], 3), "launches": v[1], "share": round(v[0] / ktotal, 4)}
                    for k, v in ktimes.items() if v[1]},
        "gemm_tflops_executed": (round(my_executed * args.steps / (gemm_ms / 1e3) / 1e12, 2)
                                 if gemm_ms else None),
        "gpu_launches": int(launches),
        "e2e": {"value": (round(total_mats * args.e2e_steps / e2e_s, 3) if args.e2e_steps > 0 else None),
                "unit": "matrices/s",
                "h2d_bytes_per_step": e2e_total_bytes, "d2h_bytes_per_step": e2e_total_bytes,
                "api": "ns_orthogonalize_batched_host (pinned host buffers)"},
        "clocks": clock_rec,
    }
    if matrices_per_rank is None:
        out["config"]["matrices_rank0"] = len(mine)
    if configs is not None:
        out["configs"] = configs
    return out, wl


# ------------------------------------------------------------------ CPU oracle

def cpu_oracle_sample(wl, matrix_index=0):
    """One Newton-Schulz step of one matrix of the workload with the oracle's
    NumPy implementation; returns (seconds, description)."""
    import numpy as np  # noqa: F401
    import oracle
    x = oracle.to_f64(wl.matrix(matrix_index))
    t0 = time.perf_counter()
    oracle.orthogonalize_np(x, steps=1)
    dt = time.perf_counter() - t0
    M, N = wl.shapes[matrix_index]
    return dt, f"1 of {wl.steps} Newton-Schulz steps on 1 of {wl.count} matrices ({M}x{N}), " \
               f"oracle.orthogonalize_np fp64, scaled to matrices/s as 1/({wl.steps} x step time)"


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def host_cpu():
    """Architecture and model of the host CPU, as /proc/cpuinfo names it (Arm
    cores give only their part number there)."""
    import platform
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key = key.strip().lower()
                if key == "model name":
                    name = val.strip()
                    break
                if key == "cpu part" and not name:
                    name = "cpu part " + val.strip()
    except OSError:
        pass
    return f"{platform.machine()} {name}".strip()


def blas_threads():
    """Threads NumPy's OpenBLAS runs with: its thread variables as read when
    NumPy loaded (OPENBLAS_NUM_THREADS before OMP_NUM_THREADS), else every
    core this process may run on."""
    n = cores()
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        try:
            return max(1, min(n, int(os.environ[var])))
        except (KeyError, ValueError):
            continue
    return n


def run_reference(args, world, rank):
    from newton_schulz_quintic_gb300 import inputs
    if rank != 0:
        return None
    wl = inputs.WORKLOADS[args.workload or inputs.HEADLINE]
    for _ in range(max(args.warmup, 0)):
        cpu_oracle_sample(wl)
    times = []
    desc = ""
    for _ in range(args.steps):
        dt, desc = cpu_oracle_sample(wl)
        times.append(dt)
    per_matrix = wl.steps * statistics.mean(times)
    value = 1.0 / per_matrix
    out = {
        "impl": "reference",
        "metric": "NS-orthogonalized matrices/s (bf16 tensor-core TFLOP/s and fraction of peak alongside)",
        "value": round(value, 6),
        "unit": "matrices/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(times) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) bf16 inputs widened exactly to fp64)",
        "config": {"workload": wl.name, "matrices": wl.count,
                   "shapes": [list(t) for t in sorted({tuple(x) for x in wl.shapes})], "ns_steps": wl.steps},
        "cpu_baseline": {"value": round(value, 6), "unit": "matrices/s", "cores": blas_threads(), "kind": "oracle",
                         "cpu": host_cpu(), "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "matrices/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return out


def main():
    args = parse_args()
    if args.impl == "reference" and os.environ.get("RANK", "0") == "0":
        # rank 0 alone times the oracle and the other ranks do no work, so it
        # takes every host core: torchrun's default of one OpenMP thread per
        # rank would otherwise hold NumPy's BLAS to one thread. Set before
        # NumPy is first imported.
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
            os.environ[var] = str(cores())
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return
    res = run_ours(args, world, rank, local, pg)
    if res is not None:
        out, wl = res
        if world == 1 and not args.no_cpu_baseline:
            dt, desc = cpu_oracle_sample(wl)
            v = 1.0 / (wl.steps * dt)
            out["cpu_baseline"] = {"value": round(v, 6), "unit": "matrices/s", "cores": blas_threads(),
                                   "kind": "oracle", "cpu": host_cpu(), "sample": desc}
        print(json.dumps(out), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
