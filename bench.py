"""Benchmark of the Muon optimizer step on one B300 (or N replicas under torchrun).

Workload: the d26 stack -- 26 layers of width 1664, per layer four 1664 x 1664
attention matrices, the 6656 x 1664 MLP input and the 1664 x 6656 MLP output
(156 fp32 matrices, 8.64e8 elements) -- one Muon step per timed step: Nesterov
momentum (beta 0.95), Frobenius normalisation, 5 quintic Newton-Schulz
iterations, aspect-scaled update (lr 0.02).  Consecutive steps carry the
momentum and weights, and every step reads a gradient set of its own, drawn on
the device before the timed region (3.46 GB each, far above the 126 MB L2, so
no flush is needed between steps; past 32 steps the sets are reused in turn).

Metric: algorithmic Newton-Schulz TFLOP/s of the whole step (3 m^2 n + m^3 per
matrix and iteration, m <= n the oriented sides) = flops / step time; the line
also carries ms per step, the NS kernels' own TFLOP/s and their fraction of the
measured bf16 peak.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon optimizer step ms and NS TFLOP/s at d26 shapes; fraction of bf16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "d26"
WORKLOAD_DESC = ("d26 stack: 156 fp32 matrices (26 layers x [4 x 1664x1664, 6656x1664, 1664x6656]), "
                 "Nesterov beta 0.95, lr 0.02, 5 Newton-Schulz iterations, momentum carried across steps")


def workload_desc(name):
    if name == WORKLOAD:
        return WORKLOAD_DESC
    import workloads
    shapes = workloads.config_shapes(name)
    kinds = sorted(set(shapes))
    return (f"{name}: {len(shapes)} fp32 matrices of shapes {kinds}, Nesterov beta 0.95, lr 0.02, "
            "5 Newton-Schulz iterations")


MAX_GRAD_SETS = 32  # past this many steps the pre-drawn gradient sets are reused in turn

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples SM clocks, power and clock-event reasons during a timed region.

    Uses `nvidia-smi --query-gpu=... -lms 50` in a child process (the sampler
    is started before the region and stopped after it); if nvidia-smi is not on
    PATH, NVML through pynvml every 100 ms instead."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    NVML_REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
                    "sw_power_cap": 0x4}

    def __init__(self, index: int):
        self.index = index
        self.samples, self.power, self.reasons, self.max_mhz = [], [], set(), None
        self.source = None
        self._proc = None
        self._nvml = None
        self._stop = threading.Event()

    # -- nvidia-smi
    def _start_smi(self):
        import shutil
        import subprocess
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return False
        self._proc = subprocess.Popen(
            [exe, "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
             "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        # wait (up to 5 s) for the sampler's first line, so that it is live when
        # the timed region starts; that line was taken before the region and is dropped
        import select
        ready, _, _ = select.select([self._proc.stdout], [], [], 5.0)
        if ready:
            self._proc.stdout.readline()
        self.source = "nvidia-smi -lms 50"
        return True

    def _parse_smi(self, text):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in text.splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                self.samples.append(float(parts[1]))
                self.max_mhz = float(parts[2])
                self.power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:]):
                if val.lower() == "active":
                    self.reasons.add(name)

    # -- NVML fallback
    def _start_nvml(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nvml = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
        except Exception:
            self._nvml = None
            return False
        self.source = "nvml 100 ms"
        self._t = threading.Thread(target=self._run_nvml, daemon=True)
        self._t.start()
        return True

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self._nvml.nvmlDeviceGetClockInfo(self._h, self._nvml.NVML_CLOCK_SM))
                mask = self._nvml.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                for name, bit in self.NVML_REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            self._stop.wait(0.1)

    def __enter__(self):
        if not self._start_smi():
            self._start_nvml()
        return self

    def __exit__(self, *exc):
        if self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except Exception:
                self._proc.kill()
                out, _ = self._proc.communicate()
            self._parse_smi(out or "")
        if self._nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source (nvidia-smi, nvml)"]}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons), "samples": len(self.samples),
                "power_w_max": max(self.power) if self.power else None, "source": self.source}


# DRAM bytes (read + write) per Newton-Schulz launch at d26, from one ncu capture of the
# d26x2 workload (the same shapes, 2 of the 26 layers): one axpy, Gram, polynomial and final
# launch, averaged with a step's launch counts (4, 5, 5, 1) and scaled by 13; and the sha256
# of the kernel source it was taken on.  The figure is reported only while the source is
# unchanged.
NS_PAIR_TRAFFIC = {"bytes_per_launch_d26": 2.3976e+09, "source_sha256": "9bc9f998578c64f0359f7586645567a47a2d72908b5de976f3f677ba45f6d73f"}


def ns_pair_traffic():
    """DRAM bytes per NS launch at d26, or None when the kernel changed since the capture."""
    import hashlib
    src = os.path.join(ROOT, "pretraining_optimizer_step_b300", "csrc", "ns_pair.cu")
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    if NS_PAIR_TRAFFIC["source_sha256"] != digest:
        return None
    return NS_PAIR_TRAFFIC["bytes_per_launch_d26"]


def cpu_model() -> str:
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


# ---------------------------------------------------------------- multi-rank host logic
def max_over_ranks(ms: float, dist=None, device="cpu") -> float:
    """The slowest rank's time: every rank times its own replica, the job's time is the max."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs one step of its own stack in ms_per_step (the max
    over ranks), so the job does world x flops_per_rank_step in that time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------- CPU oracle leg
def default_sample(workload):
    """Matrices of the oracle's timed sample: for the stacks a square attention matrix and the
    4:1 MLP input (for d26: 0 is 1664 x 1664, 4 is 6656 x 1664), else the first matrix."""
    return (0, 4) if workload in ("d12", "d20", "d26") else (0,)


def oracle_sample(idx=(0, 4), workload=WORKLOAD, ns_steps=5):
    """Time the fp64 oracle on a bounded sample of the workload: one Muon step (ns_steps
    iterations) of the listed matrices.  Returns (TFLOP/s of algorithmic NS flops, seconds,
    description, threads, flops)."""
    import numpy as np
    import oracle
    import workloads
    oracle.build()
    idx = list(idx)
    p, g, m, shapes = workloads.make_stack(workload, "cpu", indices=idx)
    flops = 0.0
    t0 = time.perf_counter()
    for pi, gi, mi, (r, c) in zip(p, g, m, shapes):
        oracle.muon_matrix(pi.numpy(), gi.numpy(), mi.numpy(), lr=np.float32(0.02), beta=np.float32(0.95),
                           nesterov=True, ns_steps=ns_steps)
        mm, nn = min(r, c), max(r, c)
        flops += ns_steps * (3 * mm * mm * nn + mm ** 3)
    dt = time.perf_counter() - t0
    step = "full Muon step" if ns_steps == 5 else f"Muon step with {ns_steps} Newton-Schulz iteration(s)"
    desc = (f"oracle (fp64 C, OpenMP) {step} of {workload} matrices "
            + ", ".join(f"{i} ({r}x{c})" for i, (r, c) in zip(idx, shapes))
            + f"; {flops:.3e} algorithmic NS flops")
    return flops / dt / 1e12, dt, desc, oracle.num_threads(), flops


def oracle_single_core(workload):
    """The oracle on one host thread, on a smaller bounded sample (matrix 0, one iteration)."""
    import oracle
    oracle.build()
    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        tf, dt, desc, cores, _ = oracle_sample((0,), workload, ns_steps=1)
    finally:
        oracle.set_num_threads(n)
    return {"value": tf, "unit": UNIT, "cores": cores, "sample": f"{desc}; {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    # the same matrices as the GPU line's cpu_baseline leg; the untimed warm-up steps run the
    # first of them only, which keeps --steps 20 --warmup 5 within about four minutes
    sample = default_sample(args.workload)
    for _ in range(args.warmup):
        oracle_sample(sample[:1], args.workload)
    times, flops_total = [], 0.0
    for _ in range(args.steps):
        tf, dt, desc, cores, flops = oracle_sample(sample, args.workload)
        times.append(dt)
        flops_total += flops
    value = flops_total / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(args.workload), "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg
def run_ours(args, rank, world, local_rank):
    import torch
    import pretraining_optimizer_step_b300 as mu
    import workloads

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()

    # CPU oracle timed first (rank 0, N = 1 only), before any GPU work
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, desc, cores, _ = oracle_sample(default_sample(args.workload), args.workload)
        cpu = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{desc}; {dt:.1f} s", "cpu_model": cpu_model(),
               "single_core": oracle_single_core(args.workload)}

    wl = args.workload
    shapes = workloads.config_shapes(wl)
    seed = rank  # each replica works on its own stack
    p, g0, m, _ = workloads.make_stack(wl, dev, seed=seed)
    # a gradient draw of its own for every step (warm-up and timed), all drawn before timing
    n_sets = max(1, min(args.warmup + args.steps, MAX_GRAD_SETS))
    grads = [g0] + [[workloads.make_grad(wl, i, s, dev, seed, step) for i, s in enumerate(shapes)]
                    for step in range(1, n_sets)]
    stream = torch.cuda.Stream(device=dev)
    step_args = [mu.StepArgs(p, grads[k], m, shapes) for k in range(n_sets)]
    hp = workloads.HYPER
    elems = sum(r * c for r, c in shapes)

    def step(k):
        mu.muon_step(step_args[k % n_sets], lr=hp["lr"], beta=hp["beta"], nesterov=hp["nesterov"],
                     ns_steps=hp["ns_steps"], stream=stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    def timed(nsteps, fn, per_step=None):
        """Device time of nsteps calls of fn on the stream, max over ranks.  With a list as
        per_step, an event recorded after every step adds each step's own time to it."""
        barrier()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps + 1 if per_step is not None else 2)]
        evs[0].record(stream)
        for k in range(nsteps):
            fn(k)
            if per_step is not None:
                evs[k + 1].record(stream)
        evs[-1].record(stream)
        evs[-1].synchronize()
        barrier()
        if per_step is not None:
            per_step.extend(evs[k].elapsed_time(evs[k + 1]) for k in range(nsteps))
        return max_over_ranks(evs[0].elapsed_time(evs[-1]), dist, dev)

    # ---- timed region 1: plain steps (the headline value)
    mu.muon_init()
    for k in range(args.warmup):
        step(k)
    mu.muon_get_status(stream)
    step_ms = []
    with ClockSampler(local_rank) as clocks:
        total_ms = timed(args.steps, lambda k: step(args.warmup + k), step_ms)
    mu.muon_get_status(stream)
    # the carried steps one by one (momentum carried, a new gradient set every step)
    step_stats = {k: max_over_ranks(f(step_ms), dist, dev)
                  for k, f in (("median", statistics.median), ("mean", statistics.mean), ("min", min),
                               ("max", max))}
    info = mu.muon_get_step_info()
    ms_step = total_ms / args.steps
    flops_step = info["ns_alg_flops"]
    value = job_tflops(world, flops_step, ms_step)

    # ---- timed region 2: same steps with CUDA events around every launch
    mu.muon_destroy()
    mu.muon_init(debug_flags=mu.MUON_DEBUG_TIME_KERNELS)
    for k in range(args.warmup):
        step(k)
    mu.muon_get_status(stream)
    mu.muon_kernel_times()
    timed_ms2 = timed(args.steps, lambda k: step(args.warmup + k))
    kt = mu.muon_kernel_times()
    mu.muon_get_status(stream)
    ns_kinds = ("gram", "poly", "axpy", "axpy_update")
    ns_ms = sum(kt[k][0] for k in ns_kinds)
    ns_launches = sum(kt[k][1] for k in ns_kinds)
    ns_tflops = flops_step * args.steps / (ns_ms * 1e-3) / 1e12
    mom_ms, mom_launches = kt["momentum_norm"]
    mom_bytes = 14.0 * elems * args.steps
    mom_gbs = mom_bytes / (mom_ms * 1e-3) / 1e9
    q = mu.muon_plan_query(shapes, hp["ns_steps"])
    peak_tf = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_tf_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_bw = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    traffic = ns_pair_traffic() if wl == WORKLOAD else None
    # the NS launches run back to back inside a step loop of about half a second, under the
    # power cap, so their denominator is the measured sustained bf16 rate (burst beside it)
    roofline = {"bound": "tensor", "kernel": "ns_pair_kernel (Gram, polynomial, axpy launches)",
                "achieved": ns_tflops, "peak": peak_tf_sus, "unit": "TFLOP/s", "frac": ns_tflops / peak_tf_sus,
                "peak_source": f"{peak_src} bf16_tflops_sustained",
                "frac_of_burst": ns_tflops / peak_tf, "burst_peak": peak_tf,
                "traffic": traffic,
                "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the d26x2 workload "
                                   "(2 of the 26 layers) x 13; null once the kernel source has changed"),
                "avg_launch_ms": ns_ms / max(ns_launches, 1),
                "alg_flops_per_launch": flops_step * args.steps / max(ns_launches, 1),
                "executed_over_alg_flops": q["ns_executed_flops"] / q["ns_alg_flops"]}
    roofline_hbm = {"bound": "hbm", "kernel": "momentum_norm_kernel", "achieved": mom_gbs, "peak": peak_bw,
                    "unit": "GB/s", "frac": mom_gbs / peak_bw, "peak_source": f"{peak_src} hbm_gbs",
                    "alg_bytes_per_launch": mom_bytes / max(mom_launches, 1),
                    "avg_launch_ms": mom_ms / max(mom_launches, 1)}
    phase_ms = {k: v[0] / args.steps for k, v in kt.items()}

    # ---- the same step with NorMuon scaling (second moments per stored row)
    normuon = None
    if wl in workloads.STACK_DEPTHS:
        mu.muon_destroy()
        mu.muon_init(debug_flags=mu.MUON_DEBUG_TIME_KERNELS)
        V = [torch.zeros(r, device=dev) for r, _ in shapes]

        def nm_step(k):
            mu.muon_step_normuon(step_args[k % n_sets], second_moments=V, lr=hp["lr"], beta=hp["beta"],
                                 nesterov=hp["nesterov"], ns_steps=hp["ns_steps"], stream=stream)

        for k in range(args.warmup):
            nm_step(k)
        mu.muon_get_status(stream)
        mu.muon_kernel_times()
        nm_ms = timed(args.steps, lambda k: nm_step(args.warmup + k)) / args.steps
        nkt = mu.muon_kernel_times()
        mu.muon_get_status(stream)
        normuon = {"ms_per_step": nm_ms, "value": job_tflops(world, flops_step, nm_ms), "unit": UNIT,
                   "overhead_ms_vs_plain_step": nm_ms - ms_step,
                   "phase_ms_per_step": {k: v[0] / args.steps for k, v in nkt.items() if v[1]},
                   "state": "beta2 0.95, eps 1e-10, V per stored row (zero-initialised)"}
        del V

    # ---- AdamW over the same model's non-matrix parameters (embedding, lm_head,
    # scalars): one multi-tensor launch per step, HBM-bound at 28 bytes per element
    adamw = None
    if wl in workloads.STACK_DEPTHS:
        ap, ag, am, av, ashapes = workloads.make_adamw_set(wl, dev, seed=seed)
        a_args = mu.AdamWArgs(ap, ag, am, av)
        a_elems = sum(int(t.numel()) for t in ap)
        a_hp = dict(lr=3e-3, beta1=0.8, beta2=0.95, eps=1e-8, weight_decay=0.01)
        for k in range(args.warmup):
            mu.muon_adamw_step(a_args, step=k + 1, stream=stream, **a_hp)
        a_ms = timed(args.steps, lambda k: mu.muon_adamw_step(a_args, step=args.warmup + k + 1, stream=stream,
                                                              **a_hp)) / args.steps
        a_gbs = 28.0 * a_elems / (a_ms * 1e-3) / 1e9
        adamw = {"kernel": "adamw_kernel", "tensors": len(ap), "elements": a_elems, "ms_per_step": a_ms,
                 "bound": "hbm", "achieved": a_gbs, "peak": peak_bw, "unit": "GB/s", "frac": a_gbs / peak_bw,
                 "alg_bytes_per_element": 28,
                 "set": "token embedding and untied lm_head (32768 x d each), 2 scalars per layer, smear gate, "
                        "backout lambda; lr 3e-3, betas (0.8, 0.95), eps 1e-8, wd 0.01"}
        del ap, ag, am, av

    # ---- end to end through the C ABI with host buffers.  Every step uploads its
    # gradients from pinned host memory and downloads the updated weights to pinned
    # host memory, all inside the timed region.  The copies are pipelined across
    # steps: step k + 1's gradients upload on one copy stream (double-buffered)
    # while step k computes, and step k's weights are snapshotted on the device
    # and downloaded on a second copy stream while step k + 1 runs.
    e2e = None
    if not args.no_e2e:
        mu.muon_destroy()
        mu.muon_init()
        host_g = [[t.cpu().pin_memory() for t in grads[k]] for k in range(2)]
        host_p = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in p]
        dev_g = [[torch.empty_like(t) for t in g0] for _ in range(2)]
        snap = [torch.empty_like(t) for t in p]
        e2e_args = [mu.StepArgs(p, dev_g[b], m, shapes) for b in range(2)]
        h2d = sum(t.numel() * 4 for t in host_g[0])
        d2h = sum(t.numel() * 4 for t in host_p)
        copy_in = torch.cuda.Stream(device=dev)
        copy_out = torch.cuda.Stream(device=dev)

        def e2e_run(nsteps):
            """Enqueue nsteps pipelined steps; returns the elapsed ms on `stream`."""
            ev_in = [torch.cuda.Event() for _ in range(2)]      # upload into buffer b done
            ev_used = [torch.cuda.Event() for _ in range(2)]    # the step reading buffer b done
            ev_snap, ev_out = torch.cuda.Event(), torch.cuda.Event()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)

            def upload(k):
                b = k % 2
                copy_in.wait_event(ev_used[b])
                with torch.cuda.stream(copy_in):
                    for d, h in zip(dev_g[b], host_g[k % 2]):
                        d.copy_(h, non_blocking=True)
                    ev_in[b].record(copy_in)

            ev0.record(stream)
            copy_in.wait_event(ev0)
            copy_out.wait_event(ev0)
            upload(0)
            for k in range(nsteps):
                if k + 1 < nsteps:
                    upload(k + 1)
                b = k % 2
                stream.wait_event(ev_in[b])
                mu.muon_step(e2e_args[b], lr=hp["lr"], beta=hp["beta"], nesterov=hp["nesterov"],
                             ns_steps=hp["ns_steps"], stream=stream)
                ev_used[b].record(stream)
                stream.wait_event(ev_out)           # the previous download has read the snapshot
                with torch.cuda.stream(stream):
                    for s_, d in zip(snap, p):
                        s_.copy_(d, non_blocking=True)
                    ev_snap.record(stream)
                copy_out.wait_event(ev_snap)
                with torch.cuda.stream(copy_out):
                    for h, s_ in zip(host_p, snap):
                        h.copy_(s_, non_blocking=True)
                    ev_out.record(copy_out)
            stream.wait_event(ev_out)               # the region ends with the last download
            stream.wait_event(ev_in[(nsteps - 1) % 2])
            ev1.record(stream)
            ev1.synchronize()
            return ev0.elapsed_time(ev1)

        def link_gbs():
            """The host link alone: one step's gradient upload, one weight download, and both
            overlapped (pinned buffers, the copy streams the end-to-end steps use)."""
            out = {}
            for name, ups, downs in (("h2d", True, False), ("d2h", False, True), ("both", True, True)):
                barrier()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                copy_in.wait_event(e0)
                copy_out.wait_event(e0)
                done = []
                if ups:
                    with torch.cuda.stream(copy_in):
                        for d, h in zip(dev_g[0], host_g[0]):
                            d.copy_(h, non_blocking=True)
                        done.append(torch.cuda.Event())
                        done[-1].record(copy_in)
                if downs:
                    with torch.cuda.stream(copy_out):
                        for h, s_ in zip(host_p, snap):
                            h.copy_(s_, non_blocking=True)
                        done.append(torch.cuda.Event())
                        done[-1].record(copy_out)
                for ev in done:
                    stream.wait_event(ev)
                e1.record(stream)
                e1.synchronize()
                nbytes = (h2d if ups else 0) + (d2h if downs else 0)
                out[name] = nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
            return out

        e2e_steps = max(2, min(args.steps, 8))
        link_gbs()                                  # warm-up of the copy paths
        link = link_gbs()
        e2e_run(2)                                  # warm-up of the copy path
        barrier()
        ms_e2e = max_over_ranks(e2e_run(e2e_steps), dist, dev) / e2e_steps
        barrier()
        mu.muon_get_status(stream)
        e2e = {"value": job_tflops(world, flops_step, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "link_gbs": link,
               "link_bound_ms_per_step": (h2d + d2h) / (link["both"] * 1e9) * 1e3,
               "path": ("pinned host grads -> muon_step (C ABI) -> pinned host params; uploads double-buffered "
                        "on one copy stream, weights snapshotted on the device and downloaded on another, "
                        "overlapping the next step")}
    mu.muon_destroy()

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": workload_desc(wl), "matrices": len(shapes), "elements": elems,
                           "ns_alg_flops_per_step": flops_step,
                           "parallelism": "replicas" if world > 1 else "single-gpu",
                           "gradients": (f"{n_sets} gradient sets drawn on the device before timing, one per step"
                                         + ("" if n_sets >= args.warmup + args.steps
                                            else f" (reused in turn past {n_sets} steps)")),
                           "l2": (f"no flush: every step reads its own {4 * elems / 1e9:.2f} GB gradient set; "
                                  f"weights and momentum {4 * elems / 1e9:.2f} GB each"
                                  + (", all far above the 126 MB L2" if 4 * elems > 126e6
                                     else " (below the 126 MB L2: small case)")),
                           "state_dtype": "fp32 p/g/m; bf16 Newton-Schulz operands, fp32 accumulation"},
                "ns_tflops": ns_tflops, "frac_of_bf16_peak": ns_tflops / peak_tf_sus, "frac_of_bf16_burst_peak": ns_tflops / peak_tf,
                "step_ms": step_stats, "phase_ms_per_step": phase_ms, "timed_ms_with_kernel_events": timed_ms2 / args.steps,
                "roofline": roofline, "roofline_elementwise": roofline_hbm, "normuon": normuon, "adamw": adamw, "cpu_baseline": cpu, "e2e": e2e,
                "clocks": clocks.summary(), "gpu_launches": info["launches"] * args.steps,
                "workspace_bytes": info["workspace_bytes"]}
        print(json.dumps(line), flush=True)
    return 0


def run_sweep(args) -> int:
    """Newton-Schulz throughput across the shape sweep (n x n, 4n x n, n x 4n for n = 256 ... 8192),
    one GPU.  Each shape runs with an even number of matrices (low-rank and full-rank gradients
    alternate) bounded so that the fp32 state and the bf16 workspace stay under about 40 GB; every
    step is timed alone with CUDA events, with a 256 MB write between steps (outside the events) so
    that no step starts with its operands in L2.  Prints one JSON object with a row per shape."""
    import torch
    import pretraining_optimizer_step_b300 as mu
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_bw = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    rows = []
    for name in workloads.sweep_names():
        all_shapes = workloads.config_shapes(name)
        r, c = all_shapes[0]
        mm, nn = min(r, c), max(r, c)
        per_matrix = 12 * r * c + 4 * mm * nn + 4 * mm * mm
        count = max(2, min(len(all_shapes), int(40e9 // per_matrix)))
        count -= count % 2
        p, g, m, shapes = workloads.make_stack(name, dev, indices=list(range(count)))
        mu.muon_init(debug_flags=mu.MUON_DEBUG_TIME_KERNELS)
        stream = torch.cuda.Stream(device=dev)
        sargs = mu.StepArgs(p, g, m, shapes)
        for _ in range(args.warmup):
            mu.muon_step(sargs, stream=stream)
        mu.muon_get_status(stream)
        # enough steps for about half a second of timed work, so that the clock sampler (50 ms)
        # sees the short shapes run too
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mu.muon_step(sargs, stream=stream)
        e1.record(stream)
        e1.synchronize()
        nsteps = max(args.steps, min(1000, int(500.0 / max(e0.elapsed_time(e1), 1e-3)) + 1))
        mu.muon_get_status(stream)
        mu.muon_kernel_times()
        times = []
        with ClockSampler(0) as clocks:
            for _ in range(nsteps):
                with torch.cuda.stream(stream):
                    flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                mu.muon_step(sargs, stream=stream)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
        mu.muon_get_status(stream)
        kt = mu.muon_kernel_times()
        info = mu.muon_get_step_info()
        q = mu.muon_plan_query(shapes, workloads.HYPER["ns_steps"])
        ns_ms = sum(kt[k][0] for k in ("gram", "poly", "axpy", "axpy_update")) / nsteps
        mom_ms = kt["momentum_norm"][0] / nsteps
        ms = statistics.median(times)
        # ideal NS bytes per matrix and iteration: X read twice and written once (bf16, 6mn), A written
        # and read twice, B' written and read (bf16, 5m^2); below the ridge this is the bound
        ns_bytes = workloads.HYPER["ns_steps"] * count * (6.0 * mm * nn + 5.0 * mm * mm)
        intensity = info["ns_alg_flops"] / ns_bytes
        ridge = peak_sus * 1e12 / (peak_bw * 1e9)
        rows.append({"workload": name, "shape": [r, c], "matrices": count, "steps": nsteps, "ms_per_step": ms,
                     "ns_tflops": info["ns_alg_flops"] / (ns_ms * 1e-3) / 1e12,
                     "ns_frac_of_sustained_bf16": info["ns_alg_flops"] / (ns_ms * 1e-3) / 1e12 / peak_sus,
                     "ns_flop_per_byte": intensity, "ns_bound": "tensor" if intensity >= ridge else "hbm",
                     "ns_alg_gbs": ns_bytes / (ns_ms * 1e-3) / 1e9,
                     "ns_frac_of_hbm": ns_bytes / (ns_ms * 1e-3) / 1e9 / peak_bw,
                     "executed_over_alg_flops": q["ns_executed_flops"] / q["ns_alg_flops"],
                     "momentum_gbs": 14.0 * count * r * c / (mom_ms * 1e-3) / 1e9,
                     "momentum_frac_of_hbm": 14.0 * count * r * c / (mom_ms * 1e-3) / 1e9 / peak_bw,
                     "launches_per_step": info["launches"], "clocks": clocks.summary()})
        mu.muon_destroy()
        del p, g, m, sargs
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": rows, "peak_source": peak_src, "steps": args.steps, "warmup": args.warmup,
                      "timing": "median of per-step CUDA-event times; 256 MB written between steps"}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="d26 (the measured workload) or a smaller case for profiling: d2, d12, d20, sweep_*")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="one GPU: Newton-Schulz throughput over the square / 4:1 shape sweep (not the benchmark line)")
    args = ap.parse_args()
    if args.sweep:
        return run_sweep(args)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    rc = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
