#!/usr/bin/env python3
"""Benchmark of the sm_103a attention forward (one JSON line on rank 0).

A step is one attention forward over the headline workload (B=1, H=32, Nq=Nk=4096, D=128,
bf16, non-causal, Q/K/V ~ N(0,1), scale 1/sqrt(128)). FLOPs per step are 4*B*H*Nq*Nk*D
(halved when causal).

  value     TFLOP/s of the whole job: inputs resident in device memory, W warm-up steps, then
            exactly K timed steps between barrier + synchronize, timed with CUDA events on the
            launching stream, max over ranks. Consecutive steps cycle through several input
            sets whose total exceeds the 129 MB L2, so no step starts on inputs left in L2 by
            the step before.
  e2e       the same metric through fa_fwd_host (host buffers): each step copies Q, K, V from
            pinned host memory, runs the kernel and copies O back.
  roofline  the kernel against the measured dense bf16 peak (MEASURED_PEAKS.json).
  cpu_baseline  the fp64 oracle on the host cores over a bounded sample of the workload.

--impl reference times the oracle itself as the reference arm (the method's pages ship no
runnable implementation). With torchrun (N > 1) each rank runs its own replica of the workload
on its own GPU (the forward pass has no exchange step); value sums the work of all ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "attention fwd TFLOP/s and % of GB300 dense tensor peak (B=1,H=32,L=4096,D=128)"
KERNEL_SOURCES = ["tiled_online_softmax_gb300/csrc/fa_fwd_kernel.cuh",
                  "tiled_online_softmax_gb300/csrc/fa_rope_kernel.cuh",
                  "tiled_online_softmax_gb300/csrc/sm103_ptx.cuh"]
L2_BYTES = 129 * 1000 * 1000
# Timed after the headline and reported in config.extra: the large-magnitude and long causal
# workloads (L >= 4096) and causal prefill.
EXTRA_WORKLOADS = ("rescale_stress", "long_causal", "causal_prefill")
DATASHEET_DENSE_BF16_TFLOPS = 2250.0  # nominal, context only
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def env_rank():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x across the ranks of the default process group (x itself when no
    group is initialised). The timed region's length is the slowest rank's."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica of the workload (weak scaling)."""
    return world * flops_per_rank / seconds / 1e12


def workload_desc(w):
    return (f"{w.name}: B={w.B} H={w.H} Nq={w.Nq} Nk={w.Nk} D={w.D} {w.dtype} "
            f"{'causal' if w.causal else 'non-causal'}")


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_code(text: str) -> str:
    """The source with `//` comments, trailing blanks and empty lines removed: what a comment-only
    edit leaves unchanged. (The kernel sources have no block comments and no `//` in strings.)"""
    lines = []
    for line in text.splitlines():
        line = line.split("//", 1)[0].rstrip()
        if line:
            lines.append(line)
    return "\n".join(lines)


def kernel_source_hash() -> str:
    """Identifies the forward kernel's code; a profile summary taken on other code is not used."""
    h = hashlib.sha256()
    for s in KERNEL_SOURCES:
        h.update(kernel_code((ROOT / s).read_text()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel."""
    f = ROOT / "profiles" / f"fa_fwd_kernel_{workload_name}.md"
    if not f.exists():
        return None
    kv = {}
    for line in f.read_text().splitlines():
        if line.startswith("- ") and ":" in line:
            k, _, v = line[2:].partition(":")
            kv[k.strip()] = v.strip().strip("`")
    if kv.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class _Nvml:
    """Read-only NVML queries (SM clock, clock-event reasons, power draw) through the driver's
    libnvidia-ml, for a sampling thread. The device is found by its UUID, so the index NVML uses
    does not matter."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid: str):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
            raise OSError(f"no NVML device with UUID {uuid}")
        self.reasons_fn = (getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                           or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons)

    def sample(self):
        ct = self.ct
        clk, reasons, mw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(clk)) != 0:  # NVML_CLOCK_SM
            raise OSError("nvmlDeviceGetClockInfo failed")
        self.reasons_fn(self.handle, ct.byref(reasons))
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        return float(clk.value), int(reasons.value), mw.value / 1000.0


def gpu_uuid(dev) -> str | None:
    import torch

    u = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if u is None:
        return None
    u = str(u)
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    """Clock and throttle-reason samples while the GPU works, from two sources: nvidia-smi every
    100 ms (timestamps, power, the reasons), and an NVML thread in this process every ~2 ms, so
    that even a timed region of a few milliseconds holds samples. mark(name) opens a phase
    (closing the previous one). stop(primary) gives per phase the median SM clock of each source,
    and as `sm_mhz` the median NVML clock of the phase `<primary>:timed` (the timed steps of the
    headline workload); failing that, its pre-heat's (a second of the same work just before)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, uuid: str | None = None):
        import threading

        self.proc = None
        self.phases = []  # [name, epoch start, epoch end, perf start, perf end]
        self.fast = []    # (perf_counter, sm MHz, reason bits, W)
        self.nvml_error = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={uuid or gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.nvml = None
        if uuid is not None:
            try:
                self.nvml = _Nvml(uuid)
            except OSError as e:
                self.nvml_error = str(e)
        self._halt = threading.Event()
        self._thread = None
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()

    def _loop(self):
        while not self._halt.is_set():
            t = time.perf_counter()
            try:
                self.fast.append((t, *self.nvml.sample()))
            except OSError as e:
                self.nvml_error = str(e)
                return
            self._halt.wait(0.002)

    def mark(self, name: str | None):
        now, perf = time.time(), time.perf_counter()
        if self.phases and self.phases[-1][2] is None:
            self.phases[-1][2], self.phases[-1][4] = now, perf
        if name is not None:
            self.phases.append([name, now, None, perf, None])

    @staticmethod
    def _epoch(ts: str):
        try:
            base, _, frac = ts.strip().partition(".")
            return time.mktime(time.strptime(base, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
        except ValueError:
            return None

    def stop(self, primary: str | None = None):
        self.mark(None)
        self._halt.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        rows, reasons = [], set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for row in csv.reader(io.StringIO(out)):
                if len(row) < 10:
                    continue
                try:
                    rows.append((self._epoch(row[0]), float(row[2]), float(row[3]), float(row[4])))
                except ValueError:
                    continue
                for name, val in zip(names, row[6:10]):
                    if val.strip().lower() == "active":
                        reasons.add(name)
        if not rows and not self.fast:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"]}
        phases = {}
        for name, t0, t1, p0, p1 in self.phases:
            smi = [r[1] for r in rows if r[0] is not None and t0 <= r[0] <= t1]
            fast = [f for f in self.fast if p0 <= f[0] <= p1]
            for f in fast:
                reasons.update(n for bit, n in _Nvml.REASONS.items() if f[2] & bit)
            phases[name] = {"sm_mhz": statistics.median(smi) if smi else None, "samples": len(smi),
                            "sm_mhz_nvml": statistics.median(f[1] for f in fast) if fast else None,
                            "nvml_samples": len(fast),
                            "sm_mhz_nvml_min": min(f[1] for f in fast) if fast else None,
                            "seconds": t1 - t0}
        sm_mhz, source = None, None
        if primary is not None:
            timed, pre = phases.get(f"{primary}:timed"), phases.get(f"{primary}:preheat")
            if timed and timed["sm_mhz_nvml"] is not None:
                sm_mhz, source = timed["sm_mhz_nvml"], f"{primary}:timed, NVML every ~2 ms"
            elif pre and (pre["sm_mhz_nvml"] or pre["sm_mhz"]) is not None:
                sm_mhz = pre["sm_mhz_nvml"] or pre["sm_mhz"]
                source = f"{primary}:preheat (the second of the same work before the timed steps)"
        all_smi = [r[1] for r in rows]
        return {"sm_mhz": sm_mhz, "sm_mhz_source": source,
                "sm_mhz_all_samples": statistics.median(all_smi) if all_smi else None,
                "sm_max_mhz": max(r[2] for r in rows) if rows else None,
                "power_w_max": max(r[3] for r in rows) if rows else None,
                "samples": len(all_smi), "nvml_samples": len(self.fast),
                "nvml_error": self.nvml_error, "reasons": sorted(reasons), "phases": phases}


class OracleSample:
    """The fp64 oracle over whole (b, h) slices of the workload, timed on the host cores.

    One slice calibrates the per-slice time; a run then covers as many slices as fit the
    requested seconds (at least one, at most all B*H). Inputs are drawn once, outside timing."""

    def __init__(self, w):
        import oracle
        from tiled_online_softmax_gb300 import inputs

        self.w = w
        self.orc = oracle.default()
        self.cores = self.orc.num_threads()
        n_all = w.B * w.H
        bits = inputs.draw(w.with_(B=1, H=n_all))
        self.q, self.k, self.v = (inputs.bits_to_f64(bits[n][0], w.dtype) for n in "qkv")
        self.slice_flops = w.with_(B=1, H=1).flops
        self.t_slice = self._time(1)

    def _time(self, n):
        t0 = time.perf_counter()
        self.orc.attention(self.q[:n], self.k[:n], self.v[:n], self.w.scale, self.w.causal)
        return time.perf_counter() - t0

    def run(self, seconds: float):
        n = max(1, min(len(self.q), int(seconds / max(self.t_slice, 1e-4))))
        t = self._time(n)
        desc = (f"{n} of {len(self.q)} (b,h) slices of the {self.w.name} workload "
                f"({n * self.slice_flops / 1e9:.1f} GFLOP), fp64 two-pass oracle, OpenMP")
        return n * self.slice_flops / t / 1e12, t, desc


def rotating_sets(w, dev):
    """Copies of the workload's inputs (and an output each), enough that consecutive steps never
    start on inputs the step before left in L2."""
    import torch

    from tiled_online_softmax_gb300 import inputs

    bits = inputs.draw(w)
    base = {n: inputs.to_torch(bits[n], w.dtype).to(dev) for n in "qkv"}
    set_bytes = sum(t.numel() * 2 for t in base.values()) + base["q"].numel() * 2
    n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)
    sets = []
    for i in range(n_sets):
        q, k, v = (base[n] if i == 0 else base[n].clone() for n in "qkv")
        sets.append((q, k, v, torch.empty_like(q)))
    return bits, sets, set_bytes


def kernel_time(kernels: dict, ms_per_step: float, steps: int):
    """The attention kernel's time per launch and how it was taken. When a step is exactly one
    attention launch, the timed region's own CUDA events (K launches back to back, as the step
    runs) time the kernel itself. Otherwise the kernel timer's events around each attention launch
    separate it from the merge; those events cut the overlap of consecutive launches (a dependent
    launch's set-up and first loads during its predecessor's tail), so they read a little long.
    Returns (ms, source, ms by the per-launch events)."""
    fwd_ms, fwd_n = kernels["fwd"]
    per_launch = fwd_ms / fwd_n
    if fwd_n == steps and sum(n for _, n in kernels.values()) == steps:
        return (ms_per_step, "CUDA events on the launching stream over the timed region: one "
                "attention launch per step, K launches back to back", per_launch)
    return (per_launch, "CUDA events recorded on the launching stream around each attention "
            "launch (the kernel timer pass: K more steps)", per_launch)


def time_extra(w, dev, stream, steps, warmup, peak, sampler=None, peak_burst=None):
    """One more workload timed the way the headline is (rotating inputs, W warm-up steps and about
    a second of the same work, then K steps between synchronizes with CUDA events on the
    launching stream, then the same K steps with the kernel timer on). Not part of `value`."""
    import torch

    from tiled_online_softmax_gb300 import fa

    _, sets, set_bytes = rotating_sets(w, dev)
    n = len(sets)

    def step(i):
        q, k, v, o = sets[i % n]
        fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=o, stream=stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark(f"{w.name}:preheat")
    t_end = time.perf_counter() + 1.0
    i = 0
    while time.perf_counter() < t_end:
        for _ in range(4):
            step(i)
            i += 1
        torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark(f"{w.name}:timed")
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / steps
    if sampler:
        sampler.mark(f"{w.name}:kernel_timer")
    fa.timer_start()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize(dev)
    kernels = fa.timer_stop()
    if sampler:
        sampler.mark(None)
    kernel_ms, kernel_src, per_launch_ms = kernel_time(kernels, ms, steps)
    tflops = w.flops / (ms * 1e-3) / 1e12
    kernel_tflops = w.flops / (kernel_ms * 1e-3) / 1e12
    del sets
    return {"workload": workload_desc(w), "flops_per_step": w.flops, "ms_per_step": ms,
            "tflops": tflops, "pct_of_measured_peak": 100 * tflops / peak,
            "pct_of_measured_burst_peak": 100 * tflops / (peak_burst or peak),
            "kernel_ms": kernel_ms, "kernel_ms_source": kernel_src,
            "kernel_ms_per_launch_events": per_launch_ms, "kernel_tflops": kernel_tflops,
            "kernel_frac": kernel_tflops / peak, "launches_per_step": sum(c for _, c in kernels.values()) / steps,
            "l2": f"{n} rotating input sets of {set_bytes / 2**20:.0f} MiB"}


def run_reference(args, w):
    """The reference arm: the fp64 oracle on the host cores (rank 0 only), each step a bounded
    sample of the workload sized so that the whole run takes about two minutes."""
    rank, _, world = env_rank()
    if rank != 0:
        return 0
    sample = OracleSample(w)
    per_step = min(args.ref_seconds, 120.0 / (args.warmup + args.steps))
    tflops_runs, desc = [], ""
    for i in range(args.warmup + args.steps):
        tf, _, desc = sample.run(per_step)
        if i >= args.warmup:
            tflops_runs.append(tf)
    value = statistics.median(tflops_runs)
    ms = w.flops / (value * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": w.B, "seq_len": w.Nq,
                   "parallelism": "cpu"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": sample.cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_other_pass(args, w):
    """Timing of the backward pass or of the rotary-embedding pass on one GPU (one JSON line;
    not the headline metric)."""
    import torch

    from tiled_online_softmax_gb300 import fa, inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.lib()
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).to(dev) for n in "qkv")
    stream = torch.cuda.current_stream(dev)
    if args.which == "bwd":
        do = inputs.to_torch(inputs.draw(w.with_(seed=w.seed + 1000))["q"], w.dtype).to(dev)
        o, lse = fa.forward_lse(q, k, v, causal=w.causal, scale=w.scale)
        ws = torch.empty(fa.lib().fa_bwd_workspace_bytes(w.B, w.H, w.Nq), dtype=torch.uint8, device=dev)
        step = lambda: fa.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale,
                                   workspace=ws, stream=stream)
        work, unit = 2.5 * w.flops, "TFLOP/s"
        metric = "attention bwd TFLOP/s (10*B*H*Nq*Nk*D, halved for causal)"
        # Tensor-core work each kernel executes: 2*B*H*Nq*Nk*D (halved causal) per product;
        # dK/dV recomputes S and dP and forms dV and dK (4 products), dQ recomputes S and dP and
        # forms dQ (3 products).
        kernel_work = {"bwd_dkdv": 2.0 * w.flops, "bwd_dq": 1.5 * w.flops}
    else:
        half = w.D // 2
        ang = np.arange(max(w.Nq, w.Nk))[:, None] * 10000.0 ** (-np.arange(half) / half)
        ct = torch.from_numpy(np.cos(ang).astype(np.float32)).to(dev)
        st_ = torch.from_numpy(np.sin(ang).astype(np.float32)).to(dev)
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        if args.which == "rope":
            def step():
                fa.rope(q, ct[:w.Nq], st_[:w.Nq], out=qo, stream=stream)
                fa.rope(k, ct[:w.Nk], st_[:w.Nk], out=ko, stream=stream)
            # algorithmic bytes: read and write Q and K once; the cos/sin tables ([N, D/2] fp32,
            # shared by every batch and head) once
            work = 2 * (q.numel() + k.numel()) * 2 + (w.Nq + w.Nk) * half * 8
            unit = "GB/s"
            kernel_work = {"rope": work}
            metric = "rotary embedding of Q and K, GB/s"
        else:
            # attention on rotary-embedded Q and K: fa_fwd_rope (K rotated by its own pass, Q
            # inside the attention kernel), against the same work as three separate passes
            o = torch.empty_like(q)
            ws = torch.empty(fa.lib().fa_rope_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.D),
                             dtype=torch.uint8, device=dev)
            cq, sq, ck, sk = ct[:w.Nq], st_[:w.Nq], ct[:w.Nk], st_[:w.Nk]

            def step():
                fa.forward_rope(q, k, v, cq, sq, ck, sk, causal=w.causal, scale=w.scale, out=o,
                                workspace=ws, stream=stream)

            def step_separate():
                fa.rope(q, cq, sq, out=qo, stream=stream)
                fa.rope(k, ck, sk, out=ko, stream=stream)
                fa.forward(qo, ko, v, causal=w.causal, scale=w.scale, out=o, stream=stream)
            work, unit = w.flops, "TFLOP/s"
            kernel_work = {"fwd": w.flops}
            metric = "attention fwd with rotary Q and K, TFLOP/s (4*B*H*Nq*Nk*D, halved causal)"
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # About a second of the same work first, as for the forward pass, so that the timed steps
    # run at the clock this load settles to.
    sampler = ClockSampler(dev.index, gpu_uuid(dev))
    sampler.mark(f"{w.name}:preheat")
    t_end = time.perf_counter() + 1.0
    while time.perf_counter() < t_end:
        step()
        torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark(f"{w.name}:timed")
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark(None)
    # Per-kernel device times from a second pass with the library's kernel timer on (its events
    # add small gaps between launches, so it stays out of the timed region).
    fa.timer_start()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    kernels = fa.timer_stop()
    st, site = fa.last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"kernel error word set (site {site})")
    ms = e0.elapsed_time(e1) / args.steps
    value = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    separate = None
    if args.which == "rope_fwd":
        # The two forms alternate in blocks of K steps (6 rounds), so that both see the same
        # clocks under the power cap; the medians are compared.
        for _ in range(args.warmup):
            step_separate()
        torch.cuda.synchronize(dev)
        blocks = {"fused": [], "separate": []}
        for _ in range(6):
            for form, fn in (("fused", step), ("separate", step_separate)):
                e0.record(stream)
                for _ in range(args.steps):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                blocks[form].append(e0.elapsed_time(e1) / args.steps)
        med = {f: float(np.median(v)) for f, v in blocks.items()}
        separate = {"form": "fa_rope(Q), fa_rope(K), fa_fwd: three passes",
                    "ms_per_step": med["separate"], "tflops": work / (med["separate"] * 1e-3) / 1e12,
                    "interleaved_rounds": 6, "fused_ms_per_step_interleaved": med["fused"],
                    "fused_over_separate_time": med["fused"] / med["separate"]}
    peaks, kind = load_peaks()
    # Pre-heated like the forward pass: the sustained figure for tensor work.
    peak = float(peaks["bf16_tflops_sustained"] if unit == "TFLOP/s" else peaks["hbm_gbs"])
    # Roofline of the dominant kernel: its work per step over its own event-timed device time.
    top = max(kernel_work, key=lambda k: kernels[k][0])
    top_ms = kernels[top][0] / args.steps
    achieved = kernel_work[top] / (top_ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({
        "metric": metric, "pass": args.which, "value": value, "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "dtype": w.dtype, "data": "synthetic", "config": {"workload": workload_desc(w)},
        "roofline": {"bound": "tensor" if unit == "TFLOP/s" else "hbm", "achieved": achieved,
                     "peak": peak, "unit": unit, "frac": achieved / peak, "kernel": top,
                     "kernel_ms_per_step": top_ms,
                     "kernels_ms_per_step": {k: v[0] / args.steps for k, v in kernels.items()},
                     "peak_kind": f"{kind} " + ("bf16 dense, sustained" if unit == "TFLOP/s" else "copy bandwidth"),
                     "frac_of_burst_peak": (achieved / float(peaks["bf16_tflops"])) if unit == "TFLOP/s" else None},
        "separate_passes": separate, "clocks": sampler.stop(w.name),
        "gpu_launches": sum(n for _, n in kernels.values())}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd", "rope", "rope_fwd"],
                    default="fwd",
                    help="fwd: the forward pass (the headline metric); bwd: fa_bwd after one "
                         "forward; rope: the rotary-embedding pass over Q and K; rope_fwd: "
                         "attention on rotary-embedded Q and K (fa_fwd_rope) against three "
                         "separate passes")
    ap.add_argument("--splits", type=int, default=0,
                    help="N > 1: time the split-KV entry with N key ranges (non-causal); "
                         "0: fa_fwd, which splits few-unit shapes over keys by itself")
    ap.add_argument("--ref-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads timed after the headline (config.extra)")
    ap.add_argument("--profile", action="store_true",
                    help="profiler runs: only the warm-up and timed launches (no clock pre-heat, "
                         "e2e or CPU leg); the printed numbers are not bench values")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from tiled_online_softmax_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.which != "fwd":
        return run_other_pass(args, w)

    import torch
    import torch.distributed as dist

    from tiled_online_softmax_gb300 import fa

    rank, local_rank, world = env_rank()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    fa.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    # Input sets: cycle through enough of them that consecutive steps never share L2 contents.
    bits, sets, set_bytes = rotating_sets(w, dev)
    n_sets = len(sets)
    stream = torch.cuda.current_stream(dev)

    # fa_fwd balances work by itself (few units: every unit split over keys, then merged). An
    # explicit --splits N > 1 times the split-KV entry with N key ranges instead.
    use_split = (not w.causal) and args.splits > 1
    workspace = None
    if use_split:
        workspace = torch.empty(max(1, fa.splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.D,
                                                                  args.splits)),
                                dtype=torch.uint8, device=dev)

    def step(i):
        q, k, v, o = sets[i % n_sets]
        if use_split:
            fa.forward_splitkv(q, k, v, num_splits=args.splits, scale=w.scale, out=o,
                               workspace=workspace, stream=stream)
        else:
            fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=o, stream=stream)

    # Warm-up, then about a second of the same work with the clock sampler already running,
    # so its samples describe the GPU under this load.
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index, gpu_uuid(dev)) if not args.profile else None
    if sampler:
        sampler.mark(f"{w.name}:preheat")
    t_end = time.perf_counter() + (0.0 if args.profile else 1.0)
    i = 0
    while time.perf_counter() < t_end:
        for _ in range(8):
            step(i)
            i += 1
        torch.cuda.synchronize(dev)

    # Timed region: exactly K steps.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark(f"{w.name}:timed")
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    if sampler:
        sampler.mark(f"{w.name}:kernel_timer")
    # The same K steps again with the library's kernel timer on: CUDA events around each launch,
    # on its stream, give every kernel's own device time. The events add small gaps between
    # launches, so this pass is kept out of the timed region above.
    fa.timer_start()
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize(dev)
    kernels = fa.timer_stop()
    if sampler:
        sampler.mark(None)
    # The other workloads the target names (L >= 4096, and causal prefill), timed the same way
    # while the clock sampler still runs.
    peaks, peaks_kind = load_peaks()
    # The timed steps run back to back after a second of the same work, in the power-capped
    # steady state, like the sustained GEMM loop of the peak measurement: that is the denominator
    # (the burst figure, taken on a cold GPU at its highest clocks, is reported beside it).
    peak = float(peaks["bf16_tflops_sustained"])
    peak_burst = float(peaks["bf16_tflops"])
    extra = {}
    if not args.profile and not args.no_extra and args.workload == "headline":
        del sets
        torch.cuda.empty_cache()
        for name in EXTRA_WORKLOADS:
            extra[name] = time_extra(inputs.WORKLOADS[name], dev, stream, args.steps, args.warmup,
                                     peak, sampler, peak_burst)
            torch.cuda.empty_cache()
    clocks = sampler.stop(w.name) if sampler else None
    ms_total = max_over_ranks(ms_total, dev)
    ms_per_step = ms_total / args.steps
    value = job_throughput(w.flops, world, ms_per_step * 1e-3)

    if args.profile:
        if rank == 0:
            print(json.dumps({"profile_run": True, "ms_per_step": ms_per_step}), flush=True)
        return 0

    # e2e: host buffers through fa_fwd_host, copies inside the timed region.
    qh, kh, vh = (inputs.to_torch(bits[n], w.dtype).pin_memory() for n in "qkv")
    oh = torch.empty_like(qh).pin_memory()
    fa.forward_host(qh, kh, vh, oh, causal=w.causal, scale=w.scale, stream=stream,
                    device=dev.index)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        fa.forward_host(qh, kh, vh, oh, causal=w.causal, scale=w.scale, stream=stream,
                        device=dev.index)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, dev)
    h2d = sum(t.numel() * 2 for t in (qh, kh, vh))
    d2h = oh.numel() * 2

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # The dominant kernel: the attention kernel, one launch per step (the merge of a split
    # last wave, when there is one, is a second, short launch).
    fwd_ms = kernels["fwd"][0]
    kernel_ms, kernel_src, per_launch_ms = kernel_time(kernels, ms_per_step, args.steps)
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    all_ms = sum(v[0] for v in kernels.values())
    traffic, traffic_src = profiled_traffic(w.name), None
    if traffic is not None:
        traffic_src = (f"ncu dram__bytes_read.sum + dram__bytes_write.sum from "
                       f"profiles/fa_fwd_kernel_{w.name}.md, taken on kernel code hash "
                       f"{kernel_source_hash()} (the code benched here)")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "kernel": "fa_fwd_kernel", "kernel_ms": kernel_ms, "kernel_ms_source": kernel_src,
                "kernel_ms_per_launch_events": per_launch_ms,
                "kernels_ms_per_step": {k: v[0] / args.steps for k, v in kernels.items()},
                "fwd_share_of_kernel_time": fwd_ms / all_ms if all_ms else None,
                "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                "peak_kind": f"{peaks_kind} bf16 dense, sustained (the kernel is timed back to back "
                             f"after 1 s of the same work, power-capped)",
                "frac_of_burst_peak": achieved / peak_burst, "burst_peak": peak_burst,
                "frac_of_datasheet": achieved / DATASHEET_DENSE_BF16_TFLOPS}

    cpu = None
    if not args.no_cpu_baseline:
        sample = OracleSample(w)
        tf, secs, desc = sample.run(args.ref_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": sample.cores, "kind": "oracle",
               "sample": desc, "seconds": secs}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": w.B * world, "seq_len": w.Nq,
                   "parallelism": f"replicas{world}",
                   "l2": f"{n_sets} rotating input sets of {set_bytes / 2**20:.0f} MiB "
                         f"(> L2 between consecutive steps)",
                   "pct_of_measured_peak": 100 * value / peak,
                   "pct_of_measured_burst_peak": 100 * value / peak_burst,
                   "kernel_pct_of_measured_peak": 100 * achieved / peak,
                   "key_splits": args.splits if use_split else "auto",
                   "extra": extra or None},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_throughput(w.flops, world, e2e_s), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3},
        "clocks": clocks,
        "gpu_launches": sum(n for _, n in kernels.values()),  # per K steps, by the timer
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
