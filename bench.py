#!/usr/bin/env python3
"""Benchmark of FP8 Lean-P causal prefill attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one call of the whole hot path -- ``attn_fwd_fp8`` (one kernel
launch) -- on the headline workload: FP8 e4m3, B=1, Hq=Hkv=32, S=32768,
Dqk=Dv=128, Gaussian inputs quantised per tensor.  Q, K and V (3 x 134 MB)
exceed the 129 MB L2, so no flush is needed between steps.

Rank 0 prints one JSON line.  ``value`` is TFLOP/s over all ranks with the
algorithmic causal FLOP count 2*B*Hq*(Dqk+Dv)*S*(S+1)/2; the count of the
formula 2*B*Hq*S^2*(Dqk+Dv) (twice the causal work) is reported beside it.
Under torchrun every rank runs its own copy of the workload (independent
problems, no collective on the data path: weak scaling).

``--impl reference`` times the CPU oracle (the Lean-P emulation) on the host
cores instead, on bounded row samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "fp8_h32_s32k_d128"
METRIC = "causal prefill attn TFLOP/s (FP8 hd128 S=32K) and % of GB300 dense FP8 peak"
FP8_OVER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor-core ratio (4.5 : 2.25 PFLOP/s)


def causal_flops(B, Hq, S, Dqk, Dv):
    return 2.0 * B * Hq * (Dqk + Dv) * S * (S + 1) / 2.0


def square_flops(B, Hq, S, Dqk, Dv):
    return 2.0 * B * Hq * S * S * (Dqk + Dv)


def rows_flops(rows, Dqk, Dv):
    return float(sum(2.0 * (Dqk + Dv) * (int(i) + 1) for _, _, i in rows))


# The articles' own figure for this metric and workload: 2672 TFLOP/s for
# FP8 Lean-P at head dim 128, S = 32K, Gaussian inputs ("Zyphra ZYFA: FP8
# FlashAttention for AMD MI355X", "How fast is ZYFA?").  It was measured on an
# AMD MI355X, so the ratio is context, not a target.  The articles give 53% of
# that GPU's dense FP8 peak for it, which fits the causal FLOP count used here.
PAGES_TFLOPS = 2672.0
PAGES_NOTE = ("value / 2672 TFLOP/s, the articles' figure for FP8 Lean-P at hd128, S=32K on "
              "AMD MI355X (other hardware; causal FLOP count)")


def max_over_ranks(ms, device=None):
    """Largest per-rank step time (the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, world, ms_max):
    """Whole-job throughput: every rank processes its own copy of the workload."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# DRAM traffic of one Lean-P launch on the headline workload, read from an ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum; profiles/ has the
# summary and the command).  It belongs to the kernel sources it was taken
# with: for any other sources the bench reports null.
PROFILED_TRAFFIC = {"bytes": 3951305216,
                    "sources_sha256": "2c0543fb1e52dfcebee2e8a494b84e0e9945b325b0108f8bcc904c0c1700463d"}
# (the kernel, its PTX helpers and its launch; the host-only split planner in
# split_plan.h does not touch the whole-item launch and is not part of the key)
KERNEL_SOURCES = ("fp8_causal_prefill_flash_gb300/csrc/attn_fwd.cuh",
                  "fp8_causal_prefill_flash_gb300/csrc/ptx.cuh",
                  "fp8_causal_prefill_flash_gb300/csrc/api.cu")


def _code_only(src):
    """Source text without comments and blank lines, so that a comment edit
    does not count as a kernel change."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def profiled_traffic():
    if PROFILED_TRAFFIC["bytes"] is None:
        return None
    return PROFILED_TRAFFIC["bytes"] if kernel_sources_sha256() == PROFILED_TRAFFIC["sources_sha256"] \
        else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_burst": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured",
                "sustained_mhz": (d.get("clocks_under_load") or {}).get("sm_mhz_median")}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback", "sustained_mhz": None}


# Tensor-pipe work per SM and clock, measured on GB300 with one-CTA
# microbenchmarks: a 128x128x32 FP8 MMA (kind::f8f6f4, also block-scaled)
# every 64 clocks, a 128x128x16 BF16 MMA every 64 clocks.  Times the SM count
# and a clock, this is the clock-rated ceiling of a contraction.
MMA_FLOP_PER_CLK_SM = {"fp8": 16384.0, "bf16": 8192.0}


def clock_rated_peak(kind, sms, mhz):
    """TFLOP/s the tensor pipes of `sms` SMs issue at `mhz` (None if unknown)."""
    if not mhz:
        return None
    return MMA_FLOP_PER_CLK_SM[kind] * sms * mhz * 1e6 / 1e12


def clock_normalised(achieved, kind, peaks, sms, kernel_mhz):
    """The achieved rate against two clock-aware denominators: the measured
    sustained bf16 GEMM scaled from the clock it ran at to the kernel's
    median clock (x2 for FP8, the nominal ratio), and the tensor pipes'
    clock-rated ceiling at the kernel's median clock."""
    out = {"kernel_sm_mhz": kernel_mhz}
    if kernel_mhz and peaks.get("sustained_mhz"):
        ratio = FP8_OVER_BF16 if kind == "fp8" else 1.0
        p = peaks["bf16_sustained"] * ratio * kernel_mhz / peaks["sustained_mhz"]
        out["measured_sustained_at_kernel_clock"] = {
            "peak": p, "frac": achieved / p,
            "how": (f"{peaks['bf16_sustained']} TFLOP/s bf16 sustained at a median "
                    f"{peaks['sustained_mhz']} MHz, x {ratio} x (kernel MHz / that MHz)")}
    p = clock_rated_peak(kind, sms, kernel_mhz)
    if p:
        out["mma_issue_rate_at_kernel_clock"] = {
            "peak": p, "frac": achieved / p,
            "how": f"{MMA_FLOP_PER_CLK_SM[kind]:.0f} FLOP/clk/SM x {sms} SMs x kernel MHz"}
    return out


# --------------------------------------------------------------------------- energy
class E2EPipeline:
    """Pipelined end-to-end steps through the public API.  Step i uses device
    buffer set i % 2: its upload runs on one copy stream after the call of
    step i-2 (same set) has finished reading the inputs, the call waits for
    the upload and for the download of step i-2 (same output buffer), and
    the download runs on a second copy stream after the call."""

    def __init__(self, torch, fa, dev, host_in, descales, host_out, stream):
        self.torch, self.fa, self.d, self.stream = torch, fa, descales, stream
        self.host_in, self.host_out = host_in, host_out
        self.dev_in = [[torch.empty_like(h, device=dev) for h in host_in] for _ in range(2)]
        self.dev_out = [torch.empty(host_out.shape, dtype=host_out.dtype, device=dev)
                        for _ in range(2)]
        self.up, self.down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.uploaded, self.called, self.downloaded = ev(), ev(), ev()
        self.i = 0

    def step(self):
        torch, s = self.torch, self.i % 2
        if self.i >= 2:
            self.up.wait_event(self.called[s])
        with torch.cuda.stream(self.up):
            for dst, src in zip(self.dev_in[s], self.host_in):
                dst.copy_(src, non_blocking=True)
            self.uploaded[s].record(self.up)
        self.stream.wait_event(self.uploaded[s])
        if self.i >= 2:
            self.stream.wait_event(self.downloaded[s])
        q, k, v = self.dev_in[s]
        self.fa.attn_fwd_fp8(q, k, v, *self.d, out=self.dev_out[s])
        self.called[s].record(self.stream)
        self.down.wait_event(self.called[s])
        with torch.cuda.stream(self.down):
            self.host_out.copy_(self.dev_out[s], non_blocking=True)
            self.downloaded[s].record(self.down)
        self.i += 1

    def finish(self):
        """Make the compute stream wait for every outstanding download."""
        for s in range(2):
            if self.i > s:
                self.stream.wait_event(self.downloaded[s])

    def timed(self, n, warm, barrier):
        torch = self.torch
        for _ in range(warm):
            self.step()
        self.finish()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(n):
            self.step()
        self.finish()
        e1.record(self.stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(e0.elapsed_time(e1) / n, self.stream.device)


class EnergyMeter:
    """GPU energy from NVML's total-energy counter (millijoules since the
    driver loaded), read through ctypes from the driver's NVML library.
    ``read_mj`` returns None when NVML, the device or the counter is missing.
    ``nvml`` may be given an object with the same three calls (tests)."""

    def __init__(self, gpu_uuid=None, nvml=None):
        self.handle = None
        self.nvml = nvml
        try:
            if self.nvml is None:
                import ctypes
                lib = ctypes.CDLL("libnvidia-ml.so.1")
                if lib.nvmlInit_v2() != 0:
                    return
                self.nvml = lib
            import ctypes
            h = ctypes.c_void_p()
            if gpu_uuid:
                rc = self.nvml.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(h))
            else:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h))
            if rc == 0:
                self.handle = h
        except (OSError, AttributeError):
            self.handle = None

    def read_mj(self):
        if self.handle is None:
            return None
        import ctypes
        e = ctypes.c_ulonglong(0)
        if self.nvml.nvmlDeviceGetTotalEnergyConsumption(self.handle, ctypes.byref(e)) != 0:
            return None
        return int(e.value)


def energy_report(mj0, mj1, flops):
    """Joules between two counter readings and TFLOP per joule (None if unread)."""
    if mj0 is None or mj1 is None or mj1 <= mj0:
        return None
    j = (mj1 - mj0) / 1000.0
    return {"joules": j, "tflop_per_joule": flops / 1e12 / j, "source": "NVML total energy counter"}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) taken while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid=None):
        self.proc = None
        self.lines = []
        self.gpu = gpu_uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu:
            cmd += ["-i", self.gpu]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, p in zip(names, parts[5:9]):
                if p.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "power_w_median": statistics.median(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- oracle arm
def sample_rows(S, Hq, n, seed):
    rng = np.random.default_rng(seed)
    return np.stack([np.zeros(n, np.int64), rng.integers(0, Hq, n), rng.integers(0, S, n)], 1)


def oracle_leg(case, rows):
    """Time the CPU oracle (Lean-P emulation, as it stands) on `rows`."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    out, _ = oracle.emul_leanp(case.q, case.k, case.v, case.dq, case.dk, case.dv, rows=rows)
    dt = time.perf_counter() - t0
    return out, dt


def cores_used():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from fp8_causal_prefill_flash_gb300 import workloads as wl
    case = wl.make_case(WORKLOAD)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    # bounded sample: about args.ref_row_budget rows over the whole run
    n_rows = max(4, args.ref_row_budget // (args.warmup + args.steps))
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        rows = sample_rows(S, Hq, n_rows, 1000 + step)
        _, dt = oracle_leg(case, rows)
        if step >= args.warmup:
            times.append(dt)
            flops.append(rows_flops(rows, Dqk, Dv))
    tflops = sum(flops) / sum(times) / 1e12
    sample = (f"{n_rows} random (head, row) pairs of the {WORKLOAD} workload per step, "
              f"oracle_emul_leanp (C, fp64, OpenMP)")
    line = {"impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": tflops / PAGES_TFLOPS,
            "vs_baseline_note": PAGES_NOTE, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "Hq": Hq, "Hkv": Hkv, "S": S, "Dqk": Dqk,
                       "Dv": Dv, "sample_rows_per_step": n_rows},
            "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores_used(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world, local_rank):
    import torch

    import fp8_causal_prefill_flash_gb300 as fa
    from fp8_causal_prefill_flash_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa.build()
    fa.load_library()

    workload = args.workload
    case = wl.make_case(workload, S=args.S)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    F = causal_flops(B, Hq, S, Dqk, Dv)
    Fsq = square_flops(B, Hq, S, Dqk, Dv)
    pin = lambda a: torch.from_numpy(a).pin_memory()
    hq, hk, hv = pin(case.q), pin(case.k), pin(case.v)
    q, k, v = (t.to(dev) for t in (hq, hk, hv))
    d = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (case.dq, case.dk, case.dv)]
    out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def step():
        fa.attn_fwd_fp8(q, k, v, *d, out=out)

    per_launch = []

    def timed(fn, n, warm, record=False):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        evs[0].record(stream)
        for i in range(n):
            fn()
            evs[i + 1].record(stream)  # per-launch times: an event between launches
        torch.cuda.synchronize()
        barrier()
        if record:
            per_launch[:] = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
        return max_over_ranks(evs[0].elapsed_time(evs[n]) / n, dev)

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    meter = EnergyMeter(uuid)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    h_warm = output_sha256(out)
    clocks.start()
    time.sleep(0.3)
    e_start = meter.read_mj()
    ms = timed(step, args.steps, 0, record=True)
    e_end = meter.read_mj()
    clk = clocks.stop()
    h_timed = output_sha256(out)

    # exact-softmax FP8 ablation, same workload
    def step_abl():
        fa.attn_fwd_fp8_exact(q, k, v, *d, out=out)
    ms_abl = timed(step_abl, max(3, args.steps // 4), 3)
    # the diagnostic block-exact variant (Lean-P with an exponential for the
    # code), same workload: splits Lean-P's gain into its two steps
    def step_bx():
        fa.attn_fwd_ex(fa.ATTN_VARIANT_BLOCK_EXACT, q, k, v, *d, out=out,
                       out_dtype=fa.ATTN_OUT_BF16)
    ms_bx = timed(step_bx, max(3, args.steps // 4), 3)
    # Lean-P with the code grid anchored at the running row maximum
    def step_a3():
        fa.attn_fwd_ex(fa.ATTN_VARIANT_LEANP_A3, q, k, v, *d, out=out,
                       out_dtype=fa.ATTN_OUT_BF16)
    ms_a3 = timed(step_a3, max(3, args.steps // 4), 3)
    # sustained: back-to-back Lean-P calls for about args.sustained_s seconds,
    # with the SM clock sampled throughout
    n_sus = max(10, int(args.sustained_s * 1e3 / max(ms, 1e-3)))
    clk_sus = ClockSampler(uuid)
    clk_sus.start()
    time.sleep(0.3)
    ms_sus = timed(step, n_sus, 0)
    clk_sus = clk_sus.stop()

    # end to end through the public API with host buffers: every step copies
    # its q, k, v from pinned memory and its output back into pinned memory.
    # Serial: copy in, call, copy out on one stream.
    hout = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16).pin_memory()

    def step_e2e_serial():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        fa.attn_fwd_fp8(q, k, v, *d, out=out)
        hout.copy_(out, non_blocking=True)
    # at least 20 steps: a short pipelined run is dominated by filling it
    n_e2e = max(20, args.steps // 10)
    ms_e2e_serial = timed(step_e2e_serial, n_e2e, 4)
    # Pipelined (a serving loop): two device buffer sets; the upload of step
    # i+1 (copy stream) and the download of step i-1 (second copy stream)
    # overlap the call of step i.  The timed region ends when the last
    # download is complete.
    e2e = E2EPipeline(torch, fa, dev, (hq, hk, hv), d, hout, stream)
    ms_e2e = e2e.timed(n_e2e, 4, barrier)
    h2d = hq.numel() + hk.numel() + hv.numel()
    d2h = hout.numel() * 2
    del e2e, hq, hk, hv, hout
    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the second target and the other shapes, each timed alone on its own
    # workload: BF16 at 16K (GQA 32/8) and Lean-P at the MLA shape
    extra = {} if args.no_extra else extra_legs(torch, fa, wl, dev, stream, timed, peaks, sms,
                                                max(5, args.steps // 4))

    peak_fp8 = peaks["bf16_burst"] * FP8_OVER_BF16
    per_gpu = F / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": job_tflops(F, world, ms), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_launch": {"median": statistics.median(per_launch), "min": min(per_launch),
                              "max": max(per_launch),
                              "how": "CUDA events between the timed launches (this rank)"},
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": job_tflops(F, world, ms) / PAGES_TFLOPS, "vs_baseline_note": PAGES_NOTE,
            "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": workload, "B": B, "Hq": Hq, "Hkv": Hkv, "S": S, "Dqk": Dqk,
                       "Dv": Dv, "inputs": "N(0,1) per-tensor e4m3, seeds 30/31/32",
                       "l2": "inputs (403 MB) larger than L2 (129 MB); no flush",
                       "flop_count": "causal 2*B*Hq*(Dqk+Dv)*S*(S+1)/2 per rank"},
            "value_square_formula": job_tflops(Fsq, world, ms),
            "frac_of_fp8_peak": per_gpu / peak_fp8,
            "frac_clock_aware": clock_normalised(per_gpu, "fp8", peaks, sms, clk.get("sm_mhz")),
            "ablation_exact_fp8": {"value": job_tflops(F, world, ms_abl), "ms_per_step": ms_abl},
            "block_exact_fp8": {"value": job_tflops(F, world, ms_bx), "ms_per_step": ms_bx,
                                "note": "Lean-P's block scale and rounded row sum with an "
                                        "exponential in place of the one-FMA code"},
            "leanp_running_max_anchor": {"value": job_tflops(F, world, ms_a3), "ms_per_step": ms_a3,
                                         "note": "Lean-P with the code grid anchored at the "
                                                 "running row maximum (exact O rescale)"},
            "sustained": {"value": job_tflops(F, world, ms_sus), "ms_per_step": ms_sus,
                          "calls": n_sus, "seconds": n_sus * ms_sus / 1e3, "clocks": clk_sus,
                          "tflops_per_ghz": (per_gpu * ms / ms_sus) / (clk_sus["sm_mhz"] / 1e3)
                          if clk_sus.get("sm_mhz") else None,
                          "frac_clock_aware": clock_normalised(F / (ms_sus * 1e-3) / 1e12, "fp8",
                                                               peaks, sms, clk_sus.get("sm_mhz"))},
            **extra,
            "roofline": {"bound": "tensor", "achieved": per_gpu, "peak": peak_fp8,
                         "unit": "TFLOP/s", "frac": per_gpu / peak_fp8,
                         "traffic": args.traffic if args.traffic is not None else profiled_traffic(),
                         "peak_note": (f"derived, not an FP8 measurement: {peaks['source']} bf16 "
                                       f"burst {peaks['bf16_burst']} TFLOP/s x {FP8_OVER_BF16} "
                                       f"(nominal FP8:BF16); clock-aware fractions in "
                                       f"frac_clock_aware")},
            "e2e": {"value": job_tflops(F, world, ms_e2e), "unit": "TFLOP/s",
                    "ms_per_step": ms_e2e, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "mode": "pipelined over steps: upload of step i+1 and download of step "
                            "i-1 overlap the call of step i (two copy streams, two buffer sets)",
                    "serial": {"value": job_tflops(F, world, ms_e2e_serial),
                               "ms_per_step": ms_e2e_serial}},
            "gpu_launches": args.steps,
            "determinism": {"output_sha256": h_timed, "same_after_warmup_and_timed_steps":
                            h_warm == h_timed},
            "clocks": clk,
            "energy": energy_report(e_start, e_end, F * args.steps)}

    if rank == 0 and world == 1 and not args.no_cpu:
        # CPU oracle on a bounded sample of the same workload, and the accuracy
        # of both GPU paths on those rows against fp64 attention
        import oracle
        rows = sample_rows(S, Hq, args.cpu_rows, 7)
        emu, dt = oracle_leg(case, rows)
        line["cpu_baseline"] = {
            "value": rows_flops(rows, Dqk, Dv) / dt / 1e12, "unit": "TFLOP/s",
            "cores": cores_used(), "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{len(rows)} random (head, row) pairs of {workload}, oracle_emul_leanp, "
                      f"{dt:.1f} s"}
        # whole-output relative RMS error against fp64 attention, estimated
        # from a stratified sample: every row with fewer than 512 keys (about
        # half of the output's sum of squares) and args.acc_rows weighted rows
        acc_rows, w = wl.stratified_rows(B, Hq, S, short=512, n_long=args.acc_rows, seed=1)
        ref = oracle.ref_fp64(case.q, case.k, case.v, case.dq, case.dk, case.dv, rows=acc_rows)
        pick = lambda o, rr: np.stack([o[b, i, h] for b, h, i in rr]).astype(np.float64)
        rel = lambda x: float(np.sqrt(np.sum(w[:, None] * (x - ref) ** 2) /
                                      np.sum(w[:, None] * ref ** 2)))
        acc = {}
        for key, var in (("leanp", fa.ATTN_VARIANT_LEANP), ("ablation", fa.ATTN_VARIANT_EXACT_FP8),
                         ("leanp_running_max_anchor", fa.ATTN_VARIANT_LEANP_A3)):
            o = fa.attn_fwd_ex(var, q, k, v, *d).cpu().numpy()
            acc[key] = rel(pick(o, acc_rows))
            if key == "leanp":
                max_abs = float(np.max(np.abs(pick(o, rows) - emu)))
            del o
        line["accuracy_whole_output"] = {
            "estimator": (f"every row i < 512 of every head ({B * Hq * min(512, S)} rows) plus "
                          f"{args.acc_rows} uniform rows beyond, weighted"),
            "leanp_rel_rms_vs_fp64": acc["leanp"], "ablation_rel_rms_vs_fp64": acc["ablation"],
            "leanp_over_ablation": acc["leanp"] / acc["ablation"],
            "leanp_running_max_anchor_rel_rms_vs_fp64": acc["leanp_running_max_anchor"],
            "leanp_running_max_anchor_over_ablation":
                acc["leanp_running_max_anchor"] / acc["ablation"],
            "leanp_max_abs_vs_emulation": max_abs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def extra_legs(torch, fa, wl, dev, stream, timed, peaks, sms, n):
    """BF16 exact softmax on bf16_gqa_h32_8_s16k_d128 and Lean-P on the MLA
    shape (fp8_mla_h16_s32k_dqk192_dv128_outliers), each timed on its own
    inputs (larger than L2) with the clock sampled."""
    legs = {}
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    for key, name in (("bf16_c3", "bf16_gqa_h32_8_s16k_d128"),
                      ("leanp_mla_c5", "fp8_mla_h16_s32k_dqk192_dv128_outliers")):
        case = wl.make_case(name)
        B, Hq, Hkv, S, Dqk, Dv = case.shape
        F = causal_flops(B, Hq, S, Dqk, Dv)
        o = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=dev)
        if key == "bf16_c3":
            q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
                       for a in (case.q, case.k, case.v))
            fn, kind = (lambda: fa.attn_fwd_bf16(q, k, v, out=o)), "bf16"
            peak = peaks["bf16_burst"]
        else:
            q, k, v = (torch.from_numpy(a).to(dev) for a in (case.q, case.k, case.v))
            d = [torch.tensor([x], dtype=torch.float32, device=dev)
                 for x in (case.dq, case.dk, case.dv)]
            fn, kind = (lambda: fa.attn_fwd_fp8(q, k, v, *d, out=o)), "fp8"
            peak = peaks["bf16_burst"] * FP8_OVER_BF16
        clk = ClockSampler(uuid)
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        clk.start()
        time.sleep(0.3)
        ms = timed(fn, n, 0)
        clk = clk.stop()
        tf = F / (ms * 1e-3) / 1e12
        legs[key] = {"workload": name, "value": tf, "unit": "TFLOP/s", "ms_per_step": ms,
                     "steps": n, "peak": peak, "frac": tf / peak,
                     "peak_note": f"{peaks['source']} bf16 burst"
                                  + (f" x {FP8_OVER_BF16} (derived: nominal FP8:BF16)"
                                     if kind == "fp8" else ""),
                     "frac_clock_aware": clock_normalised(tf, kind, peaks, sms,
                                                          clk.get("sm_mhz")),
                     "clocks": clk}
        del q, k, v, o
        torch.cuda.empty_cache()
    legs["leanp_few_heads_split"] = split_leg(torch, fa, wl, dev, peaks, n)
    legs["bf16_few_heads_split"] = split_leg(torch, fa, wl, dev, peaks, n, bf16=True)
    return legs


def split_leg(torch, fa, wl, dev, peaks, n, bf16=False):
    """Few heads (4 heads at 8K keys: 128 work items for the SMs), Lean-P on
    fp8_h4_s8k_d128 or BF16 on bf16_h4_s8k_d128, with the split schedule
    (attn_fwd_full and a workspace) and with whole items.  The inputs fit in
    L2, so a 256 MB buffer is written before every timed call and only the
    call is timed."""
    name = "bf16_h4_s8k_d128" if bf16 else "fp8_h4_s8k_d128"
    variant = fa.ATTN_VARIANT_BF16 if bf16 else fa.ATTN_VARIANT_LEANP
    case = wl.make_case(name)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    F = causal_flops(B, Hq, S, Dqk, Dv)
    if bf16:
        q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
                   for a in (case.q, case.k, case.v))
        d = [None, None, None]
    else:
        q, k, v = (torch.from_numpy(a).to(dev) for a in (case.q, case.k, case.v))
        d = [torch.tensor([x], dtype=torch.float32, device=dev)
             for x in (case.dq, case.dk, case.dv)]
    o = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=dev)
    need = fa.workspace_size(variant, B, Hq, Hkv, S, Dqk, Dv, True)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    n = max(n, 40)  # short calls: enough of them to average out the event resolution
    out = {"workload": name, "unit": "TFLOP/s", "workspace_bytes": need, "steps": n,
           "l2": "256 MB written before every timed call",
           "order": "split and whole calls alternate"}
    fns = {key: (lambda split=split: fa.attn_fwd_full(variant, q, k, v, *d, out=o, split=split,
                                                       workspace=ws if need else None))
           for key, split in (("split", True), ("whole", False))}
    for fn in fns.values():
        for _ in range(5):
            fn()
    total = {key: 0.0 for key in fns}
    for _ in range(n):
        for key, fn in fns.items():
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            total[key] += e0.elapsed_time(e1)
    for key in fns:
        ms = total[key] / n
        out[key] = {"value": F / (ms * 1e-3) / 1e12, "ms_per_step": ms}
    peak = peaks["bf16_burst"] * (1.0 if bf16 else FP8_OVER_BF16)
    out["value"] = out["split"]["value"]
    out["frac"] = out["value"] / peak
    out["speedup_over_whole_items"] = out["split"]["value"] / out["whole"]["value"]
    del q, k, v, o, ws, flush
    torch.cuda.empty_cache()
    return out


# --only PATH: the workload each path is profiled on (headline FP8 shape, the
# BF16 configuration for the BF16 path)
ONLY_PATHS = {"leanp": "fp8_h32_s32k_d128", "exact_fp8": "fp8_h32_s32k_d128",
              "leanp_a3": "fp8_h32_s32k_d128",
              "block_exact": "fp8_h32_s32k_d128", "bf16": "bf16_gqa_h32_8_s16k_d128",
              "leanp_split": "fp8_h4_s8k_d128", "bf16_split": "bf16_h4_s8k_d128",
              "quantize": "quantize_bf16_s32k_h32_d128",
              "quantize_hadamard": "quantize_bf16_s32k_h32_d128"}


def run_only(args):
    """Warm-up and timed launches of one kernel alone (for ncu captures)."""
    import torch

    import fp8_causal_prefill_flash_gb300 as fa
    from fp8_causal_prefill_flash_gb300 import workloads as wl

    fa.build()
    fa.load_library()
    dev = torch.device("cuda", 0)
    name = ONLY_PATHS[args.only]
    if args.only.startswith("quantize"):
        # a bf16 tensor of the headline Q shape (seeded), quantised per tensor
        gen = torch.Generator(device=dev)
        gen.manual_seed(60)
        x = torch.randn((1, args.S or 32768, 32, 128), generator=gen, device=dev).to(torch.bfloat16)
        codes = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        ds = torch.empty(1, dtype=torch.float32, device=dev)
        rot = args.only == "quantize_hadamard"
        fn = lambda: fa.attn_quantize_fp8(x, hadamard=rot, codes=codes, descale=ds)
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        peak = load_peaks()["hbm_gbs"]
        alg = x.numel() * 3 / (ms * 1e-3) / 1e9    # read x once (bf16) + write the codes
        moved = x.numel() * 5 / (ms * 1e-3) / 1e9  # both passes over x + the codes
        print(json.dumps({"path": args.only, "workload": name, "ms_per_step": ms,
                          "gbs_algorithmic": alg, "frac_of_peak_algorithmic": alg / peak,
                          "gbs_moved": moved, "frac_of_peak_moved": moved / peak,
                          "peak_gbs": peak}), flush=True)
        return 0
    case = wl.make_case(name, S=args.S)
    B, Hq, Hkv, S, Dqk, Dv = case.shape
    out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=dev)
    if args.only in ("bf16", "bf16_split"):
        q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
                   for a in (case.q, case.k, case.v))
        if args.only == "bf16":
            fn = lambda: fa.attn_fwd_bf16(q, k, v, out=out)
        else:
            # the split schedule (few work items), its workspace allocated once
            need = fa.workspace_size(fa.ATTN_VARIANT_BF16, B, Hq, Hkv, S, Dqk, Dv, True)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            fn = lambda: fa.attn_fwd_full(fa.ATTN_VARIANT_BF16, q, k, v, out=out,
                                          workspace=ws if need else None)
    else:
        q, k, v = (torch.from_numpy(a).to(dev) for a in (case.q, case.k, case.v))
        d = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (case.dq, case.dk, case.dv)]
        if args.only == "leanp_split":
            # the split schedule (few work items), its workspace allocated once
            need = fa.workspace_size(fa.ATTN_VARIANT_LEANP, B, Hq, Hkv, S, Dqk, Dv, True)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            fn = lambda: fa.attn_fwd_full(fa.ATTN_VARIANT_LEANP, q, k, v, *d, out=out,
                                          workspace=ws if need else None)
        else:
            variant = {"leanp": fa.ATTN_VARIANT_LEANP, "exact_fp8": fa.ATTN_VARIANT_EXACT_FP8,
                       "block_exact": fa.ATTN_VARIANT_BLOCK_EXACT,
                       "leanp_a3": fa.ATTN_VARIANT_LEANP_A3}[args.only]
            fn = lambda: fa.attn_fwd_ex(variant, q, k, v, *d, out=out,
                                        out_dtype=fa.ATTN_OUT_BF16)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"path": args.only, "workload": name, "S": S, "ms_per_step": ms,
                      "tflops_causal": causal_flops(B, Hq, S, Dqk, Dv) / (ms * 1e-3) / 1e12}),
          flush=True)
    return 0


def output_sha256(t):
    """SHA-256 of a device tensor's bytes (the determinism check)."""
    import hashlib

    import torch
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()


def cpu_model():
    """The host CPU's model name as lscpu reports it (else the platform's)."""
    try:
        txt = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in txt.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


_CPU_ONE_CORE = """
import json, sys, time
sys.path.insert(0, {root!r})
import oracle
from fp8_causal_prefill_flash_gb300 import workloads as wl
c = wl.make_case("fp8_h2_s256_d128")
oracle.build()
res = {{}}
for name, fn in (("ref_fp64", oracle.ref_fp64), ("emul_leanp", lambda *a: oracle.emul_leanp(*a)[0])):
    t0 = time.perf_counter()
    fn(c.q, c.k, c.v, c.dq, c.dk, c.dv)
    res[name] = time.perf_counter() - t0
print(json.dumps(res))
"""


def run_cpu_sweep(args):
    """The oracle on the host cores: every configuration on a bounded sample
    of rows (the pass the GPU computes, ref_fp64 and emul_leanp), and the
    2-head 256-key case (fp8_h2_s256_d128) in full on one core (a child process with OMP_NUM_THREADS=1)."""
    from fp8_causal_prefill_flash_gb300 import workloads as wl
    import oracle
    oracle.build()
    model, cores = cpu_model(), cores_used()
    for name, cfg in wl.CONFIGS.items():
        if not cfg["kind"].startswith("fp8"):
            continue
        case = wl.make_case(name)
        B, Hq, Hkv, S, Dqk, Dv = case.shape
        n = min(args.cpu_rows, B * Hq * S)
        rows = sample_rows(S, Hq, n, 7)
        res = {}
        for leg, fn in (("ref_fp64", lambda: oracle.ref_fp64(case.q, case.k, case.v, case.dq,
                                                             case.dk, case.dv, rows=rows)),
                        ("emul_leanp", lambda: oracle.emul_leanp(case.q, case.k, case.v, case.dq,
                                                                 case.dk, case.dv, rows=rows))):
            t0 = time.perf_counter()
            fn()
            dt = time.perf_counter() - t0
            res[leg] = {"s": dt, "gflops": rows_flops(rows, Dqk, Dv) / dt / 1e9}
        print(json.dumps({"workload": name, "rows": int(n), "cores": cores, "cpu_model": model,
                          **res}), flush=True)
    env = dict(os.environ, OMP_NUM_THREADS="1")
    root = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _CPU_ONE_CORE.format(root=root)], env=env,
                       capture_output=True, text=True, timeout=600)
    one = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else {"error": r.stderr[-300:]}
    print(json.dumps({"workload": "fp8_h2_s256_d128", "rows": "all", "cores": 1,
                      "cpu_model": model, "seconds": one}), flush=True)
    return 0


def run_sweep(args):
    """One JSON line per configuration of the workload table (measurement
    notes, not the bench line): each path's time, causal TFLOP/s and fraction
    of the matching measured peak; for the short case also HBM GB/s."""
    import torch

    import fp8_causal_prefill_flash_gb300 as fa
    from fp8_causal_prefill_flash_gb300 import workloads as wl

    fa.build()
    fa.load_library()
    peaks = load_peaks()
    dev = torch.device("cuda", 0)
    for name, cfg in wl.CONFIGS.items():
        case = wl.make_case(name)
        B, Hq, Hkv, S, Dqk, Dv = case.shape
        F = causal_flops(B, Hq, S, Dqk, Dv)
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=dev)
        if cfg["kind"].startswith("fp8"):
            q, k, v = (torch.from_numpy(a).to(dev) for a in (case.q, case.k, case.v))
            d = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (case.dq, case.dk, case.dv)]
            paths = {"leanp": lambda: fa.attn_fwd_fp8(q, k, v, *d, out=out),
                     # with the split schedule where the problem has few work items
                     "leanp_split": lambda: fa.attn_fwd_full(fa.ATTN_VARIANT_LEANP, q, k, v, *d,
                                                             out=out),
                     "exact_fp8_ablation": lambda: fa.attn_fwd_fp8_exact(q, k, v, *d, out=out),
                     # Lean-P's block scale and rounded sum, exponential for the code
                     "block_exact": lambda: fa.attn_fwd_ex(fa.ATTN_VARIANT_BLOCK_EXACT, q, k, v,
                                                           *d, out=out,
                                                           out_dtype=fa.ATTN_OUT_BF16),
                     "leanp_running_max_anchor": lambda: fa.attn_fwd_ex(
                         fa.ATTN_VARIANT_LEANP_A3, q, k, v, *d, out=out,
                         out_dtype=fa.ATTN_OUT_BF16)}
            peak = peaks["bf16_burst"] * FP8_OVER_BF16
            in_bytes = (case.q.nbytes + case.k.nbytes + case.v.nbytes)
        else:
            q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
                       for a in (case.q, case.k, case.v))
            paths = {"bf16": lambda: fa.attn_fwd_bf16(q, k, v, out=out)}
            peak = peaks["bf16_burst"]
            in_bytes = 2 * (case.q.size + case.k.size + case.v.size)
        io_bytes = in_bytes + out.numel() * 2
        for path, fn in paths.items():
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            n = args.steps
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            ev[0].record()
            for i in range(n):
                fn()
                ev[i + 1].record()
            torch.cuda.synchronize()
            per = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
            ms = ev[0].elapsed_time(ev[n]) / n
            tf = F / (ms * 1e-3) / 1e12
            print(json.dumps({"workload": name, "path": path, "ms": ms, "tflops_causal": tf,
                              "ms_median": statistics.median(per), "ms_min": min(per),
                              "tflops_square_formula": 2 * tf, "peak": peak,
                              "frac_of_peak": tf / peak, "hbm_gbs": io_bytes / (ms * 1e-3) / 1e9,
                              "peak_source": peaks["source"], "iterations": n}), flush=True)
        del q, k, v, out
        torch.cuda.empty_cache()
    # non-causal calls (flash_attn_func causal=False): every row sees all S keys
    for name in ("fp8_gqa_h32_8_s16k_d128_outliers", "bf16_gqa_h32_8_s16k_d128"):
        case = wl.make_case(name)
        B, Hq, Hkv, S, Dqk, Dv = case.shape
        F = square_flops(B, Hq, S, Dqk, Dv)
        if name.startswith("fp8"):
            q, k, v = (torch.from_numpy(a).to(dev) for a in (case.q, case.k, case.v))
            d = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (case.dq, case.dk, case.dv)]
            fn = lambda: fa.attn_fwd_full(fa.ATTN_VARIANT_LEANP, q, k, v, *d, causal=False)
            path, peak = "leanp_noncausal", peaks["bf16_burst"] * FP8_OVER_BF16
        else:
            q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
                       for a in (case.q, case.k, case.v))
            fn = lambda: fa.attn_fwd_full(fa.ATTN_VARIANT_BF16, q, k, v, causal=False)
            path, peak = "bf16_noncausal", peaks["bf16_burst"]
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        n = args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        tf = F / (ms * 1e-3) / 1e12
        print(json.dumps({"workload": name, "path": path, "ms": ms, "tflops": tf,
                          "flop_count": "2*B*Hq*S^2*(Dqk+Dv) (every pair computed)", "peak": peak,
                          "frac_of_peak": tf / peak, "iterations": n}), flush=True)
        del q, k, v
        torch.cuda.empty_cache()
    # the Q/K quantise pre-pass (optionally Hadamard-rotated) on a bf16 tensor
    # of the headline Q shape: HBM-bound, reads x twice, writes 1 byte/element
    x = torch.randn((1, 32768, 32, 128), device=dev).to(torch.bfloat16)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    ds = torch.empty(1, dtype=torch.float32, device=dev)
    for rot in (False, True):
        fn = lambda: fa.attn_quantize_fp8(x, hadamard=rot, codes=codes, descale=ds)
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        n = args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        alg = x.numel() * 3  # read x once (bf16) + write the codes
        moved = x.numel() * 5  # the two passes over x + the codes
        print(json.dumps({"workload": "quantize_bf16_s32k_h32_d128", "path":
                          "hadamard" if rot else "plain", "ms": ms,
                          "gbs_algorithmic": alg / (ms * 1e-3) / 1e9,
                          "gbs_moved": moved / (ms * 1e-3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
                          "frac_of_peak_algorithmic": alg / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "frac_of_peak_moved": moved / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "iterations": n}), flush=True)
    return 0


def run_clock_study(args):
    """Sustained runs (about `--study-seconds` each) of Lean-P and the ablation
    on inputs of different statistics, with the SM clock, the power and the
    energy sampled throughout: one JSON line per (input, path)."""
    import torch

    import fp8_causal_prefill_flash_gb300 as fa
    from fp8_causal_prefill_flash_gb300 import workloads as wl

    fa.build()
    fa.load_library()
    dev = torch.device("cuda", 0)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    meter = EnergyMeter(uuid)
    for name in ("fp8_h32_s32k_d128", "fp8_gqa_h32_8_s16k_d128_outliers", "fp8_sink_h8_s8k_d128"):
        case = wl.make_case(name)
        B, Hq, Hkv, S, Dqk, Dv = case.shape
        F = causal_flops(B, Hq, S, Dqk, Dv)
        q, k, v = (torch.from_numpy(a).to(dev) for a in (case.q, case.k, case.v))
        d = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (case.dq, case.dk, case.dv)]
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=dev)
        for path, fn in (("leanp", lambda: fa.attn_fwd_fp8(q, k, v, *d, out=out)),
                         ("exact_fp8_ablation", lambda: fa.attn_fwd_fp8_exact(q, k, v, *d, out=out))):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            n = max(1, int(args.study_seconds * 1000.0 / max(e0.elapsed_time(e1), 1e-3)))
            clocks = ClockSampler(uuid)
            clocks.start()
            time.sleep(0.3)
            mj0 = meter.read_mj()
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
            mj1 = meter.read_mj()
            clk = clocks.stop()
            ms = e0.elapsed_time(e1) / n
            print(json.dumps({"workload": name, "path": path, "calls": n, "ms": ms,
                              "tflops_causal": F / (ms * 1e-3) / 1e12, "clocks": clk,
                              "energy": energy_report(mj0, mj1, F * n)}), flush=True)
        del q, k, v, out
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=8192,
                    help="oracle rows timed for cpu_baseline (about 10-30 s of CPU work)")
    ap.add_argument("--acc-rows", type=int, default=2048,
                    help="rows beyond the first 512 of each head compared with fp64 attention "
                         "for the accuracy report")
    ap.add_argument("--ref-row-budget", type=int, default=8192,
                    help="oracle rows over the whole reference run")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the BF16 and MLA legs of the bench line")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of back-to-back calls for the sustained leg")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the same kernel")
    ap.add_argument("--workload", default=WORKLOAD, help="configuration name (profiling)")
    ap.add_argument("--S", type=int, default=None, help="override the sequence length (profiling)")
    ap.add_argument("--only", choices=list(ONLY_PATHS), default=None,
                    help="time one kernel alone on its workload (profiling)")
    ap.add_argument("--cpu-sweep", action="store_true",
                    help="time the oracle on every configuration (bounded samples) and the "
                         "2-head 256-key case in full on one core")
    ap.add_argument("--sweep", action="store_true",
                    help="time every path on every configuration, one JSON line each")
    ap.add_argument("--clock-study", action="store_true",
                    help="sustained runs per input distribution: SM clock, power, energy")
    ap.add_argument("--study-seconds", type=float, default=3.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: WORLD_SIZE={world} but --gpus={args.gpus}", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        return run_sweep(args)
    if args.only:
        return run_only(args)
    if args.cpu_sweep:
        return run_cpu_sweep(args)
    if args.clock_study:
        return run_clock_study(args)
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
