#!/usr/bin/env python
"""Benchmark of the GB300 dense multiply-accumulate path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--headline-only]

One step is one D = A*B + C call (operand staging, the MMA K loop and the
+C epilogue) on the headline workload: the INT8 -> INT32 GEMM with
M = N = K = 4096 (A row-major, B column-major, C/D int32), seeded synthetic
inputs already resident in HBM.  Several input sets are rotated so that the
bytes touched between two uses of a set exceed the 129 MB L2.  Rank 0 prints
one JSON line: whole-job TOP/s (all ranks' operations / max-over-ranks time),
the dominant kernel's roofline (per-launch CUDA-event durations recorded by
the library on the launching stream), an end-to-end figure through host
buffers, SM clocks sampled during the timed region, the CPU oracle timed on
a bounded sample, and a per-dtype table of the other workloads.

Multi-GPU: every rank runs its own independent problem (weak scaling, no
data-path collective); torch.distributed is used only for the barrier and
the max-over-ranks time.

``--impl reference`` times the CPU oracle (the plain C reference
implementation) on the host cores instead, on a bounded sample of the same
workload per step; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (TOP/s int8) and % of GB300 dense tensor peak per dtype"
HEADLINE = "gemm_i8_4096"
L2_BYTES = 129 * 1024 * 1024
MAX_SET_BYTES = 8 << 30  # device memory cap for the rotating input sets
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
GB300_SMS = 152
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_FP64_TFLOPS = 1.25
NOMINAL_HBM_GBS = 7900.0
# dense BF16 tensor-core rate per SM per clock (128 x 256 x 16 x 2 flops
# per 128-cycle MMA), for the nominal denominators reported beside the
# measured ones
BF16_FLOP_PER_SM_CLK = 8192.0

# DRAM bytes per launch of each dominant kernel from one ncu capture, keyed
# by the SHA-256 of the kernel source's code (comments and whitespace
# removed, see source_sha) at capture time: changed code makes the figure
# stale, and it is then reported as null.
NCU_TRAFFIC: dict = {
    # one ncu capture per workload (dram__bytes_read.sum and
    # dram__bytes_write.sum of one launch after the warm-up launches)
    "gemm_i8_4096": {"sha": "2b87d5f638b5e79f", "bytes": 157382144 + 36154880},
    "gemm_u8_4096_clamp": {"sha": "2b87d5f638b5e79f", "bytes": 156731904 + 36141568},
    "gemm_bf16_8192": {"sha": "2b87d5f638b5e79f", "bytes": 1632362496 + 258151424},
    "gemm_bf16_skinny_16384x128x4096": {"sha": "2b87d5f638b5e79f",
                                        "bytes": 143721472 + 2897408},
    "batched_bf16_16x16x16_b262144_g4_abid1": {"sha": "e9a765212730005e",
                                               "bytes": 436228352 + 225458688},
    "batched_bf16_128x128x128_b8192_g4_abid1": {"sha": "2b87d5f638b5e79f",
                                                "bytes": 904013824 + 490111488},
    "batched_bf16_64x64x64_b16384_g4_abid1": {"sha": "5e2d44fac663ee87",
                                              "bytes": 436244736 + 226981376},
    "batched_bf16_32x32x32_b65536_g4_abid1": {"sha": "7c13c61cea575839",
                                              "bytes": 436254208 + 214824960},
    "batched_i8_32x32x32_b65536_g4_abid1": {"sha": "7c13c61cea575839",
                                            "bytes": 352359168 + 213289472},
    "gemm_f64_4096_rowB": {"sha": "b947734a2fa7d71b", "bytes": 3657537000 + 130594048},
    "gemm_bf16_acc16_8192": {"sha": "2b87d5f638b5e79f", "bytes": 1482969600 + 128653824},
    "gemm_f16_256": {"sha": "2b87d5f638b5e79f", "bytes": 580096 + 0},
    "gemm_bf16_deepk_1024x1024x32768": {"sha": "b39718a8ce94b2da",
                                        "bytes": 138511104 + 3083008},
}


# --------------------------------------------------------------- helpers

def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def source_sha(rel):
    """SHA-256 (16 hex digits) of a kernel source with its comments and
    whitespace removed: what the compiler sees, so that editing a comment
    does not disown a traffic figure taken from the same code."""
    try:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
    except OSError:
        return None
    code = "".join(_COMMENT.sub(" ", text).split())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


class Dist:
    """Rank bookkeeping; torch.distributed only when WORLD_SIZE > 1."""

    def __init__(self, want_cuda: bool):
        self.rank = _env_int("RANK", 0)
        self.world = _env_int("WORLD_SIZE", 1)
        self.local_rank = _env_int("LOCAL_RANK", 0)
        self.pg = None
        if self.world > 1:
            import torch.distributed as td
            backend = "nccl" if want_cuda else "gloo"
            td.init_process_group(backend=backend)
            self.pg = td

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = torch.device("cuda", self.local_rank) if torch.cuda.is_available() \
            and self.pg.get_backend() == "nccl" else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def whole_job(units_per_step: float, steps: int, world: int, seconds: float):
    """Aggregate throughput: all ranks' units over the max-over-ranks time."""
    return units_per_step * steps * world / seconds


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []  # (host time, fields...)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win:
            win = [p for (_, p) in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        pw = [num(p[3]) for p in win if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4)
                          if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(win)}


# ------------------------------------------------------------ workloads

def workload_meta(name):
    from mixed_precision_dense_02_gb300 import synth
    w = dict(synth.WORKLOADS[name])
    if w["kind"] == "gemm":
        ops = 2.0 * w["M"] * w["N"] * w["K"]
        isz = {"f16": 2, "bf16": 2, "i8": 1, "f64": 8}[w["dtype_in"]]
        osz = 8 if w["dtype_in"] == "f64" else (2 if w.get("acc16") else 4)
        nbytes = (w["M"] * w["K"] + w["N"] * w["K"]) * isz + 2 * w["M"] * w["N"] * osz
    else:
        ops = 2.0 * w["batch"] * w["M"] * w["N"] * w["K"]
        isz = {"f16": 2, "bf16": 2, "i8": 1}[w["dtype_in"]]
        tile_in = w["M"] * w["K"] * isz
        nbytes = (w["batch"] // w["group"]) * tile_in + w["batch"] * (
            w["N"] * w["K"] * isz + 2 * w["M"] * w["N"] * 4)
    w["ops"] = ops
    w["algorithmic_bytes"] = nbytes
    w["unit"] = "TOP/s" if w["dtype_in"] == "i8" else "TFLOP/s"
    return w


# Issue-rate probes of this run (measure_probes): name -> record.
_PROBES: dict = {}
# (name, kind code of mma_peak_probe, unit, largest iteration count)
PROBE_KINDS = (("tc_f16", 1, "TFLOP/s", 1 << 21),
               ("dmma_f64", 2, "TFLOP/s", 1 << 40),
               ("imma_s8", 3, "TOP/s", 1 << 40),
               ("dfma_f64", 4, "TFLOP/s", 1 << 40))


def measure_probes(torch, target_ms=20.0, reps=3):
    """Per-pipe issue-rate probes (mma_peak_probe: every SM issues
    independent back-to-back instructions of one kind): operations per
    launch / CUDA-event launch time, best and median of `reps` launches of
    about `target_ms`.  Fills _PROBES and returns it."""
    from mixed_precision_dense_02_gb300 import binding
    stream = torch.cuda.current_stream()

    def launch(kind, n):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        st, ops = binding.mma_peak_probe(kind, n, stream.cuda_stream)
        ev1.record(stream)
        ev1.synchronize()
        if st != 0:
            raise RuntimeError(f"mma_peak_probe({kind}) returned {binding.STATUS.get(st, st)}")
        return ev0.elapsed_time(ev1), ops

    for name, kind, unit, cap in PROBE_KINDS:
        n = 16
        ms, _ = launch(kind, n)
        while ms < 2.0 and n < cap:
            n = min(cap, n * 8)
            ms, _ = launch(kind, n)
        n = int(min(cap, max(1, n * target_ms / max(ms, 1e-3))))
        times, ops = [], 0.0
        for _ in range(reps):
            ms, ops = launch(kind, n)
            times.append(ms)
        best = min(times)
        _PROBES[name] = {"rate": ops / (best * 1e-3) / 1e12, "unit": unit,
                         "rate_median": ops / (statistics.median(times) * 1e-3) / 1e12,
                         "iterations": n, "ms_best": best, "ops_per_launch": ops}
    binding.device_status()
    return _PROBES


def roofline_bound(name, w):
    """(bound, unit, peak, peak_note) of the workload's dominant kernel."""
    peaks, src = load_peaks()
    if w["ops"] < 1e9 and w["kind"] == "gemm":
        # a few 128-row tiles: pipeline latency, not a pipe, sets the time
        return ("tensor", "TFLOP/s", peaks["bf16_tflops"],
                f"bf16_tflops (burst) of {src}; launch/latency-bound problem "
                "(about 9 us of pipeline latency), no percentage target")
    if w["kind"] == "batched" or "skinny" in name:
        return "hbm", "GB/s", peaks["hbm_gbs"], f"hbm_gbs of {src}"
    if w["dtype_in"] == "f64":
        if "dmma_f64" in _PROBES:
            p = _PROBES["dmma_f64"]["rate"]
            return ("tensor", "TFLOP/s", p, "measured DMMA issue-rate probe in this "
                    f"run (mma_peak_probe, m8n8k4 FP64 on every SM): {p:.3f} TFLOP/s")
        p = peaks["bf16_tflops"] * NOMINAL_FP64_TFLOPS / NOMINAL_BF16_TFLOPS
        return "tensor", "TFLOP/s", p, f"bf16_tflops of {src} x nominal fp64/bf16 (1.25/2250)"
    return "tensor", "TFLOP/s", peaks["bf16_tflops"], f"bf16_tflops (burst) of {src}"


def kernel_source(w):
    if w["kind"] == "batched":
        if (w["M"], w["N"], w["K"]) == (16, 16, 16):
            return "mixed_precision_dense_02_gb300/csrc/batched16.cu"
        macs = w["M"] * w["N"] * w["K"]
        if w["dtype_in"] == "i8":
            if macs <= 128 ** 3 and w["M"] % 16 == 0 and w["N"] % 16 == 0 \
                    and w["K"] % 16 == 0:
                return "mixed_precision_dense_02_gb300/csrc/batched_mma.cu"
            return "mixed_precision_dense_02_gb300/csrc/gemm_tc.cu"
        if w["dtype_in"] == "f64":
            return "mixed_precision_dense_02_gb300/csrc/gemm_f64.cu"
        if all(w[d] % 64 == 0 for d in "MNK") and macs <= 1 << 20:
            return "mixed_precision_dense_02_gb300/csrc/batched_tile.cu"
        if macs <= 96 * 96 * 64 and all(w[d] % 16 == 0 for d in "MNK"):
            return "mixed_precision_dense_02_gb300/csrc/batched_mma.cu"
        return "mixed_precision_dense_02_gb300/csrc/gemm_tc.cu"
    if w["dtype_in"] == "i8" and not i8_on_tensor_pipe(w):
        return "mixed_precision_dense_02_gb300/csrc/gemm_i8.cu"
    if stream_k_applies(w):
        return "mixed_precision_dense_02_gb300/csrc/gemm_sk.cu"
    return {"f16": "mixed_precision_dense_02_gb300/csrc/gemm_tc.cu",
            "bf16": "mixed_precision_dense_02_gb300/csrc/gemm_tc.cu",
            "i8": "mixed_precision_dense_02_gb300/csrc/gemm_tc.cu",
            "f64": "mixed_precision_dense_02_gb300/csrc/gemm_f64.cu"}[w["dtype_in"]]


def stream_k_applies(w, sms=GB300_SMS):
    """FP16/BF16 -> FP32 products with column-major B, fewer than half as
    many 128 x 128 output tiles as SMs, at least 8 K steps of 64 and two per
    SM, and either at most a quarter as many tiles as SMs or at least 128 K
    steps: the library splits the tiles' K steps over every SM (gemm_sk.cu,
    the rule of gemm_sk_fits)."""
    if w["kind"] != "gemm" or w["dtype_in"] not in ("f16", "bf16"):
        return False
    if w.get("acc16") or w.get("b_layout", "col") != "col":
        return False
    tiles = -(-w["M"] // 128) * -(-w["N"] // 128)
    nk = -(-w["K"] // 64)
    return (2 * tiles < sms and nk >= 8 and tiles * nk >= 2 * sms
            and (4 * tiles <= sms or nk >= 128))


def i8_plain(w):
    """Signed x signed 8-bit inputs without saturation (mma_gemm's INT8)."""
    return w.get("a_signed", True) and w.get("b_signed", True) and not w.get("clamp")


def i8_on_tensor_pipe(w):
    """INT8 problems with M*N*K >= 2^24, and every unsigned, mixed-sign or
    saturating one, run on the tcgen05 BF16 pipe."""
    return not i8_plain(w) or float(w["M"]) * w["N"] * w["K"] >= 2.0 ** 24


def launches_per_call(w):
    """Kernels one library call launches: the exact-INT8 path adds a
    conversion kernel before the GEMM; every other path launches one."""
    if w["kind"] == "gemm" and w["dtype_in"] == "i8" and i8_on_tensor_pipe(w):
        return 2
    return 1


class GpuWorkload:
    """Device-resident input sets of one workload and its step function."""

    def __init__(self, name, seed=0):
        import numpy as np
        import torch
        from mixed_precision_dense_02_gb300 import binding, synth
        self.name = name
        self.w = workload_meta(name)
        self.binding = binding
        self.dev = torch.device("cuda", torch.cuda.current_device())
        w = self.w
        if w["kind"] == "gemm":
            g = synth.workload_gemm_inputs(name, seed)
            host = [g.A, g.B, g.C]
            self.b_layout = g.b_layout
            self.acc16 = w.get("acc16", False)
        else:
            bi = synth.batched_inputs(name, w["dtype_in"], w["batch"], w["M"],
                                      w["N"], w["K"], group=w["group"],
                                      abid=w["abid"], dist=w.get("dist", "uniform"),
                                      seed=seed)
            host = [bi.A, bi.B, bi.C]
        self.dtype_in = w["dtype_in"]
        self.host = [self._pinned(x) for x in host]
        self.acc = "same" if getattr(self, "acc16", False) else None
        # A, B, C and D of one set; rotate enough sets that more than twice
        # the L2 capacity is touched between two uses of the same set
        per_set = (sum(t.numel() * t.element_size() for t in self.host)
                   + self.host[2].numel() * self.host[2].element_size())
        self.per_set_bytes = per_set
        self.nsets = max(1, min(max(1, MAX_SET_BYTES // per_set),
                                math.ceil(2 * L2_BYTES / per_set) + 1))
        self.l2_note = (f"{self.nsets} rotating input sets of {per_set / 1e6:.1f} MB"
                        f" ({self.nsets * per_set / 1e6:.0f} MB > 2 x L2 between reuses of a set)")
        self.sets = []
        for _ in range(self.nsets):
            A, B, C = (self._dev(t) for t in self.host)
            D = torch.empty_like(C)
            self.sets.append((A, B, C, D))
        self.host_D = torch.empty(self.host[2].shape, dtype=self.sets[0][3].dtype,
                                  pin_memory=True)
        self.launches_per_step = launches_per_call(self.w)

    def _pinned(self, x):
        import numpy as np
        import torch
        if x.dtype == np.uint16:
            x = x.view(np.int16)
        t = torch.from_numpy(np.ascontiguousarray(x))
        return t.pin_memory()

    def _dev(self, t):
        import torch
        d = t.to(self.dev, non_blocking=False)
        if d.dtype == torch.int16:
            d = d.view(torch.bfloat16 if self.dtype_in == "bf16" else torch.float16)
        return d

    def call(self, A, B, C, D):
        w = self.w
        if w["kind"] == "gemm" and w["dtype_in"] == "i8" and not i8_plain(w):
            self.binding.gemm_i8_ex(A, B, C, D, clamp=w.get("clamp", False),
                                    b_layout=self.b_layout)
        elif w["kind"] == "gemm":
            self.binding.gemm_ex(A, B, C, D, b_layout=self.b_layout, acc=self.acc)
        else:
            self.binding.gemm_batched(A, B, C, D, group=w["group"], abid=w["abid"])

    def step(self, i):
        self.call(*self.sets[i % self.nsets])

    def e2e_setup(self):
        """Two CUDA streams, each with its own device input set and pinned
        result buffer: consecutive end-to-end steps alternate between them,
        so one step's uploads overlap the previous step's compute and
        download (every step still moves all of its own bytes)."""
        import torch
        while len(self.sets) < 2:
            A, B, C = (self._dev(t) for t in self.host)
            self.sets.append((A, B, C, torch.empty_like(C)))
        self.e2e_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        self.host_Ds = [self.host_D,
                        torch.empty_like(self.host_D).pin_memory()]

    def e2e_step(self, i):
        """Host -> device inputs, the call, device -> host result (step i,
        on stream i % 2)."""
        import torch
        k = i % 2
        A, B, C, D = self.sets[k]
        with torch.cuda.stream(self.e2e_streams[k]):
            for dst, src in zip((A, B, C), self.host):
                dst.view(src.dtype).copy_(src, non_blocking=True)
            self.call(A, B, C, D)
            self.host_Ds[k].copy_(D, non_blocking=True)

    @property
    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host)

    @property
    def d2h_bytes(self):
        return self.host_D.numel() * self.host_D.element_size()


def time_steps(torch, dist, fn, steps, warmup):
    """Warm up, then time exactly `steps` calls between barriers + syncs."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    start.record()
    for i in range(steps):
        fn(warmup + i)
    stop.record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    dist.barrier()
    ms = start.elapsed_time(stop)
    return ms / 1e3, t_host0, t_host1


def time_e2e(torch, dist, wl, steps, warmup):
    """time_steps for the two-stream end-to-end loop: the timed region runs
    from an event on the current stream, which both step streams wait for,
    to an event recorded after the current stream has waited for both."""
    wl.e2e_setup()
    cur = torch.cuda.current_stream()
    for i in range(warmup):
        wl.e2e_step(i)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(cur)
    for s in wl.e2e_streams:
        s.wait_stream(cur)
    for i in range(steps):
        wl.e2e_step(warmup + i)
    for s in wl.e2e_streams:
        cur.wait_stream(s)
    stop.record(cur)
    torch.cuda.synchronize()
    dist.barrier()
    return start.elapsed_time(stop) / 1e3


def measure_workload(torch, dist, name, steps, warmup, with_e2e, sustain_s=0.0):
    wl = GpuWorkload(name)
    w = wl.w
    b = wl.binding
    # Roofline pass: the library records one CUDA event pair on the
    # launching stream around the dominant kernel of each call.  It runs
    # right after warm-up and before the timed pass, at the same thermal
    # state; it is kept out of the timed pass because an event between the
    # INT8 widening kernel and the GEMM would defeat the GEMM's
    # programmatic-dependent launch.
    for i in range(warmup):
        wl.step(i)
    b.profile_begin()
    time_steps(torch, dist, wl.step, steps, 0)
    launch_ms = b.profile_end()
    b.device_status()
    # Throughput pass (timed): K steps between barriers and syncs.
    secs, t0, t1 = time_steps(torch, dist, wl.step, steps, 0)
    secs_max = dist.max(secs)
    if sustain_s and t1 - t0 < sustain_s:
        # The timed region is shorter than the clock sampling needs: keep the
        # same step loop running (untimed) so the sampled window, which
        # starts at the timed region, covers a sustained load.
        i = 0
        while time.time() - t0 < sustain_s:
            for _ in range(16):
                wl.step(i)
                i += 1
            torch.cuda.synchronize()
        t1 = time.time()
    value = whole_job(w["ops"], steps, dist.world, secs_max) / 1e12
    mean_ms = statistics.fmean(launch_ms) if launch_ms else float("nan")
    bound, unit, peak, note = roofline_bound(name, w)
    if unit == "GB/s":
        achieved = w["algorithmic_bytes"] / (mean_ms * 1e-3) / 1e9
    else:
        achieved = w["ops"] / (mean_ms * 1e-3) / 1e12
    src = kernel_source(w)
    traffic = None
    rec = NCU_TRAFFIC.get(name)
    if rec and rec.get("sha") == source_sha(src):
        traffic = rec["bytes"]
    res = {
        "value": value, "unit": w["unit"], "ms_per_step": secs_max * 1e3 / steps,
        "steps": steps, "warmup": warmup, "l2": wl.l2_note,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "traffic": traffic,
                     "peak_source": note, "kernel_launches_timed": len(launch_ms),
                     "kernel_ms_mean": mean_ms,
                     "kernel_ms_median": (statistics.median(launch_ms)
                                          if launch_ms else None),
                     "kernel_ms_best": min(launch_ms) if launch_ms else None,
                     "algorithmic_bytes_per_launch": w["algorithmic_bytes"],
                     "ops_per_launch": w["ops"]},
        "pct_of_bf16_peak": None, "host_window": (t0, t1),
        "gpu_launches": steps * wl.launches_per_step,
    }
    if w["kind"] == "gemm" and w["dtype_in"] != "f64":
        res["pct_of_bf16_peak"] = 100.0 * value / load_peaks()[0]["bf16_tflops"]
    if with_e2e:
        e_steps = max(3, min(steps, 20))
        secs_e = time_e2e(torch, dist, wl, e_steps, min(warmup, 3))
        secs_e = dist.max(secs_e)
        res["e2e"] = {"value": whole_job(w["ops"], e_steps, dist.world, secs_e) / 1e12,
                      "unit": w["unit"], "h2d_bytes_per_step": wl.h2d_bytes,
                      "d2h_bytes_per_step": wl.d2h_bytes, "steps": e_steps}
    del wl
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------- CPU oracle

def oracle_sample_step(name, rows, seed=0):
    """One oracle run on the first `rows` rows (or batch entries) of the
    workload; returns (seconds, operations)."""
    import numpy as np
    import oracle
    w = workload_meta(name)
    if w["kind"] == "gemm":
        g = _sample_inputs_cache(name, seed)
        A = np.ascontiguousarray(g.A[:rows])
        C = np.ascontiguousarray(g.C[:rows])
        t = time.perf_counter()
        if g.dtype_in == "i8" and not i8_plain(w):
            oracle.gemm_i8_ex(A, g.B, C, clamp=w.get("clamp", False),
                              b_layout=g.b_layout)
        else:
            fn = oracle.gemm_acc16 if w.get("acc16") else oracle.gemm
            fn(g.dtype_in, A, g.B, C, b_layout=g.b_layout)
        dt = time.perf_counter() - t
        return dt, 2.0 * rows * w["N"] * w["K"]
    bi = _sample_inputs_cache(name, seed)
    n = rows - rows % w["group"] or w["group"]
    t = time.perf_counter()
    oracle.gemm_batched(bi.dtype_in, bi.A[:n], bi.B[:n], bi.C[:n],
                        group=bi.group, abid=bi.abid)
    dt = time.perf_counter() - t
    return dt, 2.0 * n * w["M"] * w["N"] * w["K"]


_INPUT_CACHE = {}


def _sample_inputs_cache(name, seed):
    from mixed_precision_dense_02_gb300 import synth
    if name not in _INPUT_CACHE:
        w = synth.WORKLOADS[name]
        if w["kind"] == "gemm":
            _INPUT_CACHE[name] = synth.workload_gemm_inputs(name, seed)
        else:
            _INPUT_CACHE[name] = synth.batched_inputs(
                name, w["dtype_in"], w["batch"], w["M"], w["N"], w["K"],
                group=w["group"], abid=w["abid"], dist=w.get("dist", "uniform"),
                seed=seed)
    return _INPUT_CACHE[name]


def calibrate_rows(name, target_s):
    """Rows (or batch entries) of the workload that take about target_s."""
    w = workload_meta(name)
    total = w["M"] if w["kind"] == "gemm" else w["batch"]
    rows = 4 if w["kind"] == "gemm" else 4096
    dt, _ = oracle_sample_step(name, rows)
    while dt < 0.2 and rows < total:
        rows = min(total, rows * 4)
        dt, _ = oracle_sample_step(name, rows)
    rows = int(min(total, max(1, rows * target_s / max(dt, 1e-6))))
    return rows


def cpu_baseline(name, target_s=10.0):
    import oracle
    rows = calibrate_rows(name, target_s)
    dt, ops = oracle_sample_step(name, rows)
    w = workload_meta(name)
    what = "rows of A (with all of B, C)" if w["kind"] == "gemm" else "batch entries"
    return {"value": ops / dt / 1e12, "unit": w["unit"],
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {rows} {what} of {name}; {dt:.1f} s, {ops:.3e} ops"}


# ------------------------------------------------------------------ main

def run_reference(args, dist):
    if dist.rank != 0:
        return 0
    import oracle
    name = args.workload
    w = workload_meta(name)
    per_step = max(0.2, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    rows = calibrate_rows(name, per_step)
    for _ in range(args.warmup):
        oracle_sample_step(name, rows)
    tot_s, tot_ops = 0.0, 0.0
    for _ in range(args.steps):
        dt, ops = oracle_sample_step(name, rows)
        tot_s += dt
        tot_ops += ops
    value = tot_ops / tot_s / 1e12
    what = "rows of A (with all of B, C)" if w["kind"] == "gemm" else "batch entries"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": w["unit"],
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": _dtype_tag(w),
        "data": "synthetic", "config": _config(name, w, "n/a (host CPU)"),
        "cpu_baseline": {"value": value, "unit": w["unit"],
                         "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"first {rows} {what} of {name} per step"},
        "e2e": {"value": value, "unit": w["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def add_nominal(roof, sms, clk):
    """Context denominators beside the measured peak (frac stays against the
    measured one): for the BF16 tensor pipe SMs x 8192 flop/clk x the
    maximum SM clock and x the median SM clock of the row's own timed
    region, and the tcgen05 issue-rate probe of this run; for HBM the
    nominal HBM3e bandwidth.  FP64 (DMMA pipe, against its own probe) gets
    none."""
    roof["sm_mhz_run"] = clk.get("sm_mhz")
    if roof["unit"] == "GB/s":
        roof["nominal_peak"] = NOMINAL_HBM_GBS
        roof["frac_of_nominal"] = roof["achieved"] / NOMINAL_HBM_GBS
        return
    if "DMMA" in roof.get("peak_source", "") or "fp64" in roof.get("peak_source", ""):
        return
    if "tc_f16" in _PROBES:
        roof["probe_peak"] = _PROBES["tc_f16"]["rate"]
        roof["frac_of_probe"] = roof["achieved"] / _PROBES["tc_f16"]["rate"]
    mx, med = clk.get("sm_max_mhz"), clk.get("sm_mhz")
    if mx:
        roof["nominal_peak_max_clock"] = sms * BF16_FLOP_PER_SM_CLK * mx * 1e6 / 1e12
    if med:
        nom = sms * BF16_FLOP_PER_SM_CLK * med * 1e6 / 1e12
        roof["nominal_peak_run_clock"] = nom
        roof["frac_of_nominal_run_clock"] = roof["achieved"] / nom


def _dtype_tag(w):
    if w["dtype_in"] == "i8":
        sa, sb = w.get("a_signed", True), w.get("b_signed", True)
        return "i8" if sa and sb else ("u8" if not (sa or sb) else "u8/i8")
    return {"f16": "f16", "bf16": "bf16", "f64": "f64"}[w["dtype_in"]]


def _config(name, w, l2):
    cfg = {"workload": name, "l2": l2}
    for k in ("M", "N", "K", "batch", "group", "abid", "dtype_in", "a_signed",
              "b_signed", "clamp"):
        if k in w:
            cfg[k] = w[k]
    if w["kind"] == "gemm":
        cfg["layout"] = ("A row-major, B " + ("row" if w.get("b_layout") == "row"
                         else "column") + "-major, C/D row-major")
    return cfg


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--peaks", action="store_true",
                    help="run only the per-pipe issue-rate probes and print them")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        dist = Dist(want_cuda=False)
        try:
            return run_reference(args, dist)
        finally:
            dist.close()

    import torch
    torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
    dist = Dist(want_cuda=True)
    import mixed_precision_dense_02_gb300 as pkg
    pkg.load()
    w = workload_meta(args.workload)

    clocks = ClockSampler(dist.local_rank)
    clocks.start()
    time.sleep(0.5)
    # per-pipe issue-rate probes (a second or so): the FP64 row's peak and
    # context for the tensor rows
    t0p = time.time()
    probes = measure_probes(torch)
    probe_clk = clocks.summary(t0p, time.time())
    if args.peaks:
        clocks.stop()
        if dist.rank == 0:
            print(json.dumps({"probes": probes, "clocks": probe_clk,
                              "n_sms": torch.cuda.get_device_properties(
                                  dist.local_rank).multi_processor_count}), flush=True)
        dist.close()
        return 0
    res = measure_workload(torch, dist, args.workload, args.steps, args.warmup,
                           with_e2e=True, sustain_s=2.0)
    clk = clocks.summary(*res["host_window"])
    sms = torch.cuda.get_device_properties(dist.local_rank).multi_processor_count

    per_dtype = {}
    if not args.headline_only:
        from mixed_precision_dense_02_gb300 import synth
        for name in synth.WORKLOADS:
            if name == args.workload:
                continue
            wm = workload_meta(name)
            k = 3 if wm["dtype_in"] == "f64" else max(3, min(args.steps, 20))
            r = measure_workload(torch, dist, name, k, 3, with_e2e=False,
                                 sustain_s=1.0)
            # the row's own clock record (its timed region, extended to a
            # second of the same loop)
            add_nominal(r["roofline"], sms, clocks.summary(*r["host_window"]))
            per_dtype[name] = {"value": r["value"], "unit": r["unit"],
                               "ms_per_step": r["ms_per_step"], "steps": k,
                               "pct_of_bf16_peak": r["pct_of_bf16_peak"],
                               "l2": r["l2"],
                               "roofline": r["roofline"]}
            if dist.rank == 0 and dist.world == 1:
                # the oracle beside each row, on a short bounded sample
                per_dtype[name]["cpu_baseline"] = cpu_baseline(name, target_s=2.0)
                _INPUT_CACHE.pop(name, None)
    clocks.stop()
    add_nominal(res["roofline"], sms, clk)

    cpu = None
    if dist.rank == 0 and dist.world == 1:
        cpu = cpu_baseline(args.workload)

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": res["unit"],
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": _dtype_tag(w),
            "data": "synthetic (seeded Philox; shapes/distributions of the workload)",
            "config": _config(args.workload, w, res["l2"]),
            "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
            "clocks": clk, "gpu_launches": res["gpu_launches"],
            "probes": dict(probes, clocks=probe_clk),
            "per_dtype": per_dtype,
        }
        # a compact copy of every row last, so that a reader keeping only the
        # end of the line still sees all of them: value, unit, roofline
        # fraction (of the measured peak), mean kernel time in us
        line["per_dtype_summary"] = {
            name: [round(r["value"], 2), r["unit"], round(r["roofline"]["frac"], 3),
                   round(r["roofline"]["kernel_ms_mean"] * 1e3, 2)]
            for name, r in per_dtype.items()}
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
