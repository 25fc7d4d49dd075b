#!/usr/bin/env python3
"""Throughput benchmark of the pipelined GEMMs on GB300.

Default workload (one GPU): fp32 SGEMM M = N = K = 4096, row-major, A, B and
the initial C uniform in [-1, 1) from a fixed seed, alpha = 1, beta = 0.5 --
the FFMA path.  The bf16 8192^3 and int8 4096^3 workloads, and the bf16 K
sweep (M = N = 4096, K in {32, 64, 128, 512, 2048, 16384}) with the ragged
4095 x 4097 x 4100 shape, are measured in the same run and reported under
"also", each with its own roofline and clock record.

A step is one library call C <- alpha*A*B + beta*C on operands already
resident in HBM.  Between timed steps L2 is flushed by writing a buffer larger
than L2 and reading it back (so that L2 holds only clean lines when the call
starts), and each step is timed with CUDA events on the launching stream;
the K timed steps are bracketed by a barrier and a device synchronise, and the
reported time is the maximum over ranks.

``e2e`` times the same call end to end: the pinned host operands are copied to
the device, the GEMM runs, and C is copied back, every step.

``--impl reference`` times the CPU oracle (the reference arm of this
comparison) on the host cores, on a bounded sample of the same workload.

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the GEMM is not partitioned across GPUs); ``value`` is the FLOPs of all ranks
divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "GEMM TFLOP/s (TOP/s int8) at 4096-8192^3 and % of GB300 dtype peak, 1 GPU"

# name -> (dtype, M, N, K, recipe, seed)
WORKLOADS = {
    "sgemm_fp32_4096": ("f32", 4096, 4096, 4096, "f32_uniform_beta", si.config_seed(2)),
    "igemm_i8_4096": ("i8", 4096, 4096, 4096, "i8_uniform", si.config_seed(3)),
    "gemm_bf16_8192": ("bf16", 8192, 8192, 8192, "bf16_normal", si.config_seed(4)),
}
# The bf16 K sweep and the ragged shape: short K (fewer K-tiles than stages)
# is bound by writing C, long K by the tensor pipe.  Same seeds as the
# parity tests of these shapes.
K_SWEEP = (32, 64, 128, 512, 2048, 16384)
for _k in K_SWEEP:
    WORKLOADS[f"gemm_bf16_4096x4096_k{_k}"] = ("bf16", 4096, 4096, _k, "bf16_normal",
                                               si.config_seed(5, _k % 251))
WORKLOADS["gemm_bf16_ragged_4095x4097x4100"] = ("bf16", 4095, 4097, 4100, "bf16_normal",
                                                si.config_seed(6))
DEFAULT_WORKLOAD = "sgemm_fp32_4096"
# The pages' own figure for a workload, where they print one (TFLOP/s): the
# double-buffered SGEMM of "Double Buffering: Software Pipelining the K-Loop"
# (its results table: 4096^3 in 4.281 ms, 32107.5 GFLOP/s, hardware not
# stated).  Context from another machine, not a target.
PAGE_FIGURES = {"sgemm_fp32_4096": (32.1075, "the SGEMM page's double-buffered kernel, "
                                              "4096^3 fp32, 32.1 TFLOP/s on unstated hardware")}


def vs_baseline(workload: str, value: float):
    """value / the pages' figure for this workload, or None where they print none."""
    fig = PAGE_FIGURES.get(workload)
    return None if fig is None else float(f"{value / fig[0]:.4g}")
L2_FLUSH_BYTES = 512 << 20  # > 129 MB of L2


def l2_flush(flush, i: int):
    """Evict A, B and C from L2 between timed steps: write a buffer larger
    than L2, then read it back whole.  The read leaves L2 holding clean lines
    only; after the write alone it would be full of dirty lines, and the next
    call would pay for writing them back to HBM as its own data came in (an
    HBM-bound call most of all)."""
    flush.fill_(float(i))
    return flush.sum()


# ------------------------------------------------------------------ peaks ---
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def ffma_peak_tflops(sm_count: int, mhz: float) -> float:
    """FP32 FFMA peak: SMs x 128 FP32 lanes x 2 FLOP per FMA x clock."""
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


INT8_MMA_CEILING_TOPS = 153.5  # 128.0 TOP/s measured at 83.4 % integer-subpipe activity


def algorithmic_bytes(dtype: str, M: int, N: int, K: int, beta) -> int:
    """HBM bytes a call must move at least: A and B read once, C written once
    (and read once when beta != 0)."""
    eb = {"f32": 4, "bf16": 2, "i8": 1}[dtype]
    return (M * K + K * N) * eb + M * N * 4 * (2 if beta != 0 else 1)


def roofline_point(dtype: str, M: int, N: int, K: int, beta, ms: float, sm_count: int,
                   peaks: dict) -> dict:
    """Roofline of one call timed at `ms`: against the HBM copy rate when its
    arithmetic intensity is below the ridge (peak FLOP/s over HBM bytes/s),
    else against the compute peak of its dtype."""
    flops = 2.0 * M * N * K
    tflops = flops / (ms * 1e-3) / 1e12
    nbytes = algorithmic_bytes(dtype, M, N, K, beta)
    if dtype != "f32":
        ridge = float(peaks["bf16_tflops"]) * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
        if flops / nbytes < ridge:
            gbs = nbytes / (ms * 1e-3) / 1e9
            peak = float(peaks["hbm_gbs"])
            return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(gbs / peak, 4), "bytes": int(nbytes),
                    "peak_source": f"{peaks['source']} HBM copy rate",
                    "intensity_flop_per_byte": round(flops / nbytes, 1),
                    "ridge_flop_per_byte": round(ridge, 1)}
    return roofline_for(dtype, tflops, sm_count, peaks)


def roofline_for(dtype: str, achieved_tflops: float, sm_count: int, peaks: dict) -> dict:
    if dtype == "f32":
        peak = ffma_peak_tflops(sm_count, float(peaks.get("sm_max_mhz", 2070.0)))
        return {"bound": "alu", "achieved": round(achieved_tflops, 2), "peak": round(peak, 2),
                "unit": "TFLOP/s", "frac": round(achieved_tflops / peak, 4),
                "peak_source": f"derived: {sm_count} SMs x 128 FP32 lanes x 2 x "
                               f"{peaks.get('sm_max_mhz', 2070.0)} MHz"}
    # bf16, and int8 run as fp16 on the same kind::f16 tensor pipe (same nominal rate)
    peak = float(peaks["bf16_tflops"])
    out = {"bound": "tensor", "achieved": round(achieved_tflops, 2), "peak": peak,
           "unit": "TFLOP/s" if dtype == "bf16" else "TOP/s",
           "frac": round(achieved_tflops / peak, 4),
           "peak_source": f"{peaks['source']} bf16 dense (burst)" +
                          ("; int8 runs as exact fp16 products on the same pipe" if dtype == "i8" else "")}
    sustained = peaks.get("bf16_tflops_sustained")
    if sustained:
        # the measured rate of a seconds-long loop under the power cap, for
        # context beside the burst figure the fraction is taken against
        out["sustained_peak"] = float(sustained)
        out["frac_of_sustained"] = round(achieved_tflops / float(sustained), 4)
    if dtype == "i8":
        # the integer MMA rate of this GPU, for context: the mma.sync engine's
        # 128 TOP/s on int8 4096^3 at 83 % integer-subpipe activity (ncu)
        out["int8_mma_ceiling"] = {"value": INT8_MMA_CEILING_TOPS, "unit": "TOP/s",
                                   "ratio": round(achieved_tflops / INT8_MMA_CEILING_TOPS, 2),
                                   "source": "derived from ncu: 128.0 TOP/s / 0.834 integer tensor "
                                             "subpipe active"}
    return out


def traffic_for(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e.get("dram_bytes_per_launch")


def launches_per_call(dtype: str, M: int, N: int, K: int) -> int:
    """This library's kernel launches in one default call: the operand pre-pass
    (int8 widening of A and B in one launch; one launch repacking every
    bf16/fp32 operand whose pitch is not a multiple of 16 bytes), then the
    GEMM, which for fp32 is two grids when the stream-K tail is in use."""
    import software_pipelined_tiled_loop_gb300 as pg
    eb = {"f32": 4, "bf16": 2, "i8": 1}[dtype]
    n = 0
    if K > 0:
        if dtype == "i8":
            n += 1
        else:
            n += int((K * eb) % 16 != 0 or (N * eb) % 16 != 0)
    s = pg.pgemm_schedule(dtype, M, N, K)
    if dtype == "f32" and s["split_tiles"] > 0:
        n += 1 + int(s["tiles"] > s["split_tiles"])
    else:
        n += 1
    return n


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "software_pipelined_tiled_loop_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm ---
def _torch_dtype(torch, np_dtype):
    return {np.float32: torch.float32, np.int8: torch.int8, np.int32: torch.int32,
            np.uint16: torch.int16}[np.dtype(np_dtype).type]


def _to_dev(torch, x):
    if x.dtype == np.uint16:
        x = x.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host_ahead(torch, stream, steps):
    """Queue a bounded spin (torch's own sleep kernel, about 0.2 ms a step)
    ahead of the timed steps, so that the host has queued them all before the
    GPU reaches the first: the events then time the GPU's work, not gaps
    where it waited for the host to launch the next call."""
    torch.cuda._sleep(int(min(steps, 200) * 0.2e-3 * 2.0e9))


def run_e2e(torch, fn, dtype, M, N, K, alpha, beta, A, B, C0, dA, dB, dC, e_steps, dist_ctx,
            flops, stream) -> dict:
    """End to end through the public call: every step copies its A, B and C
    from pinned host memory to the device, runs the GEMM and reads C back.

    The steps are software-pipelined across streams the way the kernel
    pipelines its K-loop: three device buffer sets, host-to-device copies on
    one copy stream, the GEMM on the compute stream, the read-back on
    another, so that step i's copies overlap step i - 1's GEMM.  A step's
    copies into a buffer set wait until the step three before it has read its
    result back from that set (with two sets, a copy held up behind the
    previous read-back held up the next GEMM).  The serial loop (copy, GEMM, read back, one after
    another) is timed too and reported beside it."""
    hA = torch.from_numpy(A.view(np.int16) if A.dtype == np.uint16 else A).pin_memory()
    hB = torch.from_numpy(B.view(np.int16) if B.dtype == np.uint16 else B).pin_memory()
    hC = torch.from_numpy(C0).pin_memory()
    NSETS = 3
    hOut = [torch.empty_like(hC).pin_memory() for _ in range(NSETS)]
    sets = [(dA, dB, dC)] + [(torch.empty_like(dA), torch.empty_like(dB), torch.empty_like(dC))
                             for _ in range(NSETS - 1)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def serial(n):
        for _ in range(n):
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            dC.copy_(hC, non_blocking=True)
            fn(M, N, K, alpha, dA, dB, beta, dC, stream=stream)
            hOut[0].copy_(dC, non_blocking=True)

    def pipelined(n, t0):
        s_in.wait_event(t0)
        read_back = []
        for i in range(n):
            a, b, c = sets[i % NSETS]
            with torch.cuda.stream(s_in):
                if i >= NSETS:
                    s_in.wait_event(read_back[i - NSETS])
                a.copy_(hA, non_blocking=True)
                b.copy_(hB, non_blocking=True)
                c.copy_(hC, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            fn(M, N, K, alpha, a, b, beta, c, stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                hOut[i % NSETS].copy_(c, non_blocking=True)
                back = torch.cuda.Event()
                back.record(s_out)
            read_back.append(back)
        stream.wait_event(read_back[-1])

    def timed(body, n):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        dist_ctx.barrier()
        torch.cuda.synchronize()
        host_ahead(torch, stream, n)
        t0.record(stream)
        if body is pipelined:
            pipelined(n, t0)
        else:
            serial(n)
        t1.record(stream)
        torch.cuda.synchronize()
        dist_ctx.barrier()
        return dist_ctx.max(t0.elapsed_time(t1))

    for body in (serial, pipelined):  # untimed warm-up of both loops
        timed(body, 2)
    ms_serial = timed(serial, e_steps)
    ms_pipe = timed(pipelined, e_steps)
    for h in hOut:  # every read-back buffer holds a full result
        if not torch.equal(h, hOut[0]):
            raise RuntimeError("pipelined read-back differs between buffer sets")
    tput = lambda ms: round(flops * e_steps * dist_ctx.world / (ms * 1e-3) / 1e12, 3)
    h2d = A.nbytes + B.nbytes + C0.nbytes
    return {"value": tput(ms_pipe), "unit": "TFLOP/s" if dtype != "i8" else "TOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(C0.nbytes),
            "steps": e_steps, "ms_per_step": round(ms_pipe / e_steps, 4),
            "pipelined": "three buffer sets; copies overlap the neighbouring steps' GEMMs",
            "serial_value": tput(ms_serial), "serial_ms_per_step": round(ms_serial / e_steps, 4)}


def run_gpu_workload(name: str, steps: int, warmup: int, dist_ctx, with_e2e: bool,
                     clocks: "ClockSampler | None" = None) -> dict:
    import torch

    import software_pipelined_tiled_loop_gb300 as pg

    dtype, M, N, K, recipe, seed = WORKLOADS[name]
    A, B, C0, alpha, beta, _ = si.workload(recipe, M, N, K, seed)
    fn = {"f32": pg.gemm_f32, "bf16": pg.gemm_bf16, "i8": pg.gemm_i8}[dtype]
    dA, dB, dC = _to_dev(torch, A), _to_dev(torch, B), _to_dev(torch, C0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    flops = 2.0 * M * N * K

    for _ in range(warmup):
        fn(M, N, K, alpha, dA, dB, beta, dC)
    torch.cuda.synchronize()
    if pg.pgemm_get_device_status() != 0:
        raise RuntimeError("device status after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dist_ctx.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    t_wall = time.perf_counter()
    host_ahead(torch, stream, steps)
    for i in range(steps):
        l2_flush(flush, i)  # evict A, B, C from L2 between timed steps
        starts[i].record(stream)
        fn(M, N, K, alpha, dA, dB, beta, dC)
        ends[i].record(stream)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    per_step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    clk = None
    if clocks is not None:
        # nvidia-smi samples every 100 ms: if the timed region was shorter than
        # one second, the same steps keep running (untimed) until the clock
        # window covers a second of this load
        while time.perf_counter() - t_wall < 1.0:
            for i in range(8):
                l2_flush(flush, i)
                fn(M, N, K, alpha, dA, dB, beta, dC)
            torch.cuda.synchronize()
        clk = clocks.stop()
        clk["window_s"] = round(time.perf_counter() - t_wall, 2)
    if pg.pgemm_get_device_status() != 0:
        raise RuntimeError("device status after timed steps")
    total_ms = dist_ctx.max(sum(per_step_ms))
    res = {"dtype": dtype, "M": M, "N": N, "K": K, "alpha": alpha, "beta": beta,
           "ms_per_step": total_ms / steps, "ms_min": min(per_step_ms),
           "ms_median": statistics.median(per_step_ms),
           "tflops": aggregate_throughput(flops, steps, dist_ctx.world, total_ms),
           "per_gpu_tflops": flops * steps / (total_ms * 1e-3) / 1e12,
           "launches_per_step": launches_per_call(dtype, M, N, K),
           "config": pg.pgemm_default_config(dtype, M, N, K), "clocks": clk}

    if with_e2e:
        # as many steps as the device-timed loop: the pipeline's fill (the
        # first step's copies in) and drain (the last step's read-back) are
        # then spread over the same number of calls
        res["e2e"] = run_e2e(torch, fn, dtype, M, N, K, alpha, beta, A, B, C0, dA, dB, dC,
                             max(3, steps), dist_ctx, flops, stream)
    del dA, dB, dC, flush
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------- CPU oracle ---
def oracle_sample(name: str, target_s: float) -> dict:
    """Time the oracle, as it stands, on a bounded sample (whole rows) of the
    workload on the host cores; return throughput in the metric's unit."""
    import oracle

    dtype, M, N, K, recipe, seed = WORKLOADS[name]
    A, B, C0, alpha, beta, _ = si.workload(recipe, M, N, K, seed)
    orc = oracle.get()
    threads = orc.num_threads()
    rows = max(1, threads)
    t0 = time.perf_counter()
    orc.gemm(dtype, A, B, C0, alpha, beta, rows=(0, rows))
    dt = time.perf_counter() - t0
    # scale the sample to about target_s seconds of CPU work
    rows2 = int(min(M, max(rows, rows * target_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    orc.gemm(dtype, A, B, C0, alpha, beta, rows=(0, rows2))
    dt2 = time.perf_counter() - t0
    flops = 2.0 * rows2 * N * K
    return {"value": round(flops / dt2 / 1e12, 6), "unit": "TFLOP/s" if dtype != "i8" else "TOP/s",
            "cores": threads, "kind": "oracle",
            "sample": f"{rows2} of {M} output rows of the {name} workload "
                      f"({rows2}x{N}x{K}, {dt2:.1f} s)",
            "seconds": round(dt2, 2)}


# ------------------------------------------------------------------ sweep ---
SWEEP_SHAPES = {
    # dtype -> list of (M, N, K, recipe); the bf16 K list is the K-sweep workload
    "f32": [(4096, 4096, 4096, "f32_uniform_beta")],
    "i8": [(4096, 4096, 4096, "i8_uniform")],
    "bf16": [(8192, 8192, 8192, "bf16_normal")] +
            [(4096, 4096, k, "bf16_normal") for k in (32, 64, 128, 512, 2048, 16384)] +
            [(4095, 4097, 4100, "bf16_normal")],
}


def run_point(dtype, M, N, K, recipe, cfg, steps, warmup, seed=None):
    """Time one (shape, configuration) point; returns a dict (no correctness check:
    the parity tests cover every configuration)."""
    import torch

    import software_pipelined_tiled_loop_gb300 as pg

    seed = si.config_seed(5, K % 251) if seed is None else seed
    A, B, C0, alpha, beta, _ = si.workload(recipe, M, N, K, seed)
    fn = {"f32": pg.gemm_f32_ex, "bf16": pg.gemm_bf16_ex, "i8": pg.gemm_i8_ex}[dtype]
    dA, dB, dC = _to_dev(torch, A), _to_dev(torch, B), _to_dev(torch, C0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn(M, N, K, alpha, dA, dB, beta, dC, config=cfg)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):  # queued back to back: host work overlaps the GPU
        l2_flush(flush, i)
        ev[i][0].record(stream)
        fn(M, N, K, alpha, dA, dB, beta, dC, config=cfg)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    status = pg.pgemm_get_device_status()
    attrs = pg.pgemm_kernel_attrs(dtype, cfg)
    sched = pg.pgemm_schedule(dtype, M, N, K, cfg)
    med = statistics.median(ms)
    flops = 2.0 * M * N * K
    out_bytes = M * N * 4 * (2 if beta != 0 else 1)
    in_bytes = (M * K + K * N) * {"f32": 4, "bf16": 2, "i8": 1}[dtype]
    del dA, dB, dC, flush
    return {"dtype": dtype, "M": M, "N": N, "K": K, "bm": cfg[0], "bn": cfg[1], "bk": cfg[2],
            "stages": cfg[3], "max_k_parts": cfg[4] if len(cfg) > 4 else 0,
            "group_m": cfg[7] if len(cfg) > 7 else 0,
            "producer": {v: k for k, v in pg.PRODUCERS.items()}[cfg[5] if len(cfg) > 5 else 0],
            "engine": {v: k for k, v in pg.ENGINES.items()}[cfg[6] if len(cfg) > 6 else 0],
            "k_tiles": -(-K // cfg[2]), **attrs, **sched, "ms_median": round(med, 4),
            "ms_min": round(min(ms), 4), "tflops": round(flops / (med * 1e-3) / 1e12, 2),
            "gbs": round((in_bytes + out_bytes) / (med * 1e-3) / 1e9, 1), "status": status}


def sweep(dtypes, steps, warmup, only_k=None):
    import software_pipelined_tiled_loop_gb300 as pg
    for dtype in dtypes:
        for (M, N, K, recipe) in SWEEP_SHAPES[dtype]:
            if only_k is not None and K not in only_k:
                continue
            for cfg in pg.pgemm_list_configs(dtype):
                print(json.dumps(run_point(dtype, M, N, K, recipe, cfg, steps, warmup)), flush=True)


# ----------------------------------------------------- stage-reuse hazard ---
def hazard_stress(iters: int, delay_ns: int = 2000) -> dict:
    """Run the two-stage copy-and-reduce with and without the
    consume-before-reuse wait `iters` times each on a 4096 x 4096 integer
    array with a fresh random row order every iteration and consumer warp 0
    slowed by delay_ns per tile; count wrong row sums against the exact host
    sums, and pull one annotated overwrite out of the hazard run's trace."""
    import torch

    import software_pipelined_tiled_loop_gb300 as pg
    rows = cols = 4096
    X = si.small_int_f32((rows, cols), 77, -8, 7)
    rowsum = X.astype(np.int64).sum(axis=1)
    dX = torch.from_numpy(X).cuda()
    out = torch.zeros(rows, dtype=torch.float32, device="cuda")
    cap = 8192
    tr = torch.zeros(1 + 2 * cap, dtype=torch.int64, device="cuda")
    rng = np.random.default_rng(0x5EED)
    res = {}
    for check in (1, 0):
        fails, bad_rows, ms = 0, [], []
        for it in range(iters):
            perm = rng.permutation(rows).astype(np.int32)
            dperm = torch.from_numpy(perm).cuda()
            out.zero_()
            tr.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pg.pgemm_stage_reuse_demo(dX, rows, cols, dperm, out, check, 0, delay_ns,
                                      tr if it == 0 else None, cap if it == 0 else 0)
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
            bad = int(np.count_nonzero(out.cpu().numpy().astype(np.int64) != rowsum[perm]))
            bad_rows.append(bad)
            fails += bad > 0
            if it == 0:
                trace = tr.cpu().numpy().view(np.uint64).copy()
        status = pg.pgemm_get_device_status()
        name = "with_reuse_wait" if check else "without_reuse_wait"
        res[name] = {"iterations": iters, "iterations_with_wrong_rows": fails,
                     "wrong_rows_total": int(sum(bad_rows)), "wrong_rows_max": int(max(bad_rows)),
                     "ms_median": round(statistics.median(ms), 4),
                     "GB_per_s": round(rows * cols * 4 / (statistics.median(ms) * 1e-3) / 1e9, 1),
                     "device_status": status, "timeline": _timeline_excerpt(trace, check)}
    res["delay_ns_warp0"] = delay_ns
    return res


def _timeline_excerpt(tr, check):
    """A few events around one stage reuse of block 0, times in ns from the first event."""
    names = {1: "load issued", 2: "load landed", 3: "reuse wait begins", 4: "reuse allowed",
             5: "read begins", 6: "read ends"}
    n = int(tr[0])
    ev = sorted((int(tr[1 + 2 * i]), int(tr[2 + 2 * i]) >> 56, (int(tr[2 + 2 * i]) >> 48) & 0xFF,
                 (int(tr[2 + 2 * i]) >> 40) & 0xFF, int(tr[2 + 2 * i]) & 0xFFFFFFFF)
                for i in range(min(n, (len(tr) - 1) // 2)))
    if not ev:
        return []
    t0 = ev[0][0]
    # around tile 4 of stage 0: its load, the reads of tile 2 (same stage) by every warp
    keep = [e for e in ev if e[4] in (2, 4) and e[2] == 0]
    if not check:
        # the overwrite: tile 4's load landing before warp 0 has begun reading tile 2
        keep = [e for e in ev if (e[4] == 4 and e[1] in (1, 2)) or (e[4] == 2 and e[1] in (5, 6))]
    return [f"{e[0] - t0:>8d} ns  tile {e[4]} stage {e[2]} warp {e[3]}: {names.get(e[1], e[1])}"
            for e in keep[:24]]


# ------------------------------------------------------------ distributed ---
class DistCtx:
    """One process per GPU (torchrun); replicas only: no data-path collective.

    The process group serves the barrier around the timed region and the
    max-over-ranks of the timing.  NCCL on GPUs, gloo where there is none
    (the multi-rank logic is tested on CPU with gloo)."""

    def __init__(self, backend: str | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cpu"
        if self.world > 1:
            import torch
            import torch.distributed as dist
            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
                self.device = "cuda"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate_throughput(flops_per_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput in TFLOP/s: the FLOPs every rank did, over the
    slowest rank's time (each rank runs its own full replica)."""
    return flops_per_step * steps * world / (max_total_ms * 1e-3) / 1e12


# ------------------------------------------------------------------- main ---
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pgemm", "reference"], default="pgemm")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-also", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work of the oracle sample (cpu_baseline / reference arm)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end timing")
    ap.add_argument("--sweep", default=None,
                    help="comma list of dtypes: time every built (tile, stages) config on the "
                         "sweep shapes, one JSON line per point")
    ap.add_argument("--sweep-k", default=None, help="comma list of K values to restrict the sweep")
    ap.add_argument("--hazard", type=int, default=0,
                    help="run the stage-reuse hazard experiment this many iterations per variant")
    ap.add_argument("--point", default=None,
                    help="dtype,M,N,K,bm,bn,bk,stages[,max_k_parts[,producer[,engine[,group_m]]]]: time one point "
                         "(for profiler captures and split / no-split comparisons)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.hazard:
        from software_pipelined_tiled_loop_gb300 import build as pgbuild
        pgbuild.build()
        print(json.dumps(hazard_stress(args.hazard)))
        return
    if args.sweep or args.point:
        from software_pipelined_tiled_loop_gb300 import build as pgbuild
        pgbuild.build()
        if args.sweep:
            ks = {int(k) for k in args.sweep_k.split(",")} if args.sweep_k else None
            sweep(args.sweep.split(","), args.steps, args.warmup, ks)
        else:
            f = args.point.split(",")
            dt, nums = f[0], [int(x) for x in f[1:]]
            M, N, K = nums[:3]
            recipe = {"f32": "f32_uniform_beta", "bf16": "bf16_normal", "i8": "i8_uniform"}[dt]
            print(json.dumps(run_point(dt, M, N, K, recipe, tuple(nums[3:]), args.steps,
                                       args.warmup)))
        return

    dtype, M, N, K, recipe, seed = WORKLOADS[args.workload]
    config = {"workload": args.workload, "dtype": dtype, "M": M, "N": N, "K": K,
              "recipe": recipe, "seed": seed, "l2": "flushed between timed steps (512 MiB written, then read back: "
                    "L2 holds clean lines when each call starts)"}

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        per, secs = [], []
        for _ in range(args.warmup):
            oracle_sample(args.workload, 0.05)  # untimed: loads the library, touches the operands
        sample = None
        for _ in range(args.steps):
            sample = oracle_sample(args.workload, max(1.0, args.cpu_seconds / args.steps))
            per.append(sample["value"])
            secs.append(sample["seconds"])
        value = statistics.median(per)
        line = {"metric": METRIC, "value": value, "unit": sample["unit"], "impl": "reference",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1000 * statistics.median(secs), 1), "higher_is_better": True,
                "scaling": "weak",
                "vs_baseline": vs_baseline(args.workload, value),
                "vs_baseline_of": PAGE_FIGURES.get(args.workload, (None, None))[1],
                "dtype": {"f32": "f32", "bf16": "bf16", "i8": "int8"}[dtype],
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": sample["unit"], "cores": sample["cores"],
                                 "kind": "oracle", "sample": sample["sample"]},
                "e2e": {"value": value, "unit": sample["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    ctx = DistCtx()
    import software_pipelined_tiled_loop_gb300 as pg
    from software_pipelined_tiled_loop_gb300 import build as pgbuild
    if ctx.rank == 0:
        pgbuild.build()
    ctx.barrier()
    pg.lib()
    peaks = measured_peaks()
    sm_count = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(ctx.local_rank)).split(",")[0] or 0) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else ctx.local_rank

    main_res = run_gpu_workload(args.workload, args.steps, args.warmup, ctx,
                                with_e2e=not args.no_e2e, clocks=ClockSampler(gpu_index))
    clk = main_res["clocks"]

    also = {}
    if not args.no_also:
        for other in WORKLOADS:
            if other == args.workload:
                continue
            r = run_gpu_workload(other, max(5, args.steps // 2), args.warmup, ctx, with_e2e=False,
                                 clocks=ClockSampler(gpu_index))
            also[other] = {"value": round(r["tflops"], 2), "clocks": r["clocks"],
                           "unit": "TOP/s" if r["dtype"] == "i8" else "TFLOP/s",
                           "shape": [r["M"], r["N"], r["K"]],
                           "ms_per_step": round(r["ms_per_step"], 4),
                           "ms_median": round(r["ms_median"], 4),
                           "roofline": {**roofline_point(r["dtype"], r["M"], r["N"], r["K"], r["beta"],
                                                         r["ms_per_step"], sm_count, peaks),
                                        "traffic": traffic_for(other)},
                           "config": r["config"]}

    cpu = None
    if ctx.rank == 0 and ctx.world == 1 and not args.no_cpu:
        cpu = oracle_sample(args.workload, args.cpu_seconds)

    if ctx.rank == 0:
        roof = roofline_for(dtype, main_res["per_gpu_tflops"], sm_count, peaks)
        roof["traffic"] = traffic_for(f"{args.workload}")
        roof["timing"] = "CUDA events around each call on the launching stream, L2 flushed between"
        unit = "TOP/s" if dtype == "i8" else "TFLOP/s"
        line = {
            "metric": METRIC, "value": round(main_res["tflops"], 3), "unit": unit,
            "n_gpus": ctx.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(main_res["ms_per_step"], 4),
            "ms_median": round(main_res["ms_median"], 4), "ms_min": round(main_res["ms_min"], 4),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": vs_baseline(args.workload, main_res["tflops"]),
            "vs_baseline_of": PAGE_FIGURES.get(args.workload, (None, None))[1],
            "dtype": {"f32": "f32", "bf16": "bf16", "i8": "int8"}[dtype],
            "data": "synthetic (seeded splitmix64 draws; recipes in seeded_inputs.workload)",
            "config": {**config, "tile_stages": main_res["config"],
                       "parallelism": "replicas" if ctx.world > 1 else "single"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": main_res.get("e2e"),
            "gpu_launches": main_res["launches_per_step"] * args.steps,
            "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"),
                       "reasons": clk.get("reasons"), "samples": clk.get("samples"),
                       "window_s": clk.get("window_s")},
            "also": also,
        }
        print(json.dumps(line))
    ctx.close()


if __name__ == "__main__":
    main()
