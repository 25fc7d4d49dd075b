"""Host-side models used to read the stage sweep (no GPU, no CUDA).

* GEMM work: 2*M*N*K floating-point operations per call, the count behind
  the SGEMM page's throughput figure ("Double Buffering: Software Pipelining
  the K-Loop", section "Mechanics": 4096^3 in 4.281 ms at 32107.5 GFLOP/s).
* Register residency: registers per thread rounded up per warp to the
  allocation unit, times warps per block, divided into the register file
  (same page, section "What The Overlap Cost": 150 registers -> 4864 per
  warp -> 19456 per block of four warps -> 3 blocks per SM).
* Latency coverage: with one tile of lookahead an iteration approaches
  max(L, C) instead of L + C, and max(0, L - C) of the load latency stays
  exposed ("Software pipelines and asynchronous copies", sections "Why
  alternating load and compute leaves idle time" and "Worked example");
  each further stage adds one more tile of compute to hide it behind.
* Ring budget: S * (A panel + B panel) bytes of shared memory ("GPU-Kernel
  pipelinen", Schritt 1: the double buffer costs twice the single one).
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def throughput_gflops(M: int, N: int, K: int, ms: float) -> float:
    return gemm_flops(M, N, K) / (ms * 1e-3) / 1e9


def regs_per_warp(regs_per_thread: int, warp_size: int = 32, unit: int = 256) -> int:
    return -(-regs_per_thread * warp_size // unit) * unit


def blocks_per_sm_by_registers(regs_per_thread: int, threads_per_block: int,
                               regfile: int = 65536, warp_size: int = 32, unit: int = 256) -> int:
    warps = -(-threads_per_block // warp_size)
    return regfile // (regs_per_warp(regs_per_thread, warp_size, unit) * warps)


def uncovered_latency(load_cycles: float, compute_cycles: float, stages: int = 2) -> float:
    """Load latency left exposed per K-tile with `stages` ring slots: the
    S - 1 tiles in flight ahead of the one being computed cover (S - 1) * C."""
    return max(0.0, load_cycles - (stages - 1) * compute_cycles)


def iteration_cycles(load_cycles: float, compute_cycles: float, stages: int) -> float:
    """Steady-state cycles per K-tile: L + C with one slot, max(L, C) once
    the loads overlap the arithmetic (two or more slots)."""
    if stages <= 1:
        return load_cycles + compute_cycles
    return max(compute_cycles, load_cycles - (stages - 2) * compute_cycles, compute_cycles)


def ring_bytes(bm: int, bn: int, bk: int, elem_bytes: int, stages: int) -> int:
    return stages * (bm * bk + bk * bn) * elem_bytes
