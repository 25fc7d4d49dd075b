"""Host-side arithmetic pinned to numbers the pages print
(tests/golden/page_numbers.txt, each with its citation)."""
import os

import pytest

from software_pipelined_tiled_loop_gb300 import model

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_numbers.txt")


@pytest.fixture(scope="module")
def g():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split(":")
            out[k.strip()] = float(v)
    return out


def test_flop_count_reproduces_the_sgemm_page_throughput(g):
    # the page prints the time to 3 decimals: 2*M*N*K / t must hit the printed
    # GFLOP/s for some t that rounds to the printed time
    M, N, K = int(g["p1_gemm_m"]), int(g["p1_gemm_n"]), int(g["p1_gemm_k"])
    ms = g["p1_kernel11_ms"]
    hi = model.throughput_gflops(M, N, K, ms - 0.0005)
    lo = model.throughput_gflops(M, N, K, ms + 0.0005)
    assert lo <= g["p1_kernel11_gflops"] <= hi
    # a different FLOP count (e.g. M*N*K, or 2*M*N*K counted twice) cannot
    assert not (lo / 2 <= g["p1_kernel11_gflops"] <= hi / 2)
    assert round(100 * (g["p1_kernel10_ms"] / g["p1_kernel11_ms"] - 1), 1) == g["p1_speedup_pct"]


def test_register_residency_reproduces_the_sgemm_page(g):
    r = int(g["p1_regs_per_thread"])
    t = int(g["p1_threads_per_block"])
    assert model.regs_per_warp(r) == g["p1_regs_per_warp"]
    assert model.regs_per_warp(r) * (t // 32) == g["p1_regs_per_block"]
    assert model.blocks_per_sm_by_registers(r, t, int(g["p1_regs_per_sm"])) == g["p1_blocks_per_sm"]
    assert model.blocks_per_sm_by_registers(int(g["p1_prev_regs_per_thread"]), t) == \
        g["p1_prev_blocks_per_sm"]


def test_latency_model_reproduces_the_worked_example(g):
    L, C = g["p2_latency_cycles"], g["p2_compute_cycles"]
    assert model.uncovered_latency(L, C, stages=2) == g["p2_uncovered_cycles"]
    assert model.iteration_cycles(L, C, 1) == L + C
    assert model.iteration_cycles(L, C, 2) == max(L, C)
    # more stages never expose more latency
    assert model.uncovered_latency(L, C, 4) <= model.uncovered_latency(L, C, 2)


def test_ring_budget_doubles_with_the_second_stage(g):
    single = model.ring_bytes(64, 64, 16, 2, 1)
    assert single == g["p3_single_kb"] * 1024
    assert model.ring_bytes(64, 64, 16, 2, 2) == g["p3_double_kb"] * 1024
