"""Host logic of bench.py: how many of the library's kernel launches one
default call makes (the `gpu_launches` claim; the schedule it depends on
asks the device, so that case runs on a GPU), the roofline arithmetic and
the peaks it divides by, and the DRAM-traffic lookup that must go blank
once the kernel sources no longer match the capture."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from software_pipelined_tiled_loop_gb300 import build
    build.build()


@pytest.mark.gpu  # the schedule asks the device how many blocks are resident
@pytest.mark.parametrize("dtype,M,N,K,launches", [
    ("f32", 4096, 4096, 4096, 2),      # whole-tile grid + stream-K tail grid (1024 tiles on 304)
    ("f32", 4096, 4096, 4095, 3),      # A's pitch (16380 bytes) repacked, then both grids
    ("f32", 256, 256, 256, 1),         # 8 tiles of 128 x 64: no tail grid
    ("i8", 4096, 4096, 4096, 2),       # widening pass + GEMM
    ("i8", 4096, 4096, 0, 1),          # K = 0: no widening, C = beta * C
    ("bf16", 8192, 8192, 8192, 1),     # stream-K inside the persistent kernel
    ("bf16", 4095, 4097, 4100, 2),     # K * 2 and N * 2 not multiples of 16: one repack launch
])
def test_launches_per_call(dtype, M, N, K, launches):
    assert bench.launches_per_call(dtype, M, N, K) == launches


def test_ffma_peak_formula():
    # SMs x 128 FP32 lanes x 2 FLOP per FMA x clock
    assert bench.ffma_peak_tflops(152, 2070.0) == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)


def test_roofline_fields():
    peaks = {"bf16_tflops": 1937.8, "sm_max_mhz": 2070.0, "source": "measured"}
    r = bench.roofline_for("f32", 65.0, 152, peaks)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(65.0 / bench.ffma_peak_tflops(152, 2070.0), abs=1e-4)
    r = bench.roofline_for("bf16", 1800.0, 152, peaks)
    assert r["bound"] == "tensor" and r["peak"] == 1937.8
    assert r["frac"] == pytest.approx(1800.0 / 1937.8, abs=1e-4)
    assert "frac_of_sustained" not in r  # only when a sustained figure was measured
    r = bench.roofline_for("bf16", 1800.0, 152, {**peaks, "bf16_tflops_sustained": 1724.2})
    assert r["frac"] == pytest.approx(1800.0 / 1937.8, abs=1e-4)
    assert r["frac_of_sustained"] == pytest.approx(1800.0 / 1724.2, abs=1e-4)
    r = bench.roofline_for("i8", 1290.0, 152, peaks)
    assert r["unit"] == "TOP/s" and r["peak"] == 1937.8
    assert r["int8_mma_ceiling"]["ratio"] == pytest.approx(1290.0 / bench.INT8_MMA_CEILING_TOPS,
                                                           abs=0.01)


def test_aggregate_throughput_counts_every_rank():
    flops = 2.0 * 4096 ** 3
    one = bench.aggregate_throughput(flops, 10, 1, 21.0)
    assert one == pytest.approx(flops * 10 / 21e-3 / 1e12)
    assert bench.aggregate_throughput(flops, 10, 4, 21.0) == pytest.approx(4 * one)


def test_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """The committed capture is reported while the sources hash to it, and
    blanked (None) as soon as they do not."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        committed = json.load(f)
    entry = committed["sgemm_fp32_4096"]
    if entry["source_sha"] == bench.kernel_source_sha():
        assert bench.traffic_for("sgemm_fp32_4096") == entry["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0" * 16)
    assert bench.traffic_for("sgemm_fp32_4096") is None
    assert bench.traffic_for("no_such_workload") is None


def test_workloads_match_the_metric_shapes():
    # the bench's value is fp32 4096^3 (alpha 1, beta 0.5); int8 4096^3 and
    # bf16 8192^3 are reported beside it
    assert bench.DEFAULT_WORKLOAD == "sgemm_fp32_4096"
    assert bench.WORKLOADS["sgemm_fp32_4096"][:4] == ("f32", 4096, 4096, 4096)
    assert bench.WORKLOADS["igemm_i8_4096"][:4] == ("i8", 4096, 4096, 4096)
    assert bench.WORKLOADS["gemm_bf16_8192"][:4] == ("bf16", 8192, 8192, 8192)
    assert bench.L2_FLUSH_BYTES > 129 * 10 ** 6


def test_vs_baseline_uses_the_pages_figure_only_where_they_print_one():
    # the SGEMM page: 2 * 4096^3 FLOP in 4.281 ms = 32.1075 TFLOP/s
    assert bench.PAGE_FIGURES["sgemm_fp32_4096"][0] == pytest.approx(2 * 4096 ** 3 / 4.281e-3 / 1e12,
                                                                      rel=1e-4)
    assert bench.vs_baseline("sgemm_fp32_4096", 64.215) == pytest.approx(2.0, abs=1e-3)
    assert bench.vs_baseline("gemm_bf16_8192", 1800.0) is None
    assert bench.vs_baseline("igemm_i8_4096", 1280.0) is None


def test_k_sweep_and_ragged_are_bench_workloads():
    # the bf16 K sweep (M = N = 4096) and the ragged shape run beside the
    # headline, with the parity tests' seeds
    import seeded_inputs as si
    for k in (32, 64, 128, 512, 2048, 16384):
        w = bench.WORKLOADS[f"gemm_bf16_4096x4096_k{k}"]
        assert w[:4] == ("bf16", 4096, 4096, k) and w[5] == si.config_seed(5, k % 251)
    assert bench.WORKLOADS["gemm_bf16_ragged_4095x4097x4100"][:4] == ("bf16", 4095, 4097, 4100)


def test_roofline_point_picks_the_bound_by_intensity():
    peaks = {"bf16_tflops": 1937.8, "hbm_gbs": 6791.4, "sm_max_mhz": 2070.0, "source": "measured"}
    M = N = 4096
    # K <= 512: below the ridge (1937.8e12 / 6791.4e9 = 285 FLOP/B): HBM-bound,
    # bytes = C written once (fp32, beta = 0) + bf16 A and B read once
    for K in (32, 64, 128, 512):
        r = bench.roofline_point("bf16", M, N, K, 0.0, 0.02, 152, peaks)
        nbytes = 4 * M * N + 2 * K * (M + N)
        assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["bytes"] == nbytes
        assert r["achieved"] == pytest.approx(nbytes / 0.02e-3 / 1e9, rel=1e-3)
        assert r["frac"] == pytest.approx(r["achieved"] / 6791.4, abs=1e-4)
    for K in (2048, 16384):
        r = bench.roofline_point("bf16", M, N, K, 0.0, 0.05, 152, peaks)
        assert r["bound"] == "tensor"
        assert r["achieved"] == pytest.approx(2.0 * M * N * K / 0.05e-3 / 1e12, rel=1e-3)
    # beta != 0 reads C as well; fp32 is always against the FFMA peak
    assert bench.algorithmic_bytes("f32", 4096, 4096, 4096, 0.5) == 4 * (2 * 4096 ** 2 + 2 * 4096 ** 2)
    assert bench.roofline_point("f32", 4096, 4096, 4096, 0.5, 2.1, 152, peaks)["bound"] == "alu"
