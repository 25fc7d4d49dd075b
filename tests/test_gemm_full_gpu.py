"""Parity at the full workload sizes, in the configuration the bench times.

fp32 4096^3 (beta = 0.5) and int8 4096^3 are compared with the oracle on
every entry.  Elsewhere the oracle evaluates sampled entries one by one: a
few whole rows and columns at tile boundaries, the last row and column, one
random entry inside every 128 x 128 output tile, and random entries.  Float results
must meet max|C - C_ref| <= 1e-4 * sqrt(K) * max|A| * max|B|; int8 is
bit-exact.  The bf16 K sweep runs every built (tile, stage count) on
M = N = 4096 with K in {32, 64, 128, 512, 2048, 16384}, which includes fewer
K-tiles than stages, and the ragged 4095 x 4097 x 4100 shape.
"""
import functools
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import float_bound, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    assert pg.pgemm_get_device_status() == 0


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def sample_indices(M, N, seed, n_random=1500):
    rng = np.random.default_rng(seed)
    edge_r = sorted({r for b in range(0, M, 128) for r in (b, b + 127) if r < M} | {M - 1})
    edge_c = sorted({c for b in range(0, N, 64) for c in (b, b + 63) if c < N} | {N - 1})
    ii, jj = [], []
    # a few edge rows completely, a few edge columns completely
    for r in edge_r[:: max(1, len(edge_r) // 6)]:
        ii += [r] * N
        jj += list(range(N))
    for c in edge_c[:: max(1, len(edge_c) // 6)]:
        ii += list(range(M))
        jj += [c] * M
    # one entry inside every 128 x 128 output tile, so that no tile goes unchecked
    for bi in range(0, M, 128):
        h = min(128, M - bi)
        for bj in range(0, N, 128):
            w = min(128, N - bj)
            ii.append(bi + int(rng.integers(0, h)))
            jj.append(bj + int(rng.integers(0, w)))
    ii += list(rng.integers(0, M, n_random))
    jj += list(rng.integers(0, N, n_random))
    return np.asarray(ii, np.int64), np.asarray(jj, np.int64)


@functools.lru_cache(maxsize=4)
def operands(recipe, M, N, K, seed):
    return si.workload(recipe, M, N, K, seed)


def check_sampled(orc, recipe, M, N, K, seed, config=None):
    A, B, C, alpha, beta, dtype = operands(recipe, M, N, K, seed)
    got, status = run_gpu(dtype, A, B, C, alpha, beta, config=config)
    assert status == 0, f"device status {status}"
    ii, jj = sample_indices(M, N, seed)
    ref = orc.entries(dtype, A, B, C, alpha, beta, ii, jj)
    g = got[ii, jj]
    if dtype == "i8":
        bad = np.flatnonzero(g != ref)
        assert bad.size == 0, f"{bad.size} mismatches, e.g. ({ii[bad[0]]},{jj[bad[0]]}): {g[bad[0]]} vs {ref[bad[0]]}"
    else:
        assert np.all(np.isfinite(got))
        err = float(np.max(np.abs(g.astype(np.float64) - ref)))
        bound = float_bound(A, B, K, dtype)
        assert err <= bound, f"max err {err:g} > bound {bound:g}"


def check_full(orc, recipe, M, N, K, seed, config=None):
    """Every entry of C against the oracle's whole matrix."""
    A, B, C, alpha, beta, dtype = operands(recipe, M, N, K, seed)
    got, status = run_gpu(dtype, A, B, C, alpha, beta, config=config)
    assert status == 0, f"device status {status}"
    ref = orc.gemm(dtype, A, B, C, alpha, beta)
    if dtype == "i8":
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {tuple(bad[0])}"
    else:
        assert np.all(np.isfinite(got))
        err = float(np.max(np.abs(got.astype(np.float64) - ref)))
        bound = float_bound(A, B, K, dtype)
        assert err <= bound, f"max err {err:g} > bound {bound:g}"


def test_fp32_4096_beta_half(orc):
    check_full(orc, "f32_uniform_beta", 4096, 4096, 4096, si.config_seed(2))


def test_fp32_256(orc):
    A, B, C, alpha, beta, dtype = si.workload("f32_uniform", 256, 256, 256, si.config_seed(1))
    got, status = run_gpu(dtype, A, B, C, alpha, beta)
    assert status == 0
    ref = orc.gemm(dtype, A, B, C, alpha, beta)
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    assert err <= float_bound(A, B, 256, dtype)


def test_int8_4096(orc):
    check_full(orc, "i8_uniform", 4096, 4096, 4096, si.config_seed(3))


@pytest.mark.parametrize("bn", [128, 256])
def test_int8_4096_each_tile(orc, bn):
    check_sampled(orc, "i8_uniform", 4096, 4096, 4096, si.config_seed(3), config=(128, bn, 64, 4))


@pytest.mark.parametrize("K", [32, 256, 512])
def test_int8_4096_short_k_default(orc, K):
    """Short-K int8 at 4096^2 takes the default 128 x 256 tiles and the flat
    widening walk (rows of A under 4096 columns); whole matrix, bit-exact."""
    assert pg.pgemm_default_config("i8", 4096, 4096, K)[:2] == (128, 256)
    check_full(orc, "i8_uniform", 4096, 4096, K, si.config_seed(3, K))


def test_bf16_8192(orc):
    check_sampled(orc, "bf16_normal", 8192, 8192, 8192, si.config_seed(4))


@pytest.mark.parametrize("K", [32, 64, 128, 512, 2048, 16384])
def test_bf16_k_sweep_every_config(orc, K):
    for cfg in pg.pgemm_list_configs("bf16"):
        check_sampled(orc, "bf16_normal", 4096, 4096, K, si.config_seed(5, K % 251), config=cfg)


def test_bf16_ragged_every_config(orc):
    for cfg in pg.pgemm_list_configs("bf16"):
        check_sampled(orc, "bf16_normal", 4095, 4097, 4100, si.config_seed(6), config=cfg)


@pytest.mark.parametrize("dtype,recipe", [("f32", "f32_uniform_beta"), ("i8", "i8_uniform")])
def test_ragged_other_dtypes(orc, dtype, recipe):
    check_sampled(orc, recipe, 4095, 4097, 4100, si.config_seed(6, 1))
