"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small and medium shapes are compared element by element; they span several
output tiles and ragged M, N and K tails.  Integer-valued float operands must
match bit for bit (every partial sum is an exact integer, so a dropped or
repeated K-tile cannot hide inside the tolerance -- the pitfall "GPU-Kernel
pipelinen" warns about under "Haeufige Stolperfallen").  Random float
operands must meet max|C - C_ref| <= 1e-4 * sqrt(K) * max|A| * max|B|; int8 is
bit-exact.  The K sweep covers T = 0, 1, S-1, S, S+1 and more K-tiles for
every built stage count S ("Software pipelines and asynchronous copies",
section "Prologue, steady state, and epilogue": fewer K-tiles than stages must
work).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    pg.lib()
    assert pg.pgemm_get_device_status() == 0


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def operands(dtype, M, N, K, seed, kind="random", beta=0.0):
    """Seeded host operands.  kind: random | int (integer-valued floats)."""
    if dtype == "i8":
        A = si.uniform_i8((M, K), seed)
        B = si.uniform_i8((K, N), seed + 1)
        C = si.uniform_i8((M, N), seed + 2).astype(np.int32) * 1000
        return A, B, C
    if kind == "int":
        Af = si.small_int_f32((M, K), seed, -4, 4)
        Bf = si.small_int_f32((K, N), seed + 1, -4, 4)
        C = si.small_int_f32((M, N), seed + 2, -8, 8)
    else:
        Af = si.uniform_f32((M, K), seed) if dtype == "f32" else si.normal_f32((M, K), seed)
        Bf = si.uniform_f32((K, N), seed + 1) if dtype == "f32" else si.normal_f32((K, N), seed + 1)
        C = si.uniform_f32((M, N), seed + 2)
    if dtype == "bf16":
        return si.to_bf16_bits(Af), si.to_bf16_bits(Bf), C
    return Af, Bf, C


def check(orc, dtype, M, N, K, alpha, beta, seed, kind="random", config=None):
    A, B, C = operands(dtype, M, N, K, seed, kind)
    ref = orc.gemm(dtype, A, B, C, alpha, beta)
    got, status = run_gpu(dtype, A, B, C, alpha, beta, config=config)
    assert status == 0, f"device status {status}"
    compare(dtype, got, ref, A, B, K, exact=(kind == "int"))


# ---------------------------------------------------------------- basics ----
@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (1, 1, 1), (300, 520, 200), (257, 129, 1000), (67, 77, 131), (33, 1001, 70),
                                   (64, 1000, 96), (130, 136, 8)])
def test_small_random(orc, dtype, M, N, K):
    check(orc, dtype, M, N, K, 1, 0, seed=1000 + M + N + K)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
@pytest.mark.parametrize("M,N,K", [
    (1, 4097, 3000),     # one row; B's pitch odd (repacked / widened with padding)
    (3000, 1, 4100),     # one column: C's pitch 1 element (no TMA store), K ragged
    (1, 1, 65536),       # one output: its single tile cut along K by stream-K
    (2, 8192, 512),
    (8192, 2, 512),
])
def test_vector_like_shapes(orc, dtype, M, N, K):
    check(orc, dtype, M, N, K, 1, 0, seed=3000 + M + N + K)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 200), (257, 129, 1000)])
def test_small_integer_valued_is_bit_exact(orc, dtype, M, N, K):
    check(orc, dtype, M, N, K, 1, 0, seed=2000 + M + N + K, kind="int")


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
def test_alpha_beta(orc, dtype):
    if dtype == "i8":
        check(orc, dtype, 200, 300, 130, 3, -2, seed=31)
        check(orc, dtype, 200, 300, 130, -7, 5, seed=32)
    else:
        check(orc, dtype, 200, 300, 130, 1.5, 0.5, seed=31)
        check(orc, dtype, 200, 300, 130, -0.25, 2.0, seed=32, kind="int")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_beta_zero_does_not_read_c(orc, dtype):
    M, N, K = 160, 200, 96
    A, B, _ = operands(dtype, M, N, K, 41)
    C = np.full((M, N), np.nan, np.float32)
    ref = orc.gemm(dtype, A, B, None, 1.0, 0.0)
    got, status = run_gpu(dtype, A, B, C, 1.0, 0.0)
    assert status == 0
    compare(dtype, got, ref, A, B, K)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_beta_zero_does_not_read_c_on_stream_k_shapes(orc, dtype):
    """The stream-K paths (bf16: pieces exchanging partial sums; fp32: the tail
    grid reducing its pieces into C) must not read C either when beta = 0."""
    M, N, K = 1000, 1000, 4100
    A, B, _ = operands(dtype, M, N, K, 42)
    C = np.full((M, N), np.nan, np.float32)
    ref = orc.gemm(dtype, A, B, None, 1.0, 0.0)
    got, status = run_gpu(dtype, A, B, C, 1.0, 0.0)
    assert status == 0
    compare(dtype, got, ref, A, B, K)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
def test_alpha_zero_beta_one_returns_c(orc, dtype):
    M, N, K = 1000, 1000, 4100  # stream-K shapes: every path applies alpha and beta
    A, B, C = operands(dtype, M, N, K, 43)
    got, status = run_gpu(dtype, A, B, C, 0, 1)
    assert status == 0
    compare(dtype, got, orc.gemm(dtype, A, B, C, 0, 1), A, B, K, exact=True)
    assert np.array_equal(got.view(np.uint32), np.asarray(C).view(np.uint32))


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
def test_k_zero(orc, dtype):
    M, N = 150, 260
    A, B, C = operands(dtype, M, N, 0, 51)
    beta = 3 if dtype == "i8" else 0.75
    ref = orc.gemm(dtype, A, B, C, 2, beta)
    got, status = run_gpu(dtype, A, B, C, 2, beta)
    assert status == 0
    compare(dtype, got, ref, A, B, 0, exact=True)


def test_timeout_selftest_reports_and_context_survives(orc):
    assert pg.pgemm_selftest_wait_timeout(2000) == 5  # PGEMM_ERR_TIMEOUT
    assert pg.pgemm_get_device_status() == 0  # cleared
    check(orc, "bf16", 128, 128, 64, 1, 0, seed=61, kind="int")


# ------------------------------------------------ stage sweep: T vs S -------
def _configs(dtype):
    return pg.pgemm_list_configs(dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
def test_every_config_every_tile_count(orc, dtype):
    """For every built (tile, S): K-tile counts T = 1, S-1, S, S+1, 2S+1 plus a
    K tail; shapes of several tiles in M and N with ragged edges."""
    for cfg in _configs(dtype):
        bm, bn, bk, S = cfg[:4]
        # the in-kernel widening reads int8 rows as 16-byte vectors: K and N
        # multiples of 16 there (still a K tail within the last K-tile)
        aligned = len(cfg) > 5 and cfg[5] == pg.PRODUCERS["widen_in_kernel"]
        for T in sorted({1, max(S - 1, 1), S, S + 1, 2 * S + 1}):
            for K in (T * bk, T * bk - bk // 2 if T > 1 else bk - (16 if aligned else 3)):
                M, N = 2 * bm + 7, 2 * bn + (32 if aligned else 24)
                kind = "random" if dtype == "i8" else "int"
                check(orc, dtype, M, N, K, 1, 0, seed=7000 + 13 * S + T + K, kind=kind,
                      config=cfg)


@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_two_subtile_stages_ragged_k(orc, dtype):
    """Stages of 128 K columns land two 64-column sub-tiles under one barrier.
    In the last stage a sub-tile that starts at or beyond K is neither loaded
    nor multiplied (K mod 128 in [1, 64]), one that starts below K is
    zero-filled past it (K mod 128 in [65, 127]); exact on integer operands."""
    cfgs = [c for c in _configs(dtype) if c[0] == 256 and c[2] == 128]
    assert cfgs
    for cfg in cfgs:
        for K in (1, 63, 64, 65, 127, 129, 3 * 128 + 1, 3 * 128 + 64, 3 * 128 + 100, 1024 + 64):
            check(orc, dtype, 300, 520, K, 1, 0, seed=7500 + K + cfg[3],
                  kind="random" if dtype == "i8" else "int", config=cfg)


@pytest.mark.parametrize("K", [1024, 1025, 2048 + 64, 4096])
def test_int8_extremes_on_two_subtile_stages(orc, K):
    """The exact rounds of 1024 products are eight 128-column stages: a round
    boundary, one column past it, and a ragged last stage, at the products'
    extremes."""
    M, N = 300, 520
    for cfg in [c for c in _configs("i8") if c[0] == 256 and c[2] == 128]:
        for a, b in ((-128, -128), (127, -128)):
            A = np.full((M, K), a, np.int8)
            B = np.full((K, N), b, np.int8)
            C = np.zeros((M, N), np.int32)
            got, status = run_gpu("i8", A, B, C, 1, 0, config=cfg)
            assert status == 0
            assert np.all(got == np.int32(K * a * b)), (cfg, K, a, b)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
def test_persistent_multi_tile_per_block(orc, dtype):
    """More output tiles than resident blocks: each block runs several tiles
    (ring phases and, on the tensor-core paths, both TMEM accumulators wrap)."""
    M, N, K = 2048 + 64, 2048 + 8, 320
    A, B, C = operands(dtype, M, N, K, 81, kind="random" if dtype == "i8" else "int")
    got, status = run_gpu(dtype, A, B, C, 1, 0)
    assert status == 0
    ref = orc.gemm(dtype, A, B, C, 1, 0)
    compare(dtype, got, ref, A, B, K, exact=True)


# -------------------------------------------------------------- int8 exact ----
@pytest.mark.parametrize("K", [1, 255, 256, 257, 1023, 1024, 1025, 2049, 4096])
def test_int8_extremes_bit_exact(orc, K):
    M, N = 130, 136
    for a, b in ((-128, -128), (127, 127), (-128, 127)):
        A = np.full((M, K), a, np.int8)
        B = np.full((K, N), b, np.int8)
        C = np.zeros((M, N), np.int32)
        got, status = run_gpu("i8", A, B, C, 1, 0)
        assert status == 0
        assert np.all(got == np.int32(K * a * b))


def test_int8_wraparound(orc):
    M, N, K = 140, 150, 4096
    A = np.full((M, K), -128, np.int8)
    B = np.full((K, N), -128, np.int8)
    C = si.uniform_i8((M, N), 5).astype(np.int32) * 12345
    ref = orc.gemm("i8", A, B, C, 100, 7)
    got, status = run_gpu("i8", A, B, C, 100, 7)
    assert status == 0
    compare("i8", got, ref, A, B, K)
