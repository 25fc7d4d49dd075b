"""The mma.sync int8 engine (pgemm_config.engine = mma_sync): warp-level
s8 x s8 -> s32 MMAs on the int8 operands, B transposed by a pre-pass, on the
same TMA ring.  Exact by construction, so every case is bit-exact against the
oracle and bit-identical to the default (exact-fp16 tcgen05) engine: ragged
M, N, K (the A repack and the B transpose at odd pitches), fewer K-tiles than
stages, K = 0, alpha / beta with wrap-around, the all(-128) extreme.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

ENG = pg.ENGINES["mma_sync"]


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


def cfg(stages):
    return (128, 128, 128, stages, 0, 0, ENG)


def operands(M, N, K, seed):
    return (si.uniform_i8((M, K), seed), si.uniform_i8((K, N), seed + 1),
            si.uniform_i8((M, N), seed + 2).astype(np.int32) * 1000)


@pytest.mark.parametrize("stages", [2, 3, 4, 6])
def test_every_stage_count_and_tile_count(orc, stages):
    for T in sorted({1, max(stages - 1, 1), stages, stages + 1}):
        for K in (T * 128, T * 128 - 37):
            M, N = 2 * 128 + 7, 2 * 128 + 24
            A, B, C = operands(M, N, K, 3000 + 7 * stages + K)
            got, status = run_gpu("i8", A, B, C, 1, 0, config=cfg(stages))
            assert status == 0
            compare("i8", got, orc.gemm("i8", A, B, C, 1, 0), A, B, K)


@pytest.mark.parametrize("M,N,K,alpha,beta", [
    (300, 203, 517, 1, 0),      # A pitch 517 (repacked), odd N (B^T rows, scalar C edge)
    (129, 130, 33, -3, 2),      # one K-tile, partial
    (1, 1, 1, 1, 0),
    (64, 64, 0, 1, 5),          # K = 0: C = beta * C
    (512, 384, 4096, 100, 7),   # wraps modulo 2^32 in the epilogue
])
def test_parity_edges(orc, M, N, K, alpha, beta):
    A, B, C = operands(M, N, K, 3100 + M + K)
    got, status = run_gpu("i8", A, B, C, alpha, beta, config=cfg(4))
    assert status == 0
    compare("i8", got, orc.gemm("i8", A, B, C, alpha, beta), A, B, K)


def test_extreme_values():
    M, N, K = 130, 136, 4096
    for a, b in ((-128, -128), (127, -128)):
        A = np.full((M, K), a, np.int8)
        B = np.full((K, N), b, np.int8)
        got, status = run_gpu("i8", A, B, np.zeros((M, N), np.int32), 1, 0, config=cfg(4))
        assert status == 0
        assert np.all(got == np.int32(K * a * b))


def test_equals_default_engine():
    M, N, K = 1000, 1000, 3000
    A, B, C = operands(M, N, K, 3200)
    a, sa = run_gpu("i8", A, B, C, 3, -2, config=cfg(4))
    b, sb = run_gpu("i8", A, B, C, 3, -2)
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b)
