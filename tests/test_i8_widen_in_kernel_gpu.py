"""The exact int8 kernel on a CTA pair with the widening inside the GEMM
(pgemm_config.producer = widen_in_kernel): every CTA TMA-loads its share of
A's and B's int8 boxes, K chunk by K chunk, four of its warps widen them
into the fp16 copies, and the TMA producer of the GEMM loads from a chunk
once every CTA has published its share of it.

The arithmetic after the widening is the default kernel's, and int8 results
are exact, so every case is bit-exact against the oracle and bit-identical to
the kernel after the widening pass: fewer K-tiles than stages, a last K chunk
narrower than 64 (K a multiple of 16 only), ragged M and N, M below the
pair's second tile, K = 0, alpha / beta with wrap-around, the all(-128)
extreme, stream-K pieces, and back-to-back calls whose counters must start
from zero again.  K or N not a multiple of 16 is refused (int8 rows must be
16-byte aligned for the widening's vector loads).
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

WIK = pg.PRODUCERS["widen_in_kernel"]


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


def cfg(stages, max_parts=0):
    return (256, 256, 64, stages, max_parts, WIK)


def operands(M, N, K, seed):
    return (si.uniform_i8((M, K), seed), si.uniform_i8((K, N), seed + 1),
            si.uniform_i8((M, N), seed + 2).astype(np.int32) * 1000)


@pytest.mark.parametrize("stages", [4, 5])
def test_every_tile_count(orc, stages):
    for T in sorted({1, 2, stages - 1, stages, stages + 1}):
        for K in (T * 64, T * 64 - 16, T * 64 - 48):
            if K <= 0:
                continue
            for M, N in ((2 * 256 + 7, 256 + 32), (300, 384)):
                A, B, C = operands(M, N, K, 6000 + 11 * stages + K + N)
                got, status = run_gpu("i8", A, B, C, 1, 0, config=cfg(stages))
                assert status == 0
                compare("i8", got, orc.gemm("i8", A, B, C, 1, 0), A, B, K)


@pytest.mark.parametrize("M,N,K,alpha,beta", [
    (300, 208, 528, 1, 0),      # N a multiple of 16, not of 64; a 16-wide last K chunk
    (129, 144, 48, -3, 2),      # one narrow K chunk, the pair's second tile below C
    (1, 16, 16, 1, 0),
    (64, 64, 0, 1, 5),          # K = 0: C = beta * C, nothing widened
    (512, 384, 4096, 100, 7),   # four exact rounds; wraps modulo 2^32 in the epilogue
    (1000, 1008, 4112, 1, 0),   # stream-K halves and a 16-wide last chunk
    (2560, 2560, 3072, 3, -1),  # stream-K (24 leftover tiles on 76 pairs)
])
@pytest.mark.parametrize("stages", [4, 5])
def test_parity_edges(orc, M, N, K, alpha, beta, stages):
    A, B, C = operands(M, N, K, 6100 + M + K)
    got, status = run_gpu("i8", A, B, C, alpha, beta, config=cfg(stages))
    assert status == 0
    compare("i8", got, orc.gemm("i8", A, B, C, alpha, beta), A, B, K)


def test_extreme_values():
    M, N, K = 300, 272, 4096
    for a, b in ((-128, -128), (127, -128)):
        A = np.full((M, K), a, np.int8)
        B = np.full((K, N), b, np.int8)
        got, status = run_gpu("i8", A, B, np.zeros((M, N), np.int32), 1, 0, config=cfg(5))
        assert status == 0
        assert np.all(got == np.int32(K * a * b))


@pytest.mark.parametrize("max_parts", [0, 1, 8])
def test_stream_k_pieces(orc, max_parts):
    M, N, K = 1000, 1008, 4112
    A, B, C = operands(M, N, K, 6200)
    got, status = run_gpu("i8", A, B, C, 3, -2, config=cfg(5, max_parts))
    assert status == 0
    compare("i8", got, orc.gemm("i8", A, B, C, 3, -2), A, B, K)


def test_repeated_calls(orc):
    """Each call's chunk counters start from zero: three calls in a row on
    the same operands give the same (oracle) result."""
    M, N, K = 700, 512, 2048
    A, B, C = operands(M, N, K, 6300)
    got, status = run_gpu("i8", A, B, C, 1, 0, config=cfg(5), repeat=3)
    assert status == 0
    compare("i8", got, orc.gemm("i8", A, B, C, 1, 0), A, B, K)


@pytest.mark.parametrize("M,N,K", [(256, 256, 100), (256, 200, 256)])
def test_refuses_rows_not_16_byte_aligned(M, N, K):
    A, B, C = operands(M, N, K, 6400)
    with pytest.raises(pg.PgemmError) as e:
        run_gpu("i8", A, B, C, 1, 0, config=cfg(5))
    assert e.value.code == 6


def test_equals_widening_pass_full_size():
    """int8 4096^3: bit-identical to the pair kernel after the widening pass
    (itself checked against the oracle on every entry at this size)."""
    M = N = K = 4096
    A, B, C = operands(M, N, K, 6500)
    a, sa = run_gpu("i8", A, B, C, 1, 0, config=cfg(5))
    b, sb = run_gpu("i8", A, B, C, 1, 0, config=(256, 256, 64, 6))
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b)
