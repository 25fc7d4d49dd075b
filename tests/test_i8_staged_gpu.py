"""The exact int8 kernel on a CTA pair with the staged producer
(pgemm_config.producer = staged): TMA copies the int8 A and B tiles as they
are into a ring of int8 stages, and four warps per CTA widen each landed
stage to fp16 in shared memory, into the fp16 stages the tensor core reads.
No widening pass runs before the GEMM.

The arithmetic after the fp16 ring is the default kernel's, and int8 results
are exact, so every case is bit-exact against the oracle and bit-identical to
the TMA-fed pair kernel after the widening pass: fewer K-tiles than int8
stages, K not a multiple of 16 (rows relaid out to 16-byte pitches; the
bytes past K arrive as TMA zero fill), N not a multiple of 16, M below the
pair's second tile, K = 0, alpha / beta with wrap-around, the all(-128)
extreme, and stream-K pieces.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

STAGED = pg.PRODUCERS["staged"]


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
    return (256, 256, 64, stages, max_parts, STAGED)


def operands(M, N, K, seed):
    return (si.uniform_i8((M, K), seed), si.uniform_i8((K, N), seed + 1),
            si.uniform_i8((M, N), seed + 2).astype(np.int32) * 1000)


@pytest.mark.parametrize("stages", [4, 5, 6])
def test_every_stage_count_and_tile_count(orc, stages):
    # fewer K-tiles than the fp16 ring (2 or 3) and than the int8 ring, and a few more
    for T in sorted({1, 2, stages - 1, stages, stages + 1}):
        for K in (T * 64, T * 64 - 16, T * 64 - 37):
            for M, N in ((2 * 256 + 7, 256 + 24), (300, 384)):
                A, B, C = operands(M, N, K, 5000 + 11 * stages + K + N)
                got, status = run_gpu("i8", A, B, C, 1, 0, config=cfg(stages))
                assert status == 0
                compare("i8", got, orc.gemm("i8", A, B, C, 1, 0), A, B, K)


@pytest.mark.parametrize("M,N,K,alpha,beta", [
    (300, 203, 517, 1, 0),      # K and N off 16: both operands relaid out, tails zero-filled
    (129, 130, 33, -3, 2),      # one K-tile, the pair's second tile below C
    (1, 1, 1, 1, 0),
    (64, 64, 0, 1, 5),          # K = 0: C = beta * C
    (512, 384, 4096, 100, 7),   # four exact rounds; wraps modulo 2^32 in the epilogue
    (1000, 1000, 4100, 1, 0),   # stream-K halves (16 pair tiles on the pairs)
])
@pytest.mark.parametrize("stages", [4, 5, 6])
def test_parity_edges(orc, M, N, K, alpha, beta, stages):
    A, B, C = operands(M, N, K, 5100 + M + K)
    got, status = run_gpu("i8", A, B, C, alpha, beta, config=cfg(stages))
    assert status == 0
    compare("i8", got, orc.gemm("i8", A, B, C, alpha, beta), A, B, K)


def test_extreme_values():
    M, N, K = 300, 272, 4096
    for a, b in ((-128, -128), (127, -128)):
        A = np.full((M, K), a, np.int8)
        B = np.full((K, N), b, np.int8)
        got, status = run_gpu("i8", A, B, np.zeros((M, N), np.int32), 1, 0, config=cfg(6))
        assert status == 0
        assert np.all(got == np.int32(K * a * b))


@pytest.mark.parametrize("max_parts", [0, 1, 8])
def test_stream_k_pieces(orc, max_parts):
    """Halves (the default cap), no split, and finer pieces all give the
    oracle's result."""
    M, N, K = 1000, 1000, 4100
    A, B, C = operands(M, N, K, 5200)
    got, status = run_gpu("i8", A, B, C, 3, -2, config=cfg(5, max_parts))
    assert status == 0
    compare("i8", got, orc.gemm("i8", A, B, C, 3, -2), A, B, K)


def test_equals_tma_pair_full_size():
    """int8 4096^3: bit-identical to the TMA-fed pair kernel after the
    widening pass (itself checked against the oracle at this size)."""
    M = N = K = 4096
    A, B, C = operands(M, N, K, 5300)
    a, sa = run_gpu("i8", A, B, C, 1, 0, config=cfg(6))
    b, sb = run_gpu("i8", A, B, C, 1, 0, config=(256, 256, 64, 6))
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b)


@pytest.mark.parametrize("stages", [4, 5, 6])
def test_back_to_back_calls(orc, stages):
    """Many calls in a row on one stream, each checked bit for bit: a stage
    widened before its copy had landed, or a ring whose phases slipped, would
    show as wrong entries here."""
    M, N, K = 1024, 1024, 4096
    A, B, C = operands(M, N, K, 5400 + stages)
    ref = torch.from_numpy(orc.gemm("i8", A, B, C, 1, 0).astype(np.int32)).cuda()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = [torch.empty((M, N), dtype=torch.int32, device="cuda") for _ in range(4)]
    bad = 0
    for i in range(60):
        out = outs[i % 4]
        out.fill_(-1)
        pg.gemm_i8_ex(M, N, K, 1, dA, dB, 0, out, config=cfg(stages))
        if i % 4 == 3:
            torch.cuda.synchronize()
            bad += sum(int((o != ref).sum().item()) for o in outs)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    assert bad == 0, f"{bad} wrong entries over 60 calls"
