"""gemm_i8_noalloc: the int8 GEMM for callers that cannot let the library
allocate device memory (their memory belongs to their own allocator or a
fixed budget, or an allocation call is not allowed or could block where they
call from).  It widens the operands into one fixed device array instead of
per-call scratch; its results must equal gemm_i8's bit for bit (the
tolerance of every int8 test), call after call, and the oracle's.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.  It builds what it needs and runs
alone in a fresh process as well.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

LIMIT = pg.NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    pg.lib()


def _round_up(v, m):
    return (v + m - 1) // m * m


def scratch_needed(M, N, K):
    """Bytes of the widened operands: fp16 A (M rows, K rounded up to 8) and
    fp16 B (K rows, N rounded up to 8), each rounded up to 256 bytes."""
    return (_round_up(2 * M * _round_up(K, 8), 256) + _round_up(2 * K * _round_up(N, 8), 256))


def _operands(M, N, K, seed):
    A = si.uniform_i8((M, K), seed)
    B = si.uniform_i8((K, N), seed + 1)
    C = si.uniform_i8((M, N), seed + 2).astype(np.int32) * 977
    return A, B, C


def _run(fn, M, N, K, alpha, beta, seed):
    A, B, C = _operands(M, N, K, seed)
    dC = torch.from_numpy(C).cuda()
    fn(M, N, K, alpha, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), beta, dC)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    return dC.cpu().numpy()


# Problems back to back, then the first again: each call must match gemm_i8
# exactly, whatever the previous call left in the shared array.  The ragged
# shape (K, N odd) exercises the rounded-up pitches of the widened operands;
# 1024 x 1024 x 8192 is one that gemm_i8 splits along K (stream-K) while this
# entry point, which has no memory for the exchange, does not; so does 2560 x
# 2560 x 2048 on the CTA pair.
RAGGED = (1001, 1003, 2005, 3, -2, 31)
SPLIT = (1024, 1024, 8192, 1, 0, 41)
PAIR = (2560, 2560, 2048, 2, 1, 43)
CASES = [(1000, 1500, 2000, 1, 0, 11), (2048, 777, 3000, -3, 2, 23), RAGGED, SPLIT, PAIR,
         (1000, 1500, 2000, 1, 0, 11)]


def test_noalloc_matches_gemm_i8_on_consecutive_calls():
    assert pg.pgemm_schedule("i8", *SPLIT[:3])["split_tiles"] > 0  # gemm_i8 splits this one
    assert pg.pgemm_schedule("i8", *PAIR[:3])["split_tiles"] > 0
    for (M, N, K, alpha, beta, seed) in CASES:
        assert scratch_needed(M, N, K) <= LIMIT
        want = _run(pg.gemm_i8, M, N, K, alpha, beta, seed)
        got = _run(pg.gemm_i8_noalloc, M, N, K, alpha, beta, seed)
        assert np.array_equal(got, want), f"mismatch for {(M, N, K)}"


def test_noalloc_matches_the_oracle():
    M, N, K, alpha, beta, seed = RAGGED
    A, B, C = _operands(M, N, K, seed)
    want = oracle.get().gemm("i8", A, B, C, alpha, beta)
    got = _run(pg.gemm_i8_noalloc, M, N, K, alpha, beta, seed)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {tuple(bad[0])}"


def test_noalloc_fills_its_array_exactly():
    M, N, K = 2048, 2048, 4096  # 16 MiB of fp16 A + 16 MiB of fp16 B
    assert scratch_needed(M, N, K) == LIMIT
    want = _run(pg.gemm_i8, M, N, K, 1, 0, 53)
    got = _run(pg.gemm_i8_noalloc, M, N, K, 1, 0, 53)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096),   # twice the array
                                   (4550, 1000, 3018)])  # one 256-byte step beyond it
def test_noalloc_rejects_problems_beyond_its_array(M, N, K):
    assert scratch_needed(M, N, K) > LIMIT
    A = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    B = torch.zeros((K, N), dtype=torch.int8, device="cuda")
    C = torch.full((M, N), 5, dtype=torch.int32, device="cuda")
    with pytest.raises(pg.PgemmError) as e:
        pg.gemm_i8_noalloc(M, N, K, 1, A, B, 0, C)
    assert e.value.code == 7
    torch.cuda.synchronize()
    assert bool((C == 5).all())  # nothing was done
