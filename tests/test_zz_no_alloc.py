"""gemm_i8_noalloc: the int8 GEMM for callers that cannot let the library
allocate device memory (their memory belongs to their own allocator or a
fixed budget, or an allocation call is not allowed or could block where they
call from).  It widens the operands into one fixed device array instead of
per-call scratch; its results must equal gemm_i8's bit for bit (the
tolerance of every int8 test), call after call.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.  It builds what it needs and runs
alone in a fresh process as well.
"""
import numpy as np
import pytest

import seeded_inputs as si

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


def _run(fn, M, N, K, alpha, beta, seed):
    A = torch.from_numpy(si.uniform_i8((M, K), seed)).cuda()
    B = torch.from_numpy(si.uniform_i8((K, N), seed + 1)).cuda()
    C = torch.from_numpy(si.uniform_i8((M, N), seed + 2).astype(np.int32) * 977).cuda()
    fn(M, N, K, alpha, A, B, beta, C)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    return C.cpu().numpy()


# two different problems back to back, then the first again: each call must
# match gemm_i8 exactly, whatever the previous call left in the shared array
CASES = [(1000, 1500, 2000, 1, 0, 11), (2048, 777, 3000, -3, 2, 23), (1000, 1500, 2000, 1, 0, 11)]


def test_noalloc_matches_gemm_i8_on_consecutive_calls():
    for (M, N, K, alpha, beta, seed) in CASES:
        want = _run(pg.gemm_i8, M, N, K, alpha, beta, seed)
        got = _run(pg.gemm_i8_noalloc, M, N, K, alpha, beta, seed)
        assert np.array_equal(got, want), f"mismatch for {(M, N, K)}"


def test_noalloc_rejects_problems_beyond_its_array():
    M = N = K = 4096  # 2 * (4096*4096 + 4096*4096) bytes = 64 MiB > 32 MiB
    A = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    B = torch.zeros((K, N), dtype=torch.int8, device="cuda")
    C = torch.full((M, N), 5, dtype=torch.int32, device="cuda")
    with pytest.raises(pg.PgemmError) as e:
        pg.gemm_i8_noalloc(M, N, K, 1, A, B, 0, C)
    assert e.value.code == 7
    torch.cuda.synchronize()
    assert bool((C == 5).all())  # nothing was done
