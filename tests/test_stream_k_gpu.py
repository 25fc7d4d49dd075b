"""Parity of the persistent fp32 kernel's stream-K head.

When the output tiles leave a partial last wave, the leftover tiles'
K-iterations are dealt out to every resident block first; each piece stores
its partial sums and the last piece of a tile adds them in slot order and
writes C.  Each case first checks through pgemm_schedule that the head is in
use, then compares with the oracle: bit-exact on integer-valued operands
(every partial sum is an exact integer, so a dropped, doubled or misplaced
piece shows), within 1e-4 * sqrt(K) * max|A| * max|B| on random ones.
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


def operands(M, N, K, seed, kind):
    if kind == "int":
        return (si.small_int_f32((M, K), seed, -4, 4), si.small_int_f32((K, N), seed + 1, -4, 4),
                si.small_int_f32((M, N), seed + 2, -8, 8))
    return (si.uniform_f32((M, K), seed), si.uniform_f32((K, N), seed + 1),
            si.uniform_f32((M, N), seed + 2))


def head(M, N, K, config=None):
    s = pg.pgemm_schedule("f32", M, N, K, config)
    return s["split_tiles"], s


@pytest.mark.parametrize("cfg", [None, (128, 128, 32, 2), (128, 128, 32, 6), (128, 64, 32, 3),
                                 (128, 128, 32, 1)])
@pytest.mark.parametrize("M,N,K,kind,alpha,beta", [
    (300, 520, 8200, "int", 1.0, 0.0),      # W = 0: every tile spread over many blocks, K tail
    (1037, 1100, 2052, "int", 1.0, 0.5),    # ragged edges, beta != 0, repacked pitches
    (777, 640, 3000, "random", 0.75, -0.25),
])
def test_stream_k_parity(orc, cfg, M, N, K, kind, alpha, beta):
    sk, s = head(M, N, K, cfg)
    assert sk > 0, s
    A, B, C = operands(M, N, K, 5000 + M + K, kind)
    got, status = run_gpu("f32", A, B, C, alpha, beta, config=cfg)
    assert status == 0
    compare("f32", got, orc.gemm("f32", A, B, C, alpha, beta), A, B, K, exact=(kind == "int"))


def test_many_pieces_per_tile(orc):
    """A handful of output tiles dealt out to every resident block: each tile
    in more than fifty pieces."""
    M, N, K = 256, 256, 65536
    sk, s = head(M, N, K)
    assert sk == s["tiles"] and s["parts"] >= 50, s
    A, B, C = operands(M, N, K, 5100, "int")
    got, status = run_gpu("f32", A, B, C, 1.0, 0.0)
    assert status == 0
    compare("f32", got, orc.gemm("f32", A, B, C, 1.0, 0.0), A, B, K, exact=True)


def test_head_off_matches_within_bound_and_repeats_bitwise(orc):
    M, N, K = 1100, 1200, 2000
    sk, _ = head(M, N, K)
    assert sk > 0
    A, B, C = operands(M, N, K, 5200, "random")
    on1, s1 = run_gpu("f32", A, B, C, 1.0, 0.5)
    on2, s2 = run_gpu("f32", A, B, C, 1.0, 0.5)
    off, s3 = run_gpu("f32", A, B, C, 1.0, 0.5, config=(128, 128, 32, 3, 1))
    assert s1 == s2 == s3 == 0
    assert head(M, N, K, (128, 128, 32, 3, 1))[0] == 0
    # the pieces are added in slot order: the same bits every call
    assert np.array_equal(on1.view(np.uint32), on2.view(np.uint32))
    ref = orc.gemm("f32", A, B, C, 1.0, 0.5)
    compare("f32", on1, ref, A, B, K)
    compare("f32", off, ref, A, B, K)


def test_back_to_back_calls_stay_exact(orc):
    """The tickets and partial slots are per call (stream-ordered scratch):
    many calls queued on one stream each give the exact integer result."""
    M, N, K = 700, 900, 3000
    sk, _ = head(M, N, K)
    assert sk > 0
    A, B, C = operands(M, N, K, 5300, "int")
    ref = torch.from_numpy(orc.gemm("f32", A, B, C, 1.0, 0.0).astype(np.float32)).cuda()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(4)]
    bad = 0
    for i in range(100):
        outs[i % 4].fill_(float("nan"))
        pg.gemm_f32(M, N, K, 1.0, dA, dB, 0.0, outs[i % 4])
        if i % 4 == 3:
            torch.cuda.synchronize()
            bad += sum(int((o != ref).sum().item()) for o in outs)
    assert pg.pgemm_get_device_status() == 0
    assert bad == 0


def test_bench_shape_uses_the_head():
    sk, s = head(4096, 4096, 4096)
    rem = s["tiles"] % s["slots"]
    assert sk == (rem if rem else 0), s
