"""The register-staged fp32 comparator (pgemm_config.producer = registers).

It runs the same block tile, register tile and FFMA2 sequence as the TMA
kernel with two buffers; only who fills the buffers differs.  So besides
oracle parity (bit-exact on integer-valued operands, within
1e-4 * sqrt(K) * max|A| * max|B| on random ones, ragged M, N, K with the
element-wise edge loads, beta != 0, K = 0), its result must equal the TMA
kernel's with the same tile bit for bit: the products are summed in the same
order.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

REG = pg.PRODUCERS["registers"]


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


@pytest.mark.parametrize("bn", [128, 64])
@pytest.mark.parametrize("M,N,K,kind,alpha,beta", [
    (256, 256, 64, "int", 1.0, 0.0),          # two K-tiles
    (300, 203, 517, "int", 1.0, 0.5),         # ragged M, N (N % 4 != 0), K tail, repacked pitches
    (129, 130, 33, "int", 2.0, -1.0),         # one full K-tile plus one column
    (520, 264, 1000, "random", 0.75, 0.25),
    (64, 64, 0, "random", 1.0, 0.5),          # K = 0: C = beta * C
    (1, 1, 1, "int", 1.0, 0.0),
])
def test_regstage_parity(orc, bn, M, N, K, kind, alpha, beta):
    A, B, C = operands(M, N, K, 900 + M + K, kind)
    cfg = (128, bn, 32, 2, 0, REG)
    got, status = run_gpu("f32", A, B, C, alpha, beta, config=cfg)
    assert status == 0
    ref = orc.gemm("f32", A, B, C, alpha, beta)
    compare("f32", got, ref, A, B, K, exact=(kind == "int"))


@pytest.mark.parametrize("bn", [128, 64])
def test_regstage_equals_tma_kernel_bitwise(bn):
    M, N, K = 1000, 1000, 1000
    A, B, C = operands(M, N, K, 950, "random")
    a, st_a = run_gpu("f32", A, B, C, 1.0, 0.5, config=(128, bn, 32, 2, 0, REG))
    # the TMA kernel without its stream-K head, which would add pieces in another order
    b, st_b = run_gpu("f32", A, B, C, 1.0, 0.5, config=(128, bn, 32, 2, 1))
    assert st_a == 0 and st_b == 0
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_regstage_is_fp32_only():
    with pytest.raises(pg.PgemmError):
        d = torch.zeros(64 * 64, dtype=torch.int16, device="cuda")
        c = torch.zeros(64 * 64, dtype=torch.float32, device="cuda")
        pg.gemm_bf16_ex(64, 64, 64, 1.0, d, d, 0.0, c, config=(128, 128, 64, 2, 0, REG))
