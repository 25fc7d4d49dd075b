"""Maximum sizes: an output of more than 2^31 elements (65536 x 32832, 8.6 GB
of fp32 or int32), so that row offsets into C, and the TMA coordinates of
the last rows, pass the 32-bit range.  Whole rows near the top, the middle
and the bottom are gathered on the device and compared with the oracle run
on the same rows of A (the rows of a GEMM are independent).  fp32 uses
beta = 0.5 on C = 1 everywhere, so C is read at those offsets too."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_harness import compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

M, N, K = 65536, 32832, 64
ROWS = [0, 1, M // 2 - 1, M // 2, M - 2, M - 1]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 12 << 30:
        pytest.skip("needs 12 GB of free device memory")
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    pg.lib()
    assert pg.pgemm_get_device_status() == 0


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i8"])
def test_output_beyond_2_31_elements(orc, dtype):
    assert M * N > 2 ** 31 and (M - 1) * N > 2 ** 31
    seed = 9100 + ["f32", "bf16", "i8"].index(dtype)
    if dtype == "i8":
        A = si.uniform_i8((M, K), seed)
        B = si.uniform_i8((K, N), seed + 1)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.empty((M, N), dtype=torch.int32, device="cuda")
        alpha, beta, C0 = 1, 0, None
    elif dtype == "bf16":
        A = si.to_bf16_bits(si.normal_f32((M, K), seed))
        B = si.to_bf16_bits(si.normal_f32((K, N), seed + 1))
        dA = torch.from_numpy(A.view(np.int16)).cuda()
        dB = torch.from_numpy(B.view(np.int16)).cuda()
        dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
        alpha, beta, C0 = 1.0, 0.0, None
    else:
        A = si.uniform_f32((M, K), seed)
        B = si.uniform_f32((K, N), seed + 1)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.ones((M, N), dtype=torch.float32, device="cuda")
        alpha, beta, C0 = 1.0, 0.5, np.ones((len(ROWS), N), np.float32)
    getattr(pg, f"gemm_{dtype}")(M, N, K, alpha, dA, dB, beta, dC)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    got = dC[torch.tensor(ROWS, device="cuda")].cpu().numpy()
    del dC
    torch.cuda.empty_cache()
    ref = orc.gemm(dtype, A[ROWS], B, C0, alpha, beta)
    compare(dtype, got, ref, A[ROWS], B, K)
