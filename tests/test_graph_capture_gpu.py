"""The library's calls inside a CUDA graph: each call's stream work (the
stream-ordered scratch allocation and free, the counter memset, the
widening or repack pre-pass, the GEMM launched programmatically after it)
is captured once and replayed; every replay must give the direct call's
result bit for bit (int8 exact; the float kernels add in a fixed order)."""
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
    assert pg.pgemm_get_device_status() == 0


def operands(dtype, M, N, K, seed):
    if dtype == "i8":
        return (torch.from_numpy(si.uniform_i8((M, K), seed)).cuda(),
                torch.from_numpy(si.uniform_i8((K, N), seed + 1)).cuda(),
                torch.zeros((M, N), dtype=torch.int32, device="cuda"), 1, 0)
    if dtype == "bf16":
        return (torch.from_numpy(si.to_bf16_bits(si.normal_f32((M, K), seed)).view(np.int16)).cuda(),
                torch.from_numpy(si.to_bf16_bits(si.normal_f32((K, N), seed + 1)).view(np.int16)).cuda(),
                torch.zeros((M, N), dtype=torch.float32, device="cuda"), 1.0, 0.0)
    return (torch.from_numpy(si.uniform_f32((M, K), seed)).cuda(),
            torch.from_numpy(si.uniform_f32((K, N), seed + 1)).cuda(),
            torch.from_numpy(si.uniform_f32((M, N), seed + 2)).cuda(), 1.0, 0.5)


@pytest.mark.parametrize("dtype,M,N,K", [
    ("i8", 1000, 1000, 4100),    # widening pass + programmatic GEMM launch + stream-K halves
    ("bf16", 1000, 1000, 4100),  # A repacked (odd pitch) + stream-K counters memset
    ("bf16", 4096, 4096, 64),    # short K, no pre-pass
    ("f32", 1000, 1000, 4100),   # whole-tile grid + stream-K tail grid
])
def test_calls_replay_in_a_cuda_graph(dtype, M, N, K):
    fn = getattr(pg, f"gemm_{dtype}")
    A, B, C0, alpha, beta = operands(dtype, M, N, K, 7000 + K)
    C = C0.clone()
    fn(M, N, K, alpha, A, B, beta, C)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    direct = C.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # the warm-up torch asks for before a capture
        C.copy_(C0)
        fn(M, N, K, alpha, A, B, beta, C)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn(M, N, K, alpha, A, B, beta, C)
    for _ in range(3):
        C.copy_(C0)
        graph.replay()
        torch.cuda.synchronize()
        assert pg.pgemm_get_device_status() == 0
        assert torch.equal(C.view(torch.int32), direct.view(torch.int32))
