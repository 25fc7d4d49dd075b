"""Calls from several host threads on their own streams at once: each call's
stream-K exchange area, counters and widened operands are its own (stream-
ordered scratch from the library's pool), so concurrent calls must give the
same bits as the same calls made one at a time."""
import threading

import numpy as np
import pytest

import seeded_inputs as si

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

M, N, K = 1000, 1000, 4100  # stream-K halves (128 x 128 tiles) for both tensor-core dtypes


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    pg.lib()
    assert pg.pgemm_get_device_status() == 0


def device_operands(dtype, seed):
    if dtype == "i8":
        return (torch.from_numpy(si.uniform_i8((M, K), seed)).cuda(),
                torch.from_numpy(si.uniform_i8((K, N), seed + 1)).cuda(), torch.int32, 1, 0)
    return (torch.from_numpy(si.to_bf16_bits(si.normal_f32((M, K), seed)).view(np.int16)).cuda(),
            torch.from_numpy(si.to_bf16_bits(si.normal_f32((K, N), seed + 1)).view(np.int16)).cuda(),
            torch.float32, 1.0, 0.0)


def test_threads_on_their_own_streams_match_serial_calls():
    jobs = [("bf16", 8100), ("i8", 8200), ("bf16", 8300), ("i8", 8400)]
    ops = {seed: device_operands(dtype, seed) for dtype, seed in jobs}
    ref = {}
    for dtype, seed in jobs:
        A, B, ct, alpha, beta = ops[seed]
        C = torch.empty((M, N), dtype=ct, device="cuda")
        getattr(pg, f"gemm_{dtype}")(M, N, K, alpha, A, B, beta, C)
        torch.cuda.synchronize()
        ref[seed] = C.clone()
    assert pg.pgemm_get_device_status() == 0

    calls = 12
    outs = {seed: [torch.empty((M, N), dtype=ops[seed][2], device="cuda") for _ in range(calls)]
            for _, seed in jobs}
    errors = []

    def worker(dtype, seed):
        try:
            stream = torch.cuda.Stream()
            A, B, _, alpha, beta = ops[seed]
            with torch.cuda.stream(stream):
                for i in range(calls):
                    getattr(pg, f"gemm_{dtype}")(M, N, K, alpha, A, B, beta, outs[seed][i],
                                                 stream=stream)
            stream.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=job) for job in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    for _, seed in jobs:
        for i, out in enumerate(outs[seed]):
            assert torch.equal(out.view(torch.int32), ref[seed].view(torch.int32)), (seed, i)
