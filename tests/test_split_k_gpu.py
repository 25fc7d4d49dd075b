"""Parity of the K-split last wave of the persistent tensor-core kernels.

When the output tiles leave the last wave of the persistent grid at most half
full, each tile of that wave is cut along K into parts whose partial sums are
added by the part that finishes last.  These tests run shapes where the
schedule splits (checked through pgemm_schedule first, so a test cannot pass
by not splitting) and compare with the oracle: bit-exact for int8 and for
integer-valued floats (a dropped, doubled or misplaced K range changes an
exact integer), within 1e-4 * sqrt(K) * max|A| * max|B| for random bf16.  The
fp32 sum of the parts is taken in part order, so repeated calls give the same
bits however the parts finish.
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


def operands(dtype, M, N, K, seed, kind):
    if dtype == "i8":
        return (si.uniform_i8((M, K), seed), si.uniform_i8((K, N), seed + 1),
                si.uniform_i8((M, N), seed + 2).astype(np.int32) * 1000)
    if kind == "int":
        Af = si.small_int_f32((M, K), seed, -4, 4)
        Bf = si.small_int_f32((K, N), seed + 1, -4, 4)
        C = si.small_int_f32((M, N), seed + 2, -8, 8)
    else:
        Af = si.normal_f32((M, K), seed)
        Bf = si.normal_f32((K, N), seed + 1)
        C = si.uniform_f32((M, N), seed + 2)
    return si.to_bf16_bits(Af), si.to_bf16_bits(Bf), C


def splits(dtype, M, N, K, config=None):
    s = pg.pgemm_schedule(dtype, M, N, K, config)
    return s["split_tiles"] > 0 and s["parts"] >= 2, s


def check(orc, dtype, M, N, K, seed, kind="random", alpha=1, beta=0, config=None):
    A, B, C = operands(dtype, M, N, K, seed, kind)
    got, status = run_gpu(dtype, A, B, C, alpha, beta, config=config)
    assert status == 0, f"device status {status}"
    ref = orc.gemm(dtype, A, B, C, alpha, beta)
    compare(dtype, got, ref, A, B, K, exact=(dtype == "i8" or kind == "int"))
    return got


# K = 4100: 65 K-tiles, four 16-tile granules, so up to four parts, the last
# one with the ragged 17th tile.
@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_every_config_splits_exactly(orc, dtype):
    for cfg in pg.pgemm_list_configs(dtype):
        if len(cfg) > 4:  # another producer or engine: not a persistent tensor-core kernel
            continue
        M, N, K = (300, 200, 4100) if cfg[0] == 256 else (250, 260, 4100)
        ok, s = splits(dtype, M, N, K, cfg)
        assert ok, (cfg, s)
        check(orc, dtype, M, N, K, si.config_seed(20, cfg[1] % 251 + cfg[3]), kind="int",
              alpha=1 if dtype == "i8" else 1.0, beta=0 if dtype == "i8" else 0.0, config=cfg)


@pytest.mark.parametrize("max_parts", [2, 3, 8])
def test_part_caps(orc, max_parts):
    cfg = (128, 128, 64, 4, max_parts)
    ok, s = splits("bf16", 512, 512, 8192, cfg)
    assert ok and s["parts"] <= max_parts, s
    check(orc, "bf16", 512, 512, 8192, si.config_seed(21, max_parts), kind="int", alpha=1.0,
          beta=0.0, config=cfg)


def test_no_split_when_asked(orc):
    cfg = (128, 128, 64, 4, 1)
    ok, s = splits("bf16", 512, 512, 8192, cfg)
    assert not ok and s["parts"] == 1
    check(orc, "bf16", 512, 512, 8192, si.config_seed(21, 1), kind="int", alpha=1.0, beta=0.0,
          config=cfg)


def test_random_bf16_within_bound_and_beta(orc):
    # beta != 0: only the part that adds the partials reads and writes C
    ok, _ = splits("bf16", 640, 384, 6000)
    assert ok
    check(orc, "bf16", 640, 384, 6000, si.config_seed(22), kind="random", alpha=0.75, beta=0.5)


def test_int8_alpha_beta_wrap(orc):
    ok, _ = splits("i8", 384, 512, 4096)
    assert ok
    check(orc, "i8", 384, 512, 4096, si.config_seed(23), alpha=-7, beta=3)


def test_bf16_repeat_bit_identical(orc):
    """The fp32 parts are added in part order: every call gives the same bits."""
    M, N, K = 512, 512, 8192
    ok, _ = splits("bf16", M, N, K)
    assert ok
    A, B, C = operands("bf16", M, N, K, si.config_seed(24), "random")
    first, status = run_gpu("bf16", A, B, C, 1.0, 0.0)
    assert status == 0
    for _ in range(3):
        again, status = run_gpu("bf16", A, B, C, 1.0, 0.0)
        assert status == 0
        assert np.array_equal(first.view(np.uint32), again.view(np.uint32))
    ref = orc.gemm("bf16", A, B, C, 1.0, 0.0)
    compare("bf16", first, ref, A, B, K)


def test_int8_exchange_stress(orc):
    """Many back-to-back split calls on one stream, each bit-exact: a partial
    read before it was written, or counters not reset, would show here."""
    M, N, K = 1024, 1024, 4096
    ok, s = splits("i8", M, N, K)
    assert ok and s["parts"] >= 2, s
    A, B, C = operands("i8", M, N, K, si.config_seed(25), "random")
    ref = orc.gemm("i8", A, B, C, 1, 0)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    outs = [torch.empty((M, N), dtype=torch.int32, device="cuda") for _ in range(4)]
    ref_t = torch.from_numpy(ref.astype(np.int32)).cuda()
    bad = 0
    for i in range(200):
        out = outs[i % 4]
        out.fill_(-1)
        pg.gemm_i8(M, N, K, 1, dA, dB, 0, out)
        if i % 4 == 3:
            torch.cuda.synchronize()
            bad += sum(int((o != ref_t).sum().item()) for o in outs)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    assert bad == 0, f"{bad} wrong entries over 200 calls"


def test_full_size_defaults_split():
    """The bench's tensor-core workloads run with a split last wave when the
    tiles leave it at most half full (on 152 SMs: int8 4096^3 and bf16 8192^3)."""
    for dtype, n in (("i8", 4096), ("bf16", 8192)):
        s = pg.pgemm_schedule(dtype, n, n, n)
        rem = s["tiles"] % s["slots"]
        if 0 < rem <= s["slots"] // 2:
            assert s["split_tiles"] == rem and s["parts"] >= 2, s
        else:
            assert s["split_tiles"] == 0, s
