"""Parity of the schedules of the leftover tiles of the persistent
tensor-core kernels.

The tiles a partial last wave would hold have their K-iterations dealt out
to the resident slots (stream-K pieces); the pieces of a tile meet through
global memory and the last to finish adds them.  Kernels with 256-wide
tiles fed by TMA instead cut those tiles along N by default, into a left and
a right half-width unit over all of K, which exchange nothing.  These tests run shapes where the schedule
uses it (checked through pgemm_schedule first, so a test cannot pass by not
splitting) and compare with the oracle: bit-exact for int8 and for
integer-valued floats (a dropped, doubled or misplaced K range changes an
exact integer), within 1e-4 * sqrt(K) * max|A| * max|B| for random bf16.  The
fp32 sum of the pieces is taken in slot order, so repeated calls give the
same bits however the pieces finish.
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


# 1000 x 1000 x 8200: fewer tiles than slots for every configuration, so every
# element of C comes from stream-K pieces: with the cap at 8, 129 K-tiles of
# 64 columns (65 of 128) in ranges of 13 to 55, up to six pieces a tile, the
# last piece of a tile ending on the ragged last K-tile; with the default
# cap, equal halves (K beyond 2048 columns: no half-width units).  Bit-exact against the oracle on
# sampled entries and against the same call without stream-K on all of C.
@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_every_config_stream_k_exactly(orc, dtype):
    M, N, K = 1000, 1000, 8200
    A, B, C = operands(dtype, M, N, K, si.config_seed(20, 1 if dtype == "i8" else 2), "int")
    one = 1 if dtype == "i8" else 1.0
    zero = 0 if dtype == "i8" else 0.0
    rng = np.random.default_rng(20)
    ii = np.concatenate([np.arange(M), rng.integers(0, M, 3000), np.full(N, M - 1)])
    jj = np.concatenate([np.arange(N), rng.integers(0, N, 3000), np.arange(N)])
    ref = orc.entries(dtype, A, B, C, one, zero, ii, jj)
    for cfg in pg.pgemm_list_configs(dtype):
        if len(cfg) > 4:  # another producer or engine: not a persistent tensor-core kernel
            continue
        plain, status = run_gpu(dtype, A, B, C, one, zero, config=tuple(cfg) + (1,))
        assert status == 0
        assert np.array_equal(plain[ii, jj], ref.astype(plain.dtype)), cfg
        for cap in (0, 8):
            c = tuple(cfg) + (cap,)
            ok, s = splits(dtype, M, N, K, c)
            assert ok and s["split_tiles"] == s["tiles"] and s["half_tiles"] == 0, (c, s)
            assert s["parts"] == 2 if cap == 0 else s["parts"] > 2, (c, s)
            got, status = run_gpu(dtype, A, B, C, one, zero, config=c)
            assert status == 0, (c, status)
            assert np.array_equal(got, plain), c


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
    ok, _ = splits("i8", 384, 512, 8192)
    assert ok
    check(orc, "i8", 384, 512, 8192, si.config_seed(23), alpha=-7, beta=3)


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
    """The bench's tensor-core workloads deal their leftover tiles out along K
    (on 152 SMs: 28 of int8 4096^3's 256 pair tiles, 36 of bf16 8192^3's
    1024); bf16 with K of at most 2048 columns cuts them into half-width units
    (the exact-int8 kernels have no half-width units)."""
    for dtype, n in (("i8", 4096), ("bf16", 8192)):
        s = pg.pgemm_schedule(dtype, n, n, n)
        rem = s["tiles"] % s["slots"]
        assert rem > 0 and s["split_tiles"] == rem and 2 <= s["parts"] <= 8, s
        assert s["half_tiles"] == 0, s
    for K in (512, 2048):
        s = pg.pgemm_schedule("bf16", 4096, 4096, K)
        assert s["half_tiles"] == s["tiles"] % s["slots"] > 0 and s["split_tiles"] == 0, s
    s = pg.pgemm_schedule("i8", 4096, 4096, 2048)
    assert s["half_tiles"] == 0 and s["split_tiles"] > 0, s


# Half-width units (K of at most 2048 columns): bit-exact on integer-valued
# operands against the oracle and the unsplit call, on shapes whose last tile
# column is ragged (N = 1000: the right half of the last column partly beyond
# N; N = 320: entirely beyond), with beta != 0 (only the computed half's
# columns read C) and a ragged last K-tile.
@pytest.mark.parametrize("dtype", ["bf16"])
@pytest.mark.parametrize("M,N,K", [(1000, 1000, 2000), (700, 320, 1000), (2560, 2560, 1984)])
@pytest.mark.parametrize("cfg", [(256, 256, 128, 3), (256, 256, 64, 6), (256, 256, 64, 4),
                                 (128, 256, 64, 4)])
def test_half_width_units(orc, dtype, M, N, K, cfg):
    s = pg.pgemm_schedule(dtype, M, N, K, cfg)
    assert s["half_tiles"] > 0 and s["split_tiles"] == 0, s
    one = 1 if dtype == "i8" else 1.0
    beta = 3 if dtype == "i8" else 0.5
    A, B, C = operands(dtype, M, N, K, si.config_seed(27, M + N + cfg[3]), "int")
    got = check(orc, dtype, M, N, K, si.config_seed(27, M + N + cfg[3]), kind="int", alpha=one,
                beta=beta, config=cfg)
    plain, status = run_gpu(dtype, A, B, C, one, beta, config=tuple(cfg) + (1,))
    assert status == 0
    assert np.array_equal(got, plain)


def test_scratch_pool_trim_and_reuse(orc):
    """Scratch (partial sums, counters, widened int8) comes from the library's
    own pool, which keeps its memory across synchronisations; after
    pgemm_trim_scratch gives it back, the next calls map it again and stay
    bit-exact, with the stream-K counters zero at every launch."""
    M, N, K = 1000, 1000, 4100
    for dtype in ("i8", "bf16"):
        ok, _ = splits(dtype, M, N, K)
        assert ok
        kind = "random" if dtype == "i8" else "int"
        A, B, C = operands(dtype, M, N, K, si.config_seed(26), kind)
        ref = orc.gemm(dtype, A, B, C, 1, 0)
        for trim in (False, True, False):
            if trim:
                pg.pgemm_trim_scratch()
            got, status = run_gpu(dtype, A, B, C, 1, 0)
            assert status == 0
            compare(dtype, got, ref, A, B, K, exact=True)
