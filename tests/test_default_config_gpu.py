"""The per-shape default (tile, stages) table of the library (it depends on
the device's SM count, so it is checked on the GPU)."""
import pytest

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


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# (bm, bn, bk, stages); the CTA pair's stages hold 128 K columns each
@pytest.mark.parametrize("dtype,M,N,K,expect", [
    ("f32", 4096, 4096, 4096, (128, 128, 32, 3)),
    ("f32", 8192, 8192, 8192, (128, 128, 32, 3)),
    ("f32", 256, 256, 256, (128, 64, 32, 3)),      # 4 tiles of 128 x 128: too few for two per SM
    ("bf16", 8192, 8192, 8192, (256, 256, 128, 3)),
    ("i8", 4096, 4096, 4096, (256, 256, 128, 3)),
    ("bf16", 4096, 4096, 2048, (256, 256, 128, 3)),
    ("bf16", 4096, 4096, 512, (256, 256, 128, 3)),
    # short K, 128 x 256 tiles filling three waves: bound by writing C
    ("bf16", 4096, 4096, 128, (128, 256, 64, 3)),
    ("bf16", 4096, 4096, 256, (128, 256, 64, 4)),
    ("bf16", 4096, 4096, 384, (128, 256, 64, 4)),
    ("i8", 4096, 4096, 32, (128, 256, 64, 3)),
    ("i8", 4096, 4096, 512, (128, 256, 64, 4)),
    ("i8", 4096, 4096, 1024, (256, 256, 128, 3)),
    # fewer than three waves of 128 x 256 tiles: 128 x 128
    ("bf16", 2048, 4096, 32, (128, 128, 64, 4)),
    ("bf16", 1024, 1024, 64, (128, 128, 64, 4)),
    ("bf16", 2048, 2048, 8192, (128, 128, 64, 4)),  # 64 pair tiles: fewer than half the SMs
    ("bf16", 1024, 1024, 16384, (128, 128, 64, 4)),
])
def test_default_table(dtype, M, N, K, expect):
    if sms() != 152:
        pytest.skip("the expectations are written for 152 SMs")
    cfg = pg.pgemm_default_config(dtype, M, N, K)
    assert tuple(cfg[:4]) == expect, cfg
