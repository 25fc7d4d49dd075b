"""The stage-reuse hazard experiment ("Software pipelines and asynchronous
copies", section "Practice"): a two-stage copy-and-reduce over a 4096 x 4096
array.  With the consume-before-reuse wait every row sum is exact even when
one consumer warp is slowed down; without it the producer overwrites a stage
the slow warp has not read yet and row sums go wrong.  The expected row sums
come from the host (exact integer arithmetic on integer-valued data)."""
import numpy as np
import pytest

import seeded_inputs as si

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import software_pipelined_tiled_loop_gb300 as pg  # noqa: E402

ROWS = COLS = 4096


@pytest.fixture(scope="module")
def data():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    X = si.small_int_f32((ROWS, COLS), 77, -8, 7)
    rowsum = X.astype(np.int64).sum(axis=1)
    return torch.from_numpy(X).cuda(), rowsum


def run(data, check_reuse, seed, delay_ns=2000, trace_cap=0):
    dX, rowsum = data
    perm = np.random.default_rng(seed).permutation(ROWS).astype(np.int32)
    dperm = torch.from_numpy(perm).cuda()
    out = torch.zeros(ROWS, dtype=torch.float32, device="cuda")
    tr = torch.zeros(1 + 2 * trace_cap, dtype=torch.int64, device="cuda") if trace_cap else None
    pg.pgemm_stage_reuse_demo(dX, ROWS, COLS, dperm, out, check_reuse, 0, delay_ns, tr, trace_cap)
    torch.cuda.synchronize()
    assert pg.pgemm_get_device_status() == 0
    bad = int(np.count_nonzero(out.cpu().numpy().astype(np.int64) != rowsum[perm]))
    return bad, (tr.cpu().numpy().view(np.uint64) if tr is not None else None)


def test_with_the_reuse_wait_every_row_is_exact(data):
    for it in range(10):
        bad, _ = run(data, 1, 1000 + it)
        assert bad == 0


def test_without_the_reuse_wait_a_delayed_warp_reads_overwritten_stages(data):
    total = sum(run(data, 0, 2000 + it)[0] for it in range(5))
    assert total > 0


def decode(tr):
    n = int(tr[0])
    ev = []
    for i in range(min(n, (len(tr) - 1) // 2)):
        ts, w = int(tr[1 + 2 * i]), int(tr[2 + 2 * i])
        ev.append((ts, w >> 56, (w >> 48) & 0xFF, (w >> 40) & 0xFF, w & 0xFFFFFFFF))
    return sorted(ev)


def test_trace_orders_reads_before_reuse(data):
    _, tr = run(data, 1, 3000, trace_cap=4096)
    ev = decode(tr)
    assert ev, "no trace events"
    read_end = {}
    for ts, e, s, w, t in ev:
        if e == 6:
            read_end.setdefault(t, []).append(ts)
    checked = 0
    for ts, e, s, w, t in ev:
        if e == 4:  # reuse allowed for tile t: all four warps finished tile t - 2
            ends = read_end.get(t - 2, [])
            assert len(ends) == 4 and max(ends) <= ts
            checked += 1
    assert checked > 0
