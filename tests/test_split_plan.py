"""The K-split rule of the persistent tensor-core schedule (pgemm_split_plan,
host code of the library, no GPU needed).

Checked against what the rule is for rather than against a restatement of
it: the split must shorten the schedule's makespan (measured in tile-times
with each unit taking time proportional to its K range), the parts of a tile
must cover its K range exactly once in whole granules, the last wave must fit
in the slots, and the caps (8 parts, max_k_parts, whole granules) must hold.
"""
import itertools
import math

import pytest

import software_pipelined_tiled_loop_gb300 as pg


@pytest.fixture(scope="module", autouse=True)
def L():
    from software_pipelined_tiled_loop_gb300 import build
    build.build()
    return pg.lib()


def part_ranges(k_tiles, parts, gran, granules):
    """K-tile ranges of the parts of a split tile, per the documented rule."""
    out = []
    for j in range(parts):
        kb = j * granules // parts * gran
        ke = k_tiles if j == parts - 1 else (j + 1) * granules // parts * gran
        out.append((kb, ke))
    return out


def makespan(tiles, slots, k_tiles, split_tiles, parts, gran, granules):
    """Static schedule: unit u runs on slot u % slots after the slot's earlier
    units; the split tiles' parts come first, then the whole tiles.  A whole
    tile takes 1, a part (ke - kb) / k_tiles."""
    busy = [0.0] * slots
    units = []
    for _ in range(split_tiles):
        units += [(ke - kb) / k_tiles for kb, ke in part_ranges(k_tiles, parts, gran, granules)]
    units += [1.0] * (tiles - split_tiles)
    for u, t in enumerate(units):
        busy[u % slots] += t
    return max(busy) if busy else 0.0


CASES = list(itertools.product(
    [1, 5, 28, 75, 76, 77, 152, 256, 1024, 1025],   # tiles
    [1, 2, 76, 152, 304],                            # slots
    [0, 1, 16, 31, 32, 64, 65, 128, 257],            # K-tiles
    [0, 16],                                         # round tiles (0: bf16, 16: int8)
    [0, 1, 2, 3, 8],                                 # max_k_parts
))


@pytest.mark.parametrize("tiles,slots,k_tiles,rt,maxp", CASES)
def test_plan_properties(tiles, slots, k_tiles, rt, maxp):
    p = pg.pgemm_split_plan(tiles, slots, k_tiles, rt, maxp)
    gran, granules, parts, nsplit = p["gran"], p["granules"], p["parts"], p["split_tiles"]
    assert gran == (rt if rt else 16)
    assert granules == k_tiles // gran
    rem = tiles % slots
    if parts == 1:
        assert nsplit == 0
        # nothing split although it would pay: only when a rule forbids it
        if rem and 2 * rem <= slots and granules >= 2 and maxp != 1:
            pytest.fail(f"no split for {p}")
        return
    assert maxp != 1
    assert nsplit == rem > 0
    assert rem * parts <= slots                    # the split wave fits the grid
    assert 2 <= parts <= min(8, granules)
    if maxp > 1:
        assert parts <= maxp
    # parts cover [0, k_tiles) exactly, each at least one granule, rounds aligned
    ranges = part_ranges(k_tiles, parts, gran, granules)
    assert ranges[0][0] == 0 and ranges[-1][1] == k_tiles
    for (a, b), (c, _) in zip(ranges, ranges[1:]):
        assert b == c
    for kb, ke in ranges:
        assert ke - kb >= gran
        assert kb % gran == 0
    # and it shortens the schedule
    before = makespan(tiles, slots, k_tiles, 0, 1, gran, granules)
    after = makespan(tiles, slots, k_tiles, nsplit, parts, gran, granules)
    assert before == math.ceil(tiles / slots)
    assert after < before


def test_bench_shapes():
    # 4096^3 int8 on CTA pairs: 256 tiles over 76 pairs -> 28 tiles in halves
    p = pg.pgemm_split_plan(256, 76, 64, 16, 0)
    assert (p["split_tiles"], p["parts"]) == (28, 2)
    # 8192^3 bf16 on CTA pairs: 1024 tiles over 76 pairs -> 36 tiles in halves
    p = pg.pgemm_split_plan(1024, 76, 128, 0, 0)
    assert (p["split_tiles"], p["parts"]) == (36, 2)
    # a full last wave is never split
    assert pg.pgemm_split_plan(152, 76, 128, 0, 0)["parts"] == 1


@pytest.mark.parametrize("args", [(-1, 76, 64, 0, 0), (10, 0, 64, 0, 0), (10, 76, -1, 0, 0),
                                  (10, 76, 64, -1, 0), (10, 76, 64, 0, -2)])
def test_plan_rejects_bad_arguments(args):
    with pytest.raises(pg.PgemmError):
        pg.pgemm_split_plan(*args)


# ------------------------------------------------ fp32 stream-K tail ---------
def sk_slot_ranges(R, T, G):
    total = R * T
    return [(j * total // G, (j + 1) * total // G) for j in range(G)]


SK_CASES = list(itertools.product(
    [1, 4, 100, 112, 303, 304, 305, 1024, 1100],   # tiles
    [2, 76, 304],                                   # slots
    [0, 1, 7, 8, 64, 128, 513],                     # K-tiles
    [0, 1],                                         # max_k_parts
))


@pytest.mark.parametrize("tiles,slots,T,maxp", SK_CASES)
def test_stream_k_plan_properties(tiles, slots, T, maxp):
    p = pg.pgemm_stream_k_plan(tiles, slots, T, maxp)
    R = tiles % slots
    if p["sk_tiles"] == 0:
        assert p["max_pieces"] == 1
        # off only when a rule says so
        assert (maxp == 1 or T == 0 or R == 0 or R * T // slots < 8
                or 8 * -(-R * T // slots) > 7 * T)
        return
    assert maxp != 1 and p["sk_tiles"] == R and p["share"] == R * T // slots >= 8
    ranges = sk_slot_ranges(R, T, slots)
    # the slots' ranges tile the R * T iterations exactly, none is empty,
    # and none spans more than two tiles (the kernel keeps two partial slots)
    assert ranges[0][0] == 0 and ranges[-1][1] == R * T
    assert all(b == c for (_, b), (c, _) in zip(ranges, ranges[1:]))
    assert all(b > a and (b - 1) // T - a // T <= 1 for a, b in ranges)
    # pieces per tile: the kernel's closed form agrees with the ranges
    def slot_of(x):
        return ((x + 1) * slots - 1) // (R * T)
    most = 1
    for r in range(R):
        owners = [j for j, (a, b) in enumerate(ranges) if a < (r + 1) * T and b > r * T]
        assert owners == list(range(slot_of(r * T), slot_of((r + 1) * T - 1) + 1))
        most = max(most, len(owners))
    assert p["max_pieces"] == most
    # makespan in tile-times: W whole waves plus the largest share, below W + 1
    W = tiles // slots
    longest = max(b - a for a, b in ranges)
    assert W + longest / T <= math.ceil(tiles / slots) - 1 / 8


def test_stream_k_bench_shape():
    # fp32 4096^3 on 152 SMs x 2 blocks: 1024 tiles, 112 left after three waves
    p = pg.pgemm_stream_k_plan(1024, 304, 128)
    assert p["sk_tiles"] == 112 and p["share"] == 112 * 128 // 304
