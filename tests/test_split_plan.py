"""The stream-K rule of the persistent schedules (pgemm_stream_k_plan, host
code of the library, no GPU needed).

Checked against what the rule is for rather than against a restatement of
it: the slots' K ranges must cover the leftover tiles' iterations exactly
once with pieces of at most two tiles (the kernels keep two partial slabs
per slot), the reported piece counts must match the ranges, a cap must hold,
and the schedule's makespan (in tile-times, each unit taking time in
proportion to its K range) must fall by at least an eighth of a tile.
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


def slot_ranges(R, T, Gs):
    total = R * T
    return [(j * total // Gs, (j + 1) * total // Gs) for j in range(Gs)]


def makespan(tiles, slots, T, R, Gs):
    """Slot j: its stream-K share (if j < Gs), then whole tiles R + j, R + j +
    slots, ...  A whole tile takes 1, a share (b - a) / T."""
    busy = [0.0] * slots
    for j, (a, b) in enumerate(slot_ranges(R, T, Gs) if R else []):
        busy[j] += (b - a) / T
    for t in range(tiles - R):
        busy[t % slots] += 1.0
    return max(busy)


CASES = list(itertools.product(
    [1, 4, 5, 16, 28, 75, 76, 77, 112, 128, 152, 256, 303, 1024, 1025],   # tiles
    [1, 2, 76, 152, 304],                                                 # slots
    [0, 1, 7, 8, 16, 64, 65, 128, 257, 2048],                             # K-tiles
    [0, 1, 2, 3, 8],                                                      # max_parts
))


@pytest.mark.parametrize("tiles,slots,T,maxp", CASES)
def test_plan_properties(tiles, slots, T, maxp):
    p = pg.pgemm_stream_k_plan(tiles, slots, T, maxp)
    R = tiles % slots
    if p["sk_tiles"] == 0:
        assert p["max_pieces"] == 1 and p["sk_slots"] == 0
        # off only when a rule says so
        if maxp == 1 or T == 0 or R == 0 or slots < 2:
            return
        Gs = slots
        if maxp > 1:
            owners_max = max(len([1 for a, b in slot_ranges(R, T, slots)
                                  if a < (r + 1) * T and b > r * T]) for r in range(R))
            if owners_max > maxp:
                cap = min(maxp, slots // R)
                if cap < 2:
                    return
                Gs = R * cap
        assert R * T // Gs < 8 or 8 * -(-R * T // Gs) > 7 * T, p
        return
    Gs = p["sk_slots"]
    assert maxp != 1 and p["sk_tiles"] == R > 0 and R < Gs <= slots
    assert p["share"] == R * T // Gs >= 8
    ranges = slot_ranges(R, T, Gs)
    # the ranges tile the R * T iterations exactly, none is empty, and none
    # spans more than two tiles
    assert ranges[0][0] == 0 and ranges[-1][1] == R * T
    assert all(b == c for (_, b), (c, _) in zip(ranges, ranges[1:]))
    assert all(b > a and (b - 1) // T - a // T <= 1 for a, b in ranges)
    # pieces per tile: the kernels' closed form (slot holding iteration x)
    # agrees with the ranges
    def slot_of(x):
        return ((x + 1) * Gs - 1) // (R * T)
    most = 1
    for r in range(R):
        owners = [j for j, (a, b) in enumerate(ranges) if a < (r + 1) * T and b > r * T]
        assert owners == list(range(slot_of(r * T), slot_of((r + 1) * T - 1) + 1))
        most = max(most, len(owners))
    assert p["max_pieces"] == most
    if maxp > 1:
        assert most <= maxp
    if Gs < slots:
        # capped: every tile exactly p pieces, slot r * p starting tile r
        q = Gs // R
        assert Gs == R * q and most == q
        assert all(ranges[r * q][0] == r * T for r in range(R))
    # and the schedule ends at least an eighth of a tile earlier
    before = math.ceil(tiles / slots)
    assert makespan(tiles, slots, T, 0, 1) == before
    assert makespan(tiles, slots, T, R, Gs) <= before - 1 / 8


def test_bench_shapes():
    # int8 4096^3 on 76 CTA pairs, tensor-core cap 8: 28 leftover tiles over all 76
    p = pg.pgemm_stream_k_plan(256, 76, 64, 8)
    assert (p["sk_tiles"], p["sk_slots"]) == (28, 76) and p["max_pieces"] <= 4
    # capped at two pieces: the 28 tiles in halves on 56 pairs
    p = pg.pgemm_stream_k_plan(256, 76, 64, 2)
    assert (p["sk_tiles"], p["sk_slots"], p["max_pieces"]) == (28, 56, 2)
    # fp32 4096^3 on 152 SMs x 2 blocks: 1024 tiles, 112 left after three waves
    p = pg.pgemm_stream_k_plan(1024, 304, 128, 0)
    assert (p["sk_tiles"], p["sk_slots"]) == (112, 304) and p["share"] == 112 * 128 // 304
    # a full last wave is never split
    assert pg.pgemm_stream_k_plan(152, 76, 128, 0)["sk_tiles"] == 0


@pytest.mark.parametrize("args", [(-1, 76, 64, 0), (10, 0, 64, 0), (10, 76, -1, 0),
                                  (10, 76, 64, -2)])
def test_plan_rejects_bad_arguments(args):
    with pytest.raises(pg.PgemmError):
        pg.pgemm_stream_k_plan(*args)
