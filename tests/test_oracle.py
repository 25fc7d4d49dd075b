"""The oracle against its pins (facts fixed by mathematics and by the pages)."""
import numpy as np
import pytest

import oracle
import oracle_pins as pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    fails = pin(orc)
    assert not fails, "\n".join(fails[:10])


def test_rejects_bad_arguments(orc):
    A = np.zeros((2, 3), np.float32)
    B = np.zeros((4, 2), np.float32)
    with pytest.raises(ValueError):
        orc.gemm("f32", A, B)
    with pytest.raises(TypeError):
        orc.gemm("bf16", A, np.zeros((3, 2), np.float32))
    with pytest.raises(ValueError):
        orc.entries("f32", A, np.zeros((3, 2), np.float32), None, 1.0, 0.0, [2], [0])


def test_rows_and_entries_agree_on_random_case(orc):
    """The three entry points evaluate the same definition."""
    import seeded_inputs as si
    A = si.uniform_f32((37, 53), 7)
    B = si.uniform_f32((53, 29), 8)
    C = si.uniform_f32((37, 29), 9)
    full = orc.gemm("f32", A, B, C, 1.5, -0.25)
    part = orc.gemm("f32", A, B, C, 1.5, -0.25, rows=(10, 20))
    assert np.array_equal(full[10:20], part)
    ii = np.array([0, 36, 17, 5])
    jj = np.array([0, 28, 3, 11])
    e = orc.entries("f32", A, B, C, 1.5, -0.25, ii, jj)
    assert np.array_equal(full[ii, jj], e)


def test_thread_count_reported(orc):
    assert orc.num_threads() >= 1
