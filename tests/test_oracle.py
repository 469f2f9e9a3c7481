"""The fp64 oracle against its pins (CPU only)."""
import math

import numpy as np
import pytest

import oracle.attention as orc
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc)


def test_practice_exercise_tiled_vs_standard():
    """[P4 practice exercise] n=1024, d=64, block 128: the tiled result equals the
    materialised one within 1e-5 (fp64 gives far better)."""
    r = np.random.default_rng(7)
    q, k, v = (r.standard_normal((1, 1, 1024, 64)) for _ in range(3))
    o, l = orc.forward(q, k, v, 1 / 8)
    to, tl = orc.tiled_forward(q, k, v, 1 / 8, 128, 128)
    assert np.abs(to - o).max() <= 1e-5
    assert np.abs(to - o).max() <= 1e-12
    assert np.abs(tl - l).max() <= 1e-12


def test_row_chunking_matches_whole_rows():
    r = np.random.default_rng(8)
    q, k, v = (r.standard_normal((1, 2, 96, 8)) for _ in range(3))
    for causal in (False, True):
        o, l = orc.forward(q, k, v, 0.35, causal=causal)
        oc, lc = orc.forward(q, k, v, 0.35, causal=causal, row_chunk=40)
        np.testing.assert_array_equal(o, oc)
        np.testing.assert_array_equal(l, lc)


def test_fully_masked_row_convention():
    """A row with no visible key: O = 0, LSE = -inf, zero gradients."""
    r = np.random.default_rng(9)
    q, k, v, do = (r.standard_normal((1, 1, 8, 4)) for _ in range(4))
    bm = np.array([[1, 0], [0, 0]], np.uint8)   # rows 4..7 see nothing
    o, l = orc.forward(q, k, v, 0.5, block_mask=bm, block=4)
    assert np.all(o[0, 0, 4:] == 0) and np.all(np.isneginf(l[0, 0, 4:]))
    to, tl = orc.tiled_forward(q, k, v, 0.5, 3, 3, block_mask=bm, block=4)
    np.testing.assert_allclose(to, o, atol=1e-14)
    assert np.all(np.isneginf(tl[0, 0, 4:]))
    dq, dk, dv, _ = orc.backward(q, k, v, do, 0.5, block_mask=bm, block=4)
    assert np.all(dq[0, 0, 4:] == 0)
    assert np.all(dk[0, 0, 4:] == 0) and np.all(dv[0, 0, 4:] == 0)
