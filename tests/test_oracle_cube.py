"""Pins of the oracle's 3D cube token order (DSV pages, "Technische
samenvatting" 2B and the Hindi summary 2B: query grouping in small cubes of
the latent grid), independent of its nested-loop definition."""
from pathlib import Path

import numpy as np
import pytest

import oracle

GOLDEN = Path(__file__).resolve().parent / "golden"


def _golden(name):
    lines = [l for l in (GOLDEN / name).read_text().splitlines() if l.strip() and not l.startswith("#")]
    return np.array([int(v) for v in lines[0].split()])


@pytest.mark.parametrize("name, grid, cube", [
    ("cube_order_1x4x4_cube_1x2x2.txt", (1, 4, 4), (1, 2, 2)),
    ("cube_order_2x2x4_cube_2x1x2.txt", (2, 2, 4), (2, 1, 2)),
])
def test_cube_order_hand_worked(name, grid, cube):
    assert np.array_equal(oracle.cube_order(*grid, *cube), _golden(name))


@pytest.mark.parametrize("grid, cube", [((4, 8, 8), (2, 4, 4)), ((3, 6, 10), (1, 3, 5)), ((2, 4, 6), (2, 2, 3)),
                                        ((16, 32, 32), (2, 8, 8))])
def test_cube_order_is_a_permutation_of_cubes(grid, cube):
    T, Hl, Wl = grid
    ct, cy, cx = cube
    perm = oracle.cube_order(T, Hl, Wl, ct, cy, cx)
    N, blk = T * Hl * Wl, ct * cy * cx
    assert sorted(perm.tolist()) == list(range(N))          # a bijection
    t, rem = np.divmod(perm, Hl * Wl)
    y, x = np.divmod(rem, Wl)
    for g in range(N // blk):
        sl = slice(g * blk, (g + 1) * blk)
        # every group is exactly one cube: ct x cy x cx distinct, contiguous coordinates
        for coord, c in ((t, ct), (y, cy), (x, cx)):
            v = coord[sl]
            assert v.max() - v.min() == c - 1 and v.min() % c == 0
        # the cubes come in raster order of the cube grid
        cube_id = (t[sl].min() // ct * (Hl // cy) + y[sl].min() // cy) * (Wl // cx) + x[sl].min() // cx
        assert cube_id == g
        # and inside a cube the tokens in raster order
        assert np.all(np.diff(perm[sl]) > 0)


@pytest.mark.parametrize("grid, cube", [((2, 4, 8), (1, 1, 8)), ((3, 4, 6), (1, 2, 6)), ((2, 2, 4), (2, 2, 4))])
def test_full_rows_cube_is_raster_order(grid, cube):
    # a cube spanning whole rows of one frame (or the whole grid) keeps raster order
    assert np.array_equal(oracle.cube_order(*grid, *cube), np.arange(np.prod(grid)))


def test_permute_tokens_round_trip_and_rows():
    rng = np.random.default_rng(3)
    grid, cube = (2, 4, 4), (1, 2, 2)
    perm = oracle.cube_order(*grid, *cube)
    X = rng.integers(0, 1 << 15, size=(2, 3, 32, 8)).astype(np.uint16)
    Y = oracle.permute_tokens(X, perm)
    assert Y.dtype == X.dtype
    for n in range(32):
        assert np.array_equal(Y[:, :, n], X[:, :, perm[n]])
    assert np.array_equal(oracle.permute_tokens(Y, perm, inverse=True), X)


def test_cube_order_rejects_non_tiling_cube():
    with pytest.raises(ValueError):
        oracle.cube_order(2, 4, 6, 1, 2, 4)
