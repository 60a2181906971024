"""The tile raster as the library evaluates it (ts_gemm_tile_coords, no GPU).

The kernel maps a tile id to its output tile with divisions by launch constants
done as multiply-high and shift; the host runs the very same function.  These
checks pin it to the plain-division definition of the raster (groups of
`raster_group` tile rows walked down a column band, odd groups from the right)
and to a one-to-one cover of the tile grid, for ragged grids whose last group
is shorter.
"""
import itertools

import numpy as np
import pytest


def _plain(t, tm, tn, G):
    g = t // (G * tn)
    first = g * G
    gs = min(G, tm - first)
    local = t - g * G * tn
    col = local // gs
    return first + local % gs, (tn - 1 - col) if g % 2 else col


TILES = {"128x128": (128, 128), "128x256": (128, 256), "256x256": (256, 256)}


@pytest.mark.parametrize("tile", sorted(TILES))
@pytest.mark.parametrize("G", [0, 1, 2, 3, 5, 8, 13, 64])
@pytest.mark.parametrize("M,N", [(1, 1), (129, 300), (1100, 1300), (8191, 6143), (2048, 640), (40000, 257)])
def test_raster_matches_plain_division_and_covers_the_grid(ts, tile, G, M, N):
    bm, bn = TILES[tile]
    tm, tn = -(-M // bm), -(-N // bn)
    mb, nb = ts.ts_gemm_tile_coords(M, N, 64, ts.TS_OUT_BF16, "clc", tile=tile, raster_group=G)
    assert mb.size == tm * tn
    Ge = G if G > 0 else 8  # the library's default group
    want = np.array([_plain(t, tm, tn, Ge) for t in range(tm * tn)], dtype=np.int64).reshape(-1, 2)
    assert np.array_equal(mb, want[:, 0]) and np.array_equal(nb, want[:, 1])
    assert np.array_equal(np.sort(mb.astype(np.int64) * tn + nb), np.arange(tm * tn))


def test_raster_walks_group_rows_down_a_column_band(ts):
    # 4 tile rows x 3 tile columns, groups of 2 rows, the second group from the right:
    # (0,0) (1,0) (0,1) (1,1) (0,2) (1,2) (2,2) (3,2) (2,1) (3,1) (2,0) (3,0)
    mb, nb = ts.ts_gemm_tile_coords(512, 768, 64, ts.TS_OUT_F32, "static", tile="128x256", raster_group=2)
    assert list(zip(mb.tolist(), nb.tolist())) == [(0, 0), (1, 0), (0, 1), (1, 1), (0, 2), (1, 2),
                                                   (2, 2), (3, 2), (2, 1), (3, 1), (2, 0), (3, 0)]


def test_raster_large_grid_spot_checks(ts):
    # a grid of 65536 x 8 tiles, with ids up to 2^19: the multiply-high stays exact
    M, N = 65536 * 128, 8 * 256
    tm, tn = 65536, 8
    for G, first in itertools.product([1, 7, 8, 1000], [0, 123_457, tm * tn - 1000]):
        mb, nb = ts.ts_gemm_tile_coords(M, N, 64, ts.TS_OUT_BF16, "static", first=first, count=1000,
                                        tile="128x256", raster_group=G)
        want = np.array([_plain(t, tm, tn, G) for t in range(first, first + 1000)])
        assert np.array_equal(mb, want[:, 0]) and np.array_equal(nb, want[:, 1])


def test_raster_range_errors(ts):
    with pytest.raises(ts.TsError):
        ts.ts_gemm_tile_coords(256, 256, 64, tile="128x128", first=3, count=2)  # 4 tiles: [3, 5) is outside
    with pytest.raises(ts.TsError):
        ts.ts_gemm_tile_coords(256, 256, 64, tile="128x128", first=-1, count=1)
    with pytest.raises(ts.TsError):
        ts.ts_gemm_tile_coords(256, 256, 64, tile="128x128", raster_group=-1)
    mb, nb = ts.ts_gemm_tile_coords(0, 256, 64, tile="128x128")
    assert mb.size == 0 and nb.size == 0
