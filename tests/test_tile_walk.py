"""The tile walks of the tcgen05 products, read from the library on the host.

Gram matrix Y Y^T and polynomial aI + bA + cA^2 of a symmetric A: each
launched 128 x bn tile writes its elements with col >= row in place and
mirrors those with col > row, so every element of the m x m output must be
written exactly once, and no launched tile may lie wholly below the diagonal.
The count for m = 4096 with bn = 256 is 272 of the 512 tiles.

Update Q Y: the grouped raster must visit every tile of the m x n output once,
and the tiles of one group (8 tile rows sweeping the tile columns together)
must come in one run.

Groups with m >= 256 run the CTA-pair form (256 x 256 tiles, one cluster of
two CTAs per tile); its walks must satisfy the same properties.
"""
import ctypes as C

import numpy as np
import pytest

from newton_schulz_bucket_gb300 import _capi

BM = 128
GRAM, POLY, UPDATE = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    return _capi.load()


def walk(lib, op, m, n, bn):
    """Tiles of the one-CTA form (bn = 128 or 256) or, for bn = "pair", of the
    CTA-pair form (256 x 256)."""
    if bn == "pair":
        f = lambda tm, tn, cap: lib.muon_testing_tile_walk_pair(op, m, n, tm, tn, cap)
    else:
        f = lambda tm, tn, cap: lib.muon_testing_tile_walk(op, m, n, bn, tm, tn, cap)
    count = f(None, None, 0)
    assert count > 0
    tm = (C.c_int32 * count)()
    tn = (C.c_int32 * count)()
    assert f(tm, tn, count) == count
    return list(zip(tm, tn))


def tile_dims(bn):
    return (256, 256) if bn == "pair" else (BM, bn)


@pytest.mark.parametrize("bn", [128, 256, "pair"])
@pytest.mark.parametrize("m", [8, 100, 128, 129, 256, 300, 512, 1000, 1024, 1536, 4096])
def test_symmetric_outputs_written_once(lib, m, bn):
    tiles = walk(lib, GRAM, m, 0, bn)
    assert tiles == walk(lib, POLY, m, 0, bn)
    assert len(set(tiles)) == len(tiles)
    assert [t[0] for t in tiles] == sorted(t[0] for t in tiles)  # tile rows in order
    bm, bn = tile_dims(bn)
    count = np.zeros((m, m), np.int8)
    for tm, tn in tiles:
        r0, c0 = tm * bm, tn * bn
        assert 0 <= r0 < m and 0 <= c0 < m, (tm, tn)
        rows = np.arange(r0, min(r0 + bm, m))[:, None]
        cols = np.arange(c0, min(c0 + bn, m))[None, :]
        upper = cols >= rows
        assert upper.any(), f"tile ({tm}, {tn}) lies below the diagonal"
        ri, ci = np.broadcast_arrays(rows, cols)
        count[ri[upper], ci[upper]] += 1           # in place
        strict = cols > rows
        count[ci[strict], ri[strict]] += 1         # mirrored
    assert count.min() == 1 and count.max() == 1


@pytest.mark.parametrize("bn", [128, 256, "pair"])
@pytest.mark.parametrize("m,n", [(8, 8), (128, 1000), (300, 400), (1024, 1024), (1100, 7168),
                                 (4096, 16384), (2048, 7168)])
def test_update_raster_visits_every_tile_once(lib, m, n, bn):
    tiles = walk(lib, UPDATE, m, n, bn)
    bm, bn = tile_dims(bn)
    tiles_m, tiles_n = -(-m // bm), -(-n // bn)
    assert sorted(tiles) == [(a, b) for a in range(tiles_m) for b in range(tiles_n)]
    groups = [tm // 8 for tm, _ in tiles]
    assert groups == sorted(groups)  # one run per group of 8 tile rows


def test_counts_and_arguments(lib):
    assert lib.muon_testing_tile_walk(GRAM, 4096, 0, 256, None, None, 0) == 272
    assert lib.muon_testing_tile_walk(POLY, 4096, 0, 128, None, None, 0) == 32 * 33 // 2
    assert lib.muon_testing_tile_walk(UPDATE, 4096, 16384, 256, None, None, 0) == 32 * 64
    tm = (C.c_int32 * 3)(-7, -7, -7)
    tn = (C.c_int32 * 3)(-7, -7, -7)
    assert lib.muon_testing_tile_walk(GRAM, 1024, 0, 128, tm, tn, 2) == 36
    assert tm[2] == -7 and tn[2] == -7                 # nothing past cap
    for op, m, n, bn, cap in [(GRAM, 0, 0, 128, 0), (GRAM, 1 << 21, 0, 128, 0),
                              (GRAM, 512, 0, 64, 0), (GRAM, 512, 0, 128, -1),
                              (UPDATE, 512, 0, 128, 0), (3, 512, 512, 128, 0)]:
        assert lib.muon_testing_tile_walk(op, m, n, bn, None, None, cap) == -1
    assert lib.muon_testing_tile_walk(GRAM, 512, 0, 128, None, None, 4) == -1
    # the CTA-pair form: 256 x 256 tiles, for m >= 256
    assert lib.muon_testing_tile_walk_pair(GRAM, 4096, 0, None, None, 0) == 16 * 17 // 2
    assert lib.muon_testing_tile_walk_pair(UPDATE, 4096, 16384, None, None, 0) == 16 * 64
    assert lib.muon_testing_tile_walk_pair(UPDATE, 512, 0, None, None, 0) == -1
    assert [lib.muon_testing_tc_pair_form(m) for m in (128, 255, 256, 4096)] == [0, 0, 1, 1]
