"""The tile walk of the symmetric GEMMs (the Gram matrix Y Y^T and the
polynomial aI + bA + cA^2 of a symmetric A), read from the library on the
host: each launched 128 x bn tile writes its elements with col >= row in place
and mirrors those with col > row, so every element of the m x m output must
be written exactly once, and no launched tile may lie wholly below the
diagonal.  The count for m = 4096 with bn = 256 is 272 of the 512 tiles."""
import ctypes as C

import numpy as np
import pytest

from newton_schulz_bucket_gb300 import _capi

BM = 128


@pytest.fixture(scope="module")
def lib():
    return _capi.load()


def walk(lib, m, bn):
    n = lib.muon_testing_sym_tiles(m, bn, None, None, 0)
    assert n > 0
    tm = (C.c_int32 * n)()
    tn = (C.c_int32 * n)()
    assert lib.muon_testing_sym_tiles(m, bn, tm, tn, n) == n
    return list(zip(tm, tn))


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("m", [8, 100, 128, 129, 256, 300, 512, 1000, 1024, 1536, 4096])
def test_every_element_written_once(lib, m, bn):
    tiles = walk(lib, m, bn)
    assert len(set(tiles)) == len(tiles)
    assert [t[0] for t in tiles] == sorted(t[0] for t in tiles)  # tile rows in order
    count = np.zeros((m, m), np.int8)
    for tm, tn in tiles:
        r0, c0 = tm * BM, tn * bn
        assert 0 <= r0 < m and 0 <= c0 < m, (tm, tn)
        rows = np.arange(r0, min(r0 + BM, m))[:, None]
        cols = np.arange(c0, min(c0 + bn, m))[None, :]
        upper = cols >= rows
        assert upper.any(), f"tile ({tm}, {tn}) lies below the diagonal"
        ri, ci = np.broadcast_arrays(rows, cols)
        count[ri[upper], ci[upper]] += 1           # in place
        strict = cols > rows
        count[ci[strict], ri[strict]] += 1         # mirrored
    assert count.min() == 1 and count.max() == 1


def test_counts_and_arguments(lib):
    assert lib.muon_testing_sym_tiles(4096, 256, None, None, 0) == 272
    assert lib.muon_testing_sym_tiles(4096, 128, None, None, 0) == 32 * 33 // 2
    tm = (C.c_int32 * 3)(-7, -7, -7)
    tn = (C.c_int32 * 3)(-7, -7, -7)
    assert lib.muon_testing_sym_tiles(1024, 128, tm, tn, 2) == 36
    assert tm[2] == -7 and tn[2] == -7                 # nothing past cap
    for bad in [(0, 128, 0), (1 << 21, 128, 0), (512, 64, 0), (512, 128, -1)]:
        assert lib.muon_testing_sym_tiles(bad[0], bad[1], None, None, bad[2]) == -1
    assert lib.muon_testing_sym_tiles(512, 128, None, None, 4) == -1
