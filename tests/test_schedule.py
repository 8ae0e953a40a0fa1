"""The transport kernel's work split, checked on the host (no GPU needed).

eot_transport_schedule plays every CTA's tile walk with the kernel's own
code (the same walk, segments and partial-slot rule as the epilogue, the
same slot rule as the fix-up) and counts inconsistencies: a tile visited
twice or never, a row block whose partial slots are not the ones the
fix-up sums, a slot holding two row blocks.  These tests run it over an
exhaustive grid of small shapes and over the shapes of the measured
workloads, and check on top the balance and the shape of the split."""
import ctypes

import numpy as np
import pytest

from birkhoff_projection_gb300 import _lib


@pytest.fixture(scope="module")
def L():
    return _lib.lib()


def schedule(L, n_rb, n_kt, ctas):
    owner = np.full(n_rb * n_kt, -7, dtype=np.int64)
    rc = L.eot_transport_schedule(n_rb, n_kt, ctas, owner.ctypes.data_as(ctypes.c_void_p))
    return rc, owner


def check_shape(owner, n_rb, n_kt, ctas):
    counts = np.bincount(owner, minlength=ctas)
    assert counts.size == ctas
    assert counts.max() - counts.min() <= 1  # equal work up to one tile
    full = (n_rb // ctas) * ctas
    grid = owner[: full * n_kt].reshape(full, n_kt)
    assert np.all(grid == (np.arange(full) % ctas)[:, None])  # whole row blocks, round robin
    run = owner[full * n_kt:]
    assert np.all(np.diff(run) >= 0)  # the rest in contiguous runs, in CTA order


def test_small_shapes_exhaustively(L):
    for n_rb in range(1, 21):
        for n_kt in range(1, 8):
            for ctas in range(1, min(n_rb * n_kt, 40) + 1):
                rc, owner = schedule(L, n_rb, n_kt, ctas)
                assert rc == 0, (n_rb, n_kt, ctas, rc)
                check_shape(owner, n_rb, n_kt, ctas)


@pytest.mark.parametrize("n_rb,n_kt,ctas", [
    (512, 344, 152),  # 65536^2, 192-key tiles (value slices of at most 128 columns)
    (512, 258, 152),  # 65536^2, 256-key tiles
    (512, 516, 152),  # 65536^2, 128-key tiles (the moment form)
    (128, 88, 152),   # 16384^2, 192-key tiles: fewer row blocks than SMs, all in runs
    (128, 66, 152),   # 16384^2, 256-key tiles
    (4, 3, 12),       # a few hundred points: one tile per CTA
    (314, 4, 152),    # 40000 x 200 points: runs across two or three row blocks
    (1000, 1, 256),   # one key tile per row block, the largest grid
])
def test_workload_shapes(L, n_rb, n_kt, ctas):
    rc, owner = schedule(L, n_rb, n_kt, ctas)
    assert rc == 0
    check_shape(owner, n_rb, n_kt, ctas)


def test_null_owner_and_bad_arguments(L):
    assert L.eot_transport_schedule(16, 5, 7, None) == 0
    E = _lib.B4_EINVAL
    assert L.eot_transport_schedule(0, 5, 7, None) == E
    assert L.eot_transport_schedule(16, 0, 7, None) == E
    assert L.eot_transport_schedule(16, 5, 0, None) == E
    assert L.eot_transport_schedule(16, 5, 257, None) == E   # beyond the partial slots
    assert L.eot_transport_schedule(2, 3, 7, None) == E      # more CTAs than tiles
    assert L.eot_transport_schedule(1 << 20, 1 << 10, 152, None) == E  # too many tiles to play
