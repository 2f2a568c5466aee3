"""The x-run layout's definition (tests/helpers.py) on CPU: for every voxel
slot s, every (dz, dy) group and dx in {-1, 0, +1}, the row that slot s + dx
stands for in that group is the map entry nmap[(dz, dy, dx), n] of the slot's
voxel n.  This is the property the row-shifted convolution relies on."""
import numpy as np
import pytest

import workloads as W
from helpers import layout_reference


def group_row(nm, n, code, g):
    """Row that a slot code stands for in group g (dx offsets 3g, 3g+1, 3g+2)."""
    if code >= 0:
        return nm[3 * g + 1, code]
    if code <= -2:
        h = -2 - code
        v, left = h >> 1, h & 1
        return nm[3 * g + (0 if left else 2), v]
    return n


def cases():
    rng = np.random.default_rng(9)
    sh = W.random_occupancy(10, 0.35, 51)
    return {
        "random": W.random_occupancy(10, 0.35, 50),
        "shuffled": sh[rng.permutation(len(sh))],
        "dense": W.random_occupancy(8, 0.95, 52),
        "line": np.array([[1, 2, x] for x in range(40)], np.int32),
        "two_lines": np.array([[1, y, x] for y in (2, 3) for x in range(10)], np.int32),
        "isolated": np.array([[2 * z, 2 * y, 2 * x] for z in range(4) for y in range(4) for x in range(4)],
                             np.int32),
        "single": np.array([[3, 3, 3]], np.int32),
    }


@pytest.mark.parametrize("name", list(cases()))
def test_shifted_slots_stand_for_the_right_cells(oracle_mod, name):
    coords = cases()[name]
    n = len(coords)
    nm = oracle_mod.build_nmap(coords, W.offsets_3x3x3()).astype(np.int64)
    nm[(nm < 0) | (nm >= n)] = n
    slots = layout_reference(coords, nmap=nm)
    S = len(slots)
    assert np.array_equal(np.sort(slots[slots >= 0]), np.arange(n))
    for s in np.nonzero(slots >= 0)[0]:
        v = slots[s]
        for g in range(9):
            for dx in (-1, 0, 1):
                t = s + dx
                code = slots[t] if 0 <= t < S else -1
                assert group_row(nm, n, code, g) == nm[3 * g + dx + 1, v], (name, s, g, dx)


def test_separator_counts(oracle_mod):
    # two aligned lines: the first run's right cells and the second run's
    # left cells are all missing, so one separator is shared
    coords = cases()["two_lines"]
    nm = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    slots = layout_reference(coords, nmap=nm)
    assert len(slots) == 20 + 1
    # the second line shifted by one in x: each run's outer cell lies on the
    # other line, and they differ, so the boundary takes two separators; the
    # first and last voxels have no active outer cell
    coords = np.array([[1, 2, x] for x in range(10)] + [[1, 3, x] for x in range(1, 11)], np.int32)
    nm = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    slots = layout_reference(coords, nmap=nm)
    assert len(slots) == 20 + 2
    # voxel 0 at (1, 2, 1) with the next line starting at (1, 3, 0): voxel
    # 0's left cell in the (0, +1) group is active, so the layout opens with
    # a left separator; the run boundary shares one; the last voxel has none
    coords = np.array([[1, 2, x] for x in range(1, 5)] + [[1, 3, x] for x in range(0, 5)], np.int32)
    nm = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    slots = layout_reference(coords, nmap=nm)
    assert slots[0] == -3 and len(slots) == 9 + 1 + 1
    # isolated voxels: no outer cell is active, one separator per boundary
    coords = cases()["isolated"]
    nm = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    slots = layout_reference(coords, nmap=nm)
    assert len(slots) == 64 + 63


def test_tiled_shifted_sum_equals_oracle(oracle_mod):
    """The row-shifted convolution's data flow in numpy: 256-slot tiles, one
    258-row operand per (dz, dy) group gathered from the slots one before the
    tile to one after it, the three dx offsets read 0, 1 and 2 rows in.  Its
    voxel rows equal the oracle's sum."""
    coords = W.random_occupancy(14, 0.3, 60)
    n = len(coords)
    nm = oracle_mod.build_nmap(coords, W.offsets_3x3x3()).astype(np.int64)
    nm[(nm < 0) | (nm >= n)] = n
    rng = np.random.default_rng(1)
    ci, co = 8, 5
    feats = rng.standard_normal((n, ci))
    w = rng.standard_normal((27, ci, co))
    b = rng.standard_normal(co)
    slots = layout_reference(coords, nmap=nm)
    S = len(slots)
    fpad = np.vstack([feats, np.zeros((1, ci))])  # row n: a missing neighbour
    out = np.full((n, co), np.nan)
    tile = 256
    for s0 in range(0, S, tile):
        acc = np.zeros((tile, co))
        for g in range(9):
            rows = []
            for r in range(tile + 2):
                s = s0 - 1 + r
                code = slots[s] if 0 <= s < S else -1
                rows.append(group_row(nm, n, code, g))
            G = fpad[np.array(rows)]
            for dxi in range(3):
                acc += G[dxi:dxi + tile] @ w[3 * g + dxi]
        for j in range(tile):
            s = s0 + j
            if s < S and slots[s] >= 0:
                out[slots[s]] = acc[j] + b
    ref, _ = oracle_mod.conv(feats.astype(np.float32), nm.astype(np.int32), w.astype(np.float32),
                             b.astype(np.float32), "f32")
    assert not np.isnan(out).any()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-9 * np.abs(ref).max() + 1e-5)
