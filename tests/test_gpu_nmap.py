"""GPU neighbour-map builder against the oracle: bit-exact."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import submanifold_voxel_gather_gb300 as mod
    from submanifold_voxel_gather_gb300 import build
    build.build()
    return mod


def gpu_nmap(sv, coords, offsets=None):
    import torch
    c = torch.from_numpy(np.ascontiguousarray(coords, dtype=np.int32)).cuda()
    return sv.build_nmap(c, offsets).cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "tiny_shell1", "small"])
def test_nmap_configs_exact(sv, oracle_mod, name):
    coords = W.coords_only(name)
    offs = W.offsets_3x3x3()
    np.testing.assert_array_equal(gpu_nmap(sv, coords), oracle_mod.build_nmap(coords, offs))


def test_nmap_shuffled_order_exact(sv, oracle_mod):
    coords = W.coords_only("small")
    coords = coords[W.permutation(len(coords), 1)]
    np.testing.assert_array_equal(gpu_nmap(sv, coords), oracle_mod.build_nmap(coords, W.offsets_3x3x3()))


@pytest.mark.parametrize("side,frac,seed", [(5, 1.0, 1), (12, 0.3, 2), (16, 0.05, 3)])
def test_nmap_random_grids_exact(sv, oracle_mod, side, frac, seed):
    coords = W.random_occupancy(side, frac, seed)
    np.testing.assert_array_equal(gpu_nmap(sv, coords), oracle_mod.build_nmap(coords, W.offsets_3x3x3()))


def test_nmap_edge_sizes_and_offsets(sv, oracle_mod):
    base = W.random_occupancy(10, 0.4, 9)
    for n in (1, 2, 127, 128, 129):
        c = base[:n]
        np.testing.assert_array_equal(gpu_nmap(sv, c), oracle_mod.build_nmap(c, W.offsets_3x3x3()))
    centre = np.zeros((1, 3), np.int32)
    np.testing.assert_array_equal(gpu_nmap(sv, base, centre), oracle_mod.build_nmap(base, centre))
    wide = W.offsets_cube(2)
    np.testing.assert_array_equal(gpu_nmap(sv, base, wide), oracle_mod.build_nmap(base, wide))
    far = np.array([[5, -3, 2], [0, 0, 7], [-1, -1, -1]], np.int32)
    np.testing.assert_array_equal(gpu_nmap(sv, base, far), oracle_mod.build_nmap(base, far))


def test_nmap_grid_limits(sv, oracle_mod):
    hi = (1 << 20) - 1
    coords = np.array([[0, 0, 0], [hi, hi, hi], [0, hi, 0], [hi, 0, hi - 1], [hi, 0, hi]], np.int32)
    np.testing.assert_array_equal(gpu_nmap(sv, coords), oracle_mod.build_nmap(coords, W.offsets_3x3x3()))


def test_nmap_errors(sv):
    import torch
    dup = torch.tensor([[1, 2, 3], [4, 5, 6], [1, 2, 3]], dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpconvError) as e:
        sv.build_nmap(dup)
    assert e.value.code == -4
    bad = torch.tensor([[1, 2, 3], [1 << 20, 0, 0]], dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpconvError) as e:
        sv.build_nmap(bad)
    assert e.value.code == -1
    small_ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(sv.SpconvError) as e:
        sv.build_nmap(torch.zeros((3, 3), dtype=torch.int32, device="cuda"), workspace=small_ws)
    assert e.value.code == -3
    # the library stays usable after errors
    ok = torch.tensor([[1, 2, 3], [1, 2, 4]], dtype=torch.int32, device="cuda")
    assert sv.build_nmap(ok)[14, 0].item() == 1


@pytest.mark.parametrize("name", ["medium", "channel", "decoder"])
def test_nmap_large_configs(sv, oracle_mod, name):
    """Full-size maps (1.0 M, 1.9 M and 11.8 M voxels): the whole GPU map
    equals the oracle's bit for bit; the pair count the library reports
    equals the oracle's."""
    import torch
    from helpers import oracle_full_map
    coords, ref = oracle_full_map(name)
    n = len(coords)
    nm = sv.build_nmap(torch.from_numpy(coords).cuda())
    got = nm.cpu().numpy()
    assert got.shape == ref.shape
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        k, c = bad[0]
        raise AssertionError(f"{len(bad)} of {ref.size} entries differ; first at k={k}, n={c}: "
                             f"gpu={got[k, c]} oracle={ref[k, c]}")
    vp = oracle_mod.count_valid_pairs(ref)
    assert sv.count_valid_pairs(nm) == vp
    assert vp >= n


def test_nmap_sorted_paths_dense_and_row_hash(sv, oracle_mod):
    """Sorted input takes the dense-row path when its bounding box fits in the
    workspace (every workload here), else the row hash: the small workload
    with one voxel added at the far corner of the grid (still sorted) has a
    box of 2^60 cells and takes the row hash.  Both give the oracle's map."""
    small = W.coords_only("small")
    np.testing.assert_array_equal(gpu_nmap(sv, small), oracle_mod.build_nmap(small, W.offsets_3x3x3()))
    hi = (1 << 20) - 1
    wide = np.concatenate([small, np.array([[hi, hi, hi]], np.int32)])
    for offs in (W.offsets_3x3x3(), W.offsets_cube(2)):
        np.testing.assert_array_equal(gpu_nmap(sv, wide, offs), oracle_mod.build_nmap(wide, offs))
    # generic offset lists on the dense path too
    np.testing.assert_array_equal(gpu_nmap(sv, small, W.offsets_cube(2)),
                                  oracle_mod.build_nmap(small, W.offsets_cube(2)))


def test_async_build_matches_and_reports_on_device(sv, oracle_mod):
    """spconv_build_nmap_async: the same map, the verdict written to device
    memory (no host wait); two builds in flight on two streams; a duplicate
    coordinate gives SPCONV_ERR_DUPLICATE_COORD in the status word."""
    import torch
    a = W.coords_only("small")
    b = W.random_occupancy(20, 0.3, 9)
    b = b[W.permutation(len(b), 9)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    st = torch.full((2,), 123, dtype=torch.int32, device="cuda")
    ca = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    cb = torch.from_numpy(np.ascontiguousarray(b)).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        ma = sv.build_nmap(ca, status=st[0:1], stream=s1)
    with torch.cuda.stream(s2):
        mb = sv.build_nmap(cb, offsets=W.offsets_cube(2), status=st[1:2], stream=s2)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    np.testing.assert_array_equal(ma.cpu().numpy(), oracle_mod.build_nmap(a, W.offsets_3x3x3()))
    np.testing.assert_array_equal(mb.cpu().numpy(), oracle_mod.build_nmap(b, W.offsets_cube(2)))
    dup = torch.tensor([[1, 2, 3], [4, 5, 6], [1, 2, 3]], dtype=torch.int32, device="cuda")
    sv.build_nmap(dup, status=st[0:1])
    empty = torch.zeros((0, 3), dtype=torch.int32, device="cuda")
    sv.build_nmap(empty, status=st[1:2])
    torch.cuda.synchronize()
    assert st.tolist() == [-4, 0]


def test_nmap_sorted_row_path_cases(sv, oracle_mod):
    """Strictly (z, y, x)-sorted input takes the row-table path, any other
    order the voxel-hash path; both must give the oracle's map exactly.
    Cases aimed at the row path: long dense rows, rows at the grid limits,
    one single row, offset lists with duplicates and large dx, and inputs
    that are sorted except for one swapped pair (hash path)."""
    rng = np.random.default_rng(11)
    hi = (1 << 20) - 1
    dense_row = np.stack([np.full(1000, 3), np.full(1000, 4), np.arange(1000)], axis=1)
    two_runs = np.stack([np.full(40, 3), np.full(40, 5), np.r_[np.arange(20), 500 + np.arange(20)]], axis=1)
    stack = np.stack([np.repeat([2, 3, 4], 300), np.tile(np.repeat([4, 5, 6], 100), 3),
                      np.tile(np.arange(100), 9)], axis=1)
    edges = np.array([[0, 0, 0], [0, 0, 1], [0, 1, 0], [hi, hi, hi - 1], [hi, hi, hi]])
    single = np.stack([np.zeros(64, int), np.zeros(64, int), np.sort(rng.choice(5000, 64, replace=False))], axis=1)
    offset_sets = [
        W.offsets_3x3x3(),
        W.offsets_cube(2),
        np.array([[0, 0, 1], [0, 0, 1], [0, 0, -7], [1, 0, 0], [0, 0, 0], [-1, 2, 3], [0, 0, 7]], np.int32),
    ]
    for coords in (np.concatenate([dense_row, two_runs]), stack, edges, single):
        coords = np.unique(coords.astype(np.int32), axis=0)  # sorted, distinct
        for offs in offset_sets:
            np.testing.assert_array_equal(gpu_nmap(sv, coords, offs), oracle_mod.build_nmap(coords, offs))
        if len(coords) > 2:
            swapped = coords.copy()
            swapped[[0, 1]] = swapped[[1, 0]]
            np.testing.assert_array_equal(gpu_nmap(sv, swapped), oracle_mod.build_nmap(swapped, W.offsets_3x3x3()))
    import torch
    sorted_dup = torch.tensor([[1, 2, 3], [1, 2, 3], [1, 2, 4]], dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpconvError) as e:
        sv.build_nmap(sorted_dup)
    assert e.value.code == -4
