"""spconv_build_nmap_noalloc: the neighbour-map build for callers that cannot
allocate device memory (a host framework that owns every allocation, or a
fixed budget that forbids allocations after start-up).  It keeps its hash
table in a fixed device array of the library instead of a caller workspace.

Called through the C ABI and compared, bit for bit, with the map that the
workspace entry point spconv_build_nmap builds for the same input, on two
calls in a row (the second call reuses the array the first one filled), and
at exactly SPCONV_NOALLOC_MAX_VOXELS voxels (the one size whose table fills
the whole array) also with the oracle's map.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

MAX_VOXELS = 1 << 20  # SPCONV_NOALLOC_MAX_VOXELS in include/spconv.h


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import submanifold_voxel_gather_gb300 as sv
    from submanifold_voxel_gather_gb300 import build
    build.build()
    lib = sv.load_library()
    fn = lib.spconv_build_nmap_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return torch, sv, lib, fn


def _noalloc_map(env, coords_np, offsets):
    torch, sv, lib, fn = env
    coords = torch.from_numpy(np.ascontiguousarray(coords_np, dtype=np.int32)).cuda()
    offs = np.ascontiguousarray(offsets, dtype=np.int32)
    out = torch.full((offs.shape[0], coords.shape[0]), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = fn(coords.data_ptr(), coords.shape[0], offs.ctypes.data_as(ctypes.c_void_p), offs.shape[0],
            out.data_ptr(), stream)
    assert rc == 0, lib.spconv_last_error().decode()
    ref = sv.build_nmap(coords, offs)  # the existing entry point, with a workspace
    return out, ref


def test_noalloc_equals_workspace_build_on_two_calls_in_a_row(env):
    torch = env[0]
    # First call: the small workload (43 k voxels, 27 offsets).
    a = W.coords_only("small")
    out_a, ref_a = _noalloc_map(env, a, W.offsets_3x3x3())
    assert torch.equal(out_a, ref_a)
    # Second call, straight after: a different, shuffled input with 125
    # offsets, so stale table contents from the first call would show.
    b = W.random_occupancy(24, 0.3, 5)
    b = b[W.permutation(len(b), 5)]
    out_b, ref_b = _noalloc_map(env, b, W.offsets_cube(2))
    assert torch.equal(out_b, ref_b)
    assert int((out_b == len(b)).sum()) > 0 and int((out_b < len(b)).sum()) > 0


def test_noalloc_at_its_maximum_size(env, oracle_mod):
    """N = SPCONV_NOALLOC_MAX_VOXELS (a 128 x 128 x 64 block, shuffled so the
    voxel hash is used): its 2^21 slots fill the whole array.  Equal to the
    workspace build and to the oracle's map; then a small call right after
    still gives the right map."""
    torch = env[0]
    g = np.stack(np.meshgrid(np.arange(128), np.arange(128), np.arange(64), indexing="ij"), -1)
    coords = (g.reshape(-1, 3) + np.array([7, 900, 3])).astype(np.int32)
    assert len(coords) == MAX_VOXELS
    coords = coords[W.permutation(len(coords), 21)]
    offs = W.offsets_3x3x3()
    out, ref = _noalloc_map(env, coords, offs)
    assert torch.equal(out, ref)
    np.testing.assert_array_equal(out.cpu().numpy(),
                                  oracle_mod.build_nmap(coords, offs, threads=oracle_mod.host_threads()))
    out_s, ref_s = _noalloc_map(env, W.coords_only("tiny"), offs)
    assert torch.equal(out_s, ref_s)


def test_noalloc_rejects_sizes_above_its_maximum(env):
    torch, sv, lib, fn = env
    offs = W.offsets_3x3x3()
    fake = ctypes.c_void_p(0x100000)  # not dereferenced: the size check comes first
    rc = fn(fake, MAX_VOXELS + 1, offs.ctypes.data_as(ctypes.c_void_p), 27, fake, None)
    assert rc == -2  # SPCONV_ERR_UNSUPPORTED
    assert "SPCONV_NOALLOC_MAX_VOXELS" in lib.spconv_last_error().decode()


def test_noalloc_reports_duplicates(env):
    torch, sv, lib, fn = env
    coords = torch.tensor([[1, 2, 3], [4, 5, 6], [1, 2, 3]], dtype=torch.int32, device="cuda")
    offs = W.offsets_3x3x3()
    out = torch.empty((27, 3), dtype=torch.int32, device="cuda")
    rc = fn(coords.data_ptr(), 3, offs.ctypes.data_as(ctypes.c_void_p), 27, out.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == -4  # SPCONV_ERR_DUPLICATE_COORD
    # and the shared array is usable again afterwards
    out_c, ref_c = _noalloc_map(env, W.coords_only("tiny"), W.offsets_3x3x3())
    assert torch.equal(out_c, ref_c)
