"""Tile order (spconv_tile_order) and the convolution along it
(spconv_submconv3d_ordered): the order is a chunk-local permutation sorted by
neighbour mask, and the ordered convolution equals the plain one bit for bit
(and so the oracle within the tolerance)."""
import numpy as np
import pytest

import workloads as W
from helpers import assert_within, sample_rows, to_f64, torch_storage

pytestmark = pytest.mark.gpu

CHUNK = 4096


@pytest.fixture(scope="module")
def sv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import submanifold_voxel_gather_gb300 as mod
    from submanifold_voxel_gather_gb300 import build
    build.build()
    return mod


def masks(nmap):
    k, n = nmap.shape
    v = (nmap >= 0) & (nmap < n)
    m = np.zeros(n, np.int64)
    for j in range(min(k, 32)):
        m |= v[j].astype(np.int64) << j
    return m


def check_order(order, nmap):
    n = nmap.shape[1]
    assert np.array_equal(np.sort(order), np.arange(n))           # a permutation
    slots = np.arange(n)
    assert np.array_equal(order // CHUNK, slots // CHUNK)          # stays in its chunk
    m = masks(nmap)[order]
    for c0 in range(0, n, CHUNK):                                  # sorted by (mask, index)
        mm, oo = m[c0:c0 + CHUNK], order[c0:c0 + CHUNK]
        key = mm * (1 << 32) + oo
        assert np.all(np.diff(key) > 0)


@pytest.mark.parametrize("name", ["tiny", "small", "channel"])
def test_tile_order_is_a_sorted_chunk_local_permutation(sv, name):
    import torch
    coords = W.coords_only(name)
    nm = sv.build_nmap(torch.from_numpy(coords).cuda())
    order = sv.tile_order(nm).cpu().numpy()
    check_order(order, nm.cpu().numpy())


def test_tile_order_edge_sizes(sv):
    import torch
    base = W.random_occupancy(24, 0.45, 21)
    for n in (1, 2, CHUNK - 1, CHUNK, CHUNK + 1):
        c = torch.from_numpy(np.ascontiguousarray(base[:n])).cuda()
        nm = sv.build_nmap(c)
        check_order(sv.tile_order(nm).cpu().numpy(), nm.cpu().numpy())
    # more than 32 offsets: only the first 32 enter the mask
    c = torch.from_numpy(np.ascontiguousarray(base[:3000])).cuda()
    nm = sv.build_nmap(c, W.offsets_cube(2))
    check_order(sv.tile_order(nm).cpu().numpy(), nm.cpu().numpy())


def layer(seed, n, k, ci, co, dtype="bf16"):
    return (W.values(seed, 11, (n, ci), dtype), W.values(seed, 12, (k, ci, co), dtype, 1.0 / np.sqrt(k * ci)),
            W.values(seed, 13, (co,), dtype, 0.1))


@pytest.mark.parametrize("name,ci,co", [("tiny_shell1", 16, 16), ("small", 64, 64), ("small", 48, 272),
                                         ("channel", 256, 128), ("channel", 64, 256)])
def test_ordered_conv_equals_plain_conv(sv, oracle_mod, name, ci, co):
    import torch
    coords = W.coords_only(name)
    n = len(coords)
    nm = sv.build_nmap(torch.from_numpy(coords).cuda())
    order = sv.tile_order(nm)
    feats, w, b = layer(5, n, 27, ci, co)
    f, ww, bb = torch_storage(feats, "bf16"), torch_storage(w, "bf16"), torch_storage(b, "bf16")
    plain = sv.submconv3d(f, nm, ww, bb)
    ordered = sv.submconv3d(f, nm, ww, bb, order=order)
    sv.device_status()
    assert torch.equal(plain, ordered)
    rows = sample_rows(n, 600, 3) if n > 20000 else None
    ref, sabs = oracle_mod.conv(feats, nm.cpu().numpy(), w, b, "bf16", rows=rows,
                                threads=oracle_mod.host_threads())
    got = to_f64(ordered) if rows is None else to_f64(ordered[torch.from_numpy(rows).cuda()])
    assert_within(got, ref, sabs, "bf16")


def test_order_entries_outside_range_are_empty_slots(sv):
    """Slots whose order entry is outside [0, N) write nothing; every other
    row is the plain convolution's."""
    import torch
    coords = W.coords_only("tiny")
    n = len(coords)
    nm = sv.build_nmap(torch.from_numpy(coords).cuda())
    feats, w, b = layer(6, n, 27, 32, 32)
    f, ww, bb = torch_storage(feats, "bf16"), torch_storage(w, "bf16"), torch_storage(b, "bf16")
    plain = sv.submconv3d(f, nm, ww, bb)
    order = torch.arange(n, dtype=torch.int32, device="cuda")
    order[5] = -1
    order[700] = n
    out = torch.full((n, 32), 7.0, dtype=torch.bfloat16, device="cuda")
    sv.submconv3d(f, nm, ww, bb, out=out, order=order)
    sv.device_status()
    keep = torch.ones(n, dtype=torch.bool, device="cuda")
    keep[5] = False
    keep[700] = False
    assert torch.equal(out[keep], plain[keep])
    assert bool((out[~keep] == 7.0).all())


def test_ordered_f32_equals_plain(sv):
    import torch
    coords = W.coords_only("tiny")
    n = len(coords)
    nm = sv.build_nmap(torch.from_numpy(coords).cuda())
    feats, w, b = layer(7, n, 27, 16, 16, "f32")
    f, ww, bb = torch_storage(feats, "f32"), torch_storage(w, "f32"), torch_storage(b, "f32")
    assert torch.equal(sv.submconv3d(f, nm, ww, bb), sv.submconv3d(f, nm, ww, bb, order=sv.tile_order(nm)))
