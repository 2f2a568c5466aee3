"""x-run slot layout and the row-shifted convolution on the GPU.

The layout is compared entry for entry with its definition written out in
numpy (runs of consecutive indices with consecutive x on one line; one
separator between runs whose outer cells have equal map entries in all nine
(dz, dy) groups, else two; outer separators of the first and last voxel only
when one of their outer cells is active).  The convolution is compared with
the oracle's exact sum (|gpu - exact| <= 4e-3 * sum|terms|) and with the
plain tensor-core convolution: the two add each output's products in
different orders (the row-shifted kernel runs a group's three offsets chunk
by chunk), so their fp32 sums may round to neighbouring bf16 values; they
must agree to within one bf16 rounding step everywhere."""
import numpy as np
import pytest

import workloads as W
from helpers import assert_within, layout_reference, sample_rows, to_f64, torch_storage

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


def assert_near_plain(out, plain, scale=None):
    """Within one bf16 rounding step (2^-7 of the larger magnitude) of the
    plain convolution everywhere, plus 1e-4 of the output's sum |terms|
    (``scale``, numpy; else the largest |output|) for the different fp32
    summation order, and equal on most entries."""
    import torch
    a, b = out.float(), plain.float()
    diff = (a - b).abs()
    slack = (1e-4 * torch.from_numpy(np.asarray(scale, np.float32)).to(a.device) if scale is not None
             else 1e-4 * b.abs().max())
    step = 2.0 ** -7 * a.abs().maximum(b.abs()) + slack
    assert bool((diff <= step).all()), float((diff / step).max())
    assert float((diff == 0).float().mean()) >= 0.9


def gpu_layout(sv, coords, nmap):
    import torch
    c = torch.from_numpy(np.ascontiguousarray(coords, dtype=np.int32)).cuda()
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    slots, count = sv.xrun_layout(c, nm)
    s = int(count.item())
    return slots[:s].cpu().numpy(), nm, slots, count


def shapes():
    rng = np.random.default_rng(5)
    out = {
        "random": W.random_occupancy(16, 0.3, 41),
        "dense": W.random_occupancy(12, 0.9, 42),
        "line": np.array([[3, 4, x] for x in range(700)], np.int32),
        "isolated": np.array([[2 * z, 2 * y, 2 * x] for z in range(9) for y in range(9) for x in range(9)],
                             np.int32),
        "single": np.array([[5, 5, 5]], np.int32),
    }
    sh = W.random_occupancy(16, 0.3, 43)
    out["shuffled"] = sh[rng.permutation(len(sh))]
    return out


@pytest.mark.parametrize("name", ["random", "dense", "line", "isolated", "single", "shuffled"])
def test_layout_matches_definition(sv, oracle_mod, name):
    coords = shapes()[name]
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    got, _, _, _ = gpu_layout(sv, coords, nmap)
    ref = layout_reference(coords, nmap)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)
    # every voxel appears exactly once
    v = got[got >= 0]
    assert np.array_equal(np.sort(v), np.arange(len(coords)))


def run_xrun(sv, coords, nmap, feats, w, b):
    import torch
    _, nm, slots, count = gpu_layout(sv, coords, nmap)
    f, ww = torch_storage(feats, "bf16"), torch_storage(w, "bf16")
    bb = None if b is None else torch_storage(b, "bf16")
    out = sv.submconv3d_xrun(f, nm, slots, count, ww, bb)
    plain = sv.submconv3d(f, nm, ww, bb)
    sv.device_status()
    return out, plain


@pytest.mark.parametrize("co", [16, 64, 128])
@pytest.mark.parametrize("name", ["random", "dense", "line", "isolated", "single", "shuffled"])
def test_xrun_conv_matches_oracle_and_plain(sv, oracle_mod, name, co):
    coords = shapes()[name]
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(co + n, 11, (n, 128), "bf16")
    w = W.values(co + n, 12, (27, 128, co), "bf16", 1.0 / np.sqrt(27 * 128))
    b = W.values(co + n, 13, (co,), "bf16", 0.1)
    out, plain = run_xrun(sv, coords, nmap, feats, w, b)
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, "bf16", threads=oracle_mod.host_threads())
    assert_within(to_f64(out), ref, sabs, "bf16")
    assert_near_plain(out, plain, sabs)


def test_xrun_conv_without_bias(sv, oracle_mod):
    coords = shapes()["random"]
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(7, 11, (n, 128), "bf16")
    w = W.values(7, 12, (27, 128, 128), "bf16", 1.0 / np.sqrt(27 * 128))
    out, plain = run_xrun(sv, coords, nmap, feats, w, None)
    ref, sabs = oracle_mod.conv(feats, nmap, w, None, "bf16", threads=oracle_mod.host_threads())
    assert_within(to_f64(out), ref, sabs, "bf16")
    assert_near_plain(out, plain, sabs)


@pytest.mark.parametrize("workload", ["medium", "decoder"])
def test_xrun_conv_workload_sample(sv, oracle_mod, workload):
    """Full-size seeded workloads: the layout against its definition, the
    conv near the plain conv everywhere and against the oracle on sampled
    rows."""
    import torch
    wl = W.make(workload)
    layer = wl.layers[0]
    coords = wl.coords
    c = torch.from_numpy(coords).cuda()
    nm = sv.build_nmap(c)
    slots, count = sv.xrun_layout(c, nm)
    s = int(count.item())
    nmap = nm.cpu().numpy()
    if workload == "medium":
        assert np.array_equal(slots[:s].cpu().numpy(), layout_reference(coords, nmap))
    f, ww = torch_storage(layer.feats, "bf16"), torch_storage(layer.w, "bf16")
    bb = torch_storage(layer.bias, "bf16")
    out = sv.submconv3d_xrun(f, nm, slots, count, ww, bb)
    plain = sv.submconv3d(f, nm, ww, bb)
    sv.device_status()
    assert_near_plain(out, plain)
    rows = sample_rows(wl.N, 1500, seed=3)
    ref, sabs = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "bf16", rows=rows,
                                threads=oracle_mod.host_threads())
    got = to_f64(out[torch.from_numpy(rows).cuda()])
    assert_within(got, ref, sabs, "bf16")


@pytest.mark.parametrize("act", ["relu", "silu", None])
@pytest.mark.parametrize("name,co", [("random", 128), ("line", 48), ("shuffled", 128), ("single", 16)])
def test_xrun_fused_epilogue_matches_oracle(sv, oracle_mod, name, co, act):
    """out = act(conv + bias + residual) over the layout: against the
    oracle (tolerance scaled by the activation's slope bound, as for the
    voxel-tile epilogue) and near the voxel-tile kernel's fused epilogue."""
    coords = shapes()[name]
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(co + n, 31, (n, 128), "bf16")
    w = W.values(co + n, 32, (27, 128, co), "bf16", 1.0 / np.sqrt(27 * 128))
    b = W.values(co + n, 33, (co,), "bf16", 0.1)
    res = W.values(co + n, 34, (n, co), "bf16")
    ref, scale = oracle_mod.conv_fused(feats, nmap, w, b, "bf16", residual=res, act=act or "none",
                                       threads=oracle_mod.host_threads())
    _, nm, slots, count = gpu_layout(sv, coords, nmap)
    f, ww, bb, r = (torch_storage(x, "bf16") for x in (feats, w, b, res))
    out = sv.submconv3d_xrun(f, nm, slots, count, ww, bb, residual=r, activation=act)
    tiles = sv.submconv3d(f, nm, ww, bb, residual=r, activation=act)
    sv.device_status()
    assert_within(to_f64(out), ref, scale, "bf16")
    assert_near_plain(out, tiles, scale)


@pytest.mark.parametrize("act", ["relu", None])
def test_xrun_fused_epilogue_in_place_and_without_residual(sv, oracle_mod, act):
    """out is the residual buffer itself; and an activation alone."""
    coords = shapes()["dense"]
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(5, 41, (n, 128), "bf16")
    w = W.values(5, 42, (27, 128, 128), "bf16", 1.0 / np.sqrt(27 * 128))
    b = W.values(5, 43, (128,), "bf16", 0.1)
    res = W.values(5, 44, (n, 128), "bf16")
    _, nm, slots, count = gpu_layout(sv, coords, nmap)
    f, ww, bb, r = (torch_storage(x, "bf16") for x in (feats, w, b, res))
    got = sv.submconv3d_xrun(f, nm, slots, count, ww, bb, out=r, residual=r, activation=act)
    assert got.data_ptr() == r.data_ptr()
    ref, scale = oracle_mod.conv_fused(feats, nmap, w, b, "bf16", residual=res, act=act or "none",
                                       threads=oracle_mod.host_threads())
    assert_within(to_f64(got), ref, scale, "bf16")
    if act is not None:
        got2 = sv.submconv3d_xrun(f, nm, slots, count, ww, bb, activation=act)
        ref2, scale2 = oracle_mod.conv_fused(feats, nmap, w, b, "bf16", residual=None, act=act,
                                             threads=oracle_mod.host_threads())
        assert_within(to_f64(got2), ref2, scale2, "bf16")
    sv.device_status()


@pytest.mark.parametrize("ci", [16, 64, 128])
@pytest.mark.parametrize("name", ["random", "dense", "line", "isolated", "shuffled"])
def test_xrun_dgrad_matches_oracle_and_plain(sv, oracle_mod, name, ci):
    """Input gradient over the layout: Co = 128 reduced channels, Ci output
    channels; against the oracle's scatter sum and the plain input gradient."""
    import torch
    coords = shapes()[name]
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    dout = W.values(ci + n, 21, (n, 128), "bf16")
    w = W.values(ci + n, 22, (27, ci, 128), "bf16", 1.0 / np.sqrt(27 * 128))
    _, nm, slots, count = gpu_layout(sv, coords, nmap)
    d, ww = torch_storage(dout, "bf16"), torch_storage(w, "bf16")
    got = sv.submconv3d_dgrad_xrun(d, nm, slots, count, ww)
    plain = sv.submconv3d_dgrad(d, nm, ww)
    sv.device_status()
    ref, dabs = oracle_mod.dgrad(dout, nmap, w, "bf16", threads=oracle_mod.host_threads())
    assert_within(to_f64(got), ref, dabs, "bf16")
    assert_near_plain(got, plain, dabs)



@pytest.mark.parametrize("name", ["random", "dense", "line", "isolated", "single", "shuffled", "small", "wide"])
def test_fused_build_and_layout_equal_the_two_calls(sv, oracle_mod, name):
    """spconv_build_nmap_xrun gives the oracle's map and the layout of its
    definition (the dense-row build writes the layout's flags itself; shuffled
    input and a box too large for the dense rows take the other build paths,
    where the layout reads the map), equal to build_nmap + xrun_layout."""
    import torch
    if name == "small":
        coords = W.coords_only("small")
    elif name == "wide":  # sorted, but a bounding box of 2^60 cells: the row-hash build
        coords = np.concatenate([W.coords_only("small"), np.array([[(1 << 20) - 1] * 3], np.int32)])
    else:
        coords = shapes()[name]
    c = torch.from_numpy(np.ascontiguousarray(coords, dtype=np.int32)).cuda()
    nm, slots, count = sv.build_nmap_xrun(c)
    s = int(count.item())
    ref_map = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    np.testing.assert_array_equal(nm.cpu().numpy(), ref_map)
    np.testing.assert_array_equal(slots[:s].cpu().numpy(), layout_reference(coords, ref_map))
    nm2 = sv.build_nmap(c)
    slots2, count2 = sv.xrun_layout(c, nm2)
    assert int(count2.item()) == s
    assert torch.equal(slots[:s], slots2[:s])
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    nm3, slots3, count3 = sv.build_nmap_xrun(c, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(nm3, nm) and int(count3.item()) == s
    assert torch.equal(slots3[:s], slots[:s])


def test_fused_build_and_layout_at_full_size(sv, oracle_mod):
    """Decoder-scale workload (11.8 M voxels, dense-row build): the fused
    call's map and layout equal the two separate calls'."""
    import torch
    c = torch.from_numpy(W.coords_only("decoder")).cuda()
    nm, slots, count = sv.build_nmap_xrun(c)
    nm2 = sv.build_nmap(c)
    slots2, count2 = sv.xrun_layout(c, nm2)
    assert torch.equal(nm, nm2)
    assert int(count.item()) == int(count2.item())
    s = int(count.item())
    assert torch.equal(slots[:s], slots2[:s])


def bracketed_runs_layout(coords, seed):
    """Another valid layout of the same voxels: every run between its own
    left and right separator (none shared), the runs in a seeded random
    order.  Voxels of one 16- or 32-slot chunk then do not have consecutive
    indices, which the fused epilogue's residual windows must handle."""
    n = len(coords)
    c = coords.astype(np.int64)
    cont = np.zeros(n, bool)
    cont[:-1] = (c[1:, 0] == c[:-1, 0]) & (c[1:, 1] == c[:-1, 1]) & (c[1:, 2] == c[:-1, 2] + 1)
    starts = np.concatenate([[0], np.nonzero(~cont[:-1])[0] + 1])
    ends = np.concatenate([starts[1:], [n]])
    runs = [np.concatenate([[-3 - 2 * a], np.arange(a, b), [-2 - 2 * (b - 1)]]) for a, b in zip(starts, ends)]
    order = np.random.default_rng(seed).permutation(len(runs))
    return np.concatenate([runs[i] for i in order]).astype(np.int32)


@pytest.mark.parametrize("name", ["random", "dense", "line"])
def test_xrun_conv_on_a_shuffled_bracketed_layout(sv, oracle_mod, name):
    """The conv, its fused epilogue and the input gradient on a layout whose
    runs come in random order: the same sums as on the regular layout."""
    import torch
    coords = shapes()[name]
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    slots_np = bracketed_runs_layout(coords, seed=n)
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    slots = torch.from_numpy(slots_np).cuda()
    count = torch.tensor([len(slots_np)], dtype=torch.int64, device="cuda")
    feats = W.values(n, 51, (n, 128), "bf16")
    w = W.values(n, 52, (27, 128, 128), "bf16", 1.0 / np.sqrt(27 * 128))
    b = W.values(n, 53, (128,), "bf16", 0.1)
    res = W.values(n, 54, (n, 128), "bf16")
    f, ww, bb, r = (torch_storage(x, "bf16") for x in (feats, w, b, res))
    out = sv.submconv3d_xrun(f, nm, slots, count, ww, bb)
    fused = sv.submconv3d_xrun(f, nm, slots, count, ww, bb, residual=r, activation="silu")
    dg = sv.submconv3d_dgrad_xrun(f, nm, slots, count, ww)
    sv.device_status()
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, "bf16", threads=oracle_mod.host_threads())
    assert_within(to_f64(out), ref, sabs, "bf16")
    assert_near_plain(out, sv.submconv3d(f, nm, ww, bb), sabs)
    fref, fscale = oracle_mod.conv_fused(feats, nmap, w, b, "bf16", residual=res, act="silu",
                                         threads=oracle_mod.host_threads())
    assert_within(to_f64(fused), fref, fscale, "bf16")
    dref, dabs = oracle_mod.dgrad(feats, nmap, w, "bf16", threads=oracle_mod.host_threads())
    assert_within(to_f64(dg), dref, dabs, "bf16")


def test_xrun_fused_epilogue_full_size_sample(sv, oracle_mod):
    """Medium workload at full size (1.0 M voxels, 1.12 M slots), residual
    + SiLU in place: sampled rows against the oracle, every row near the
    voxel-tile kernel's fused epilogue."""
    import torch
    wl = W.make("medium")
    layer = wl.layers[0]
    c = torch.from_numpy(wl.coords).cuda()
    nm, slots, count = sv.build_nmap_xrun(c)
    res = W.values(77, 61, (wl.N, layer.Co), "bf16")
    f, ww, bb = (torch_storage(x, "bf16") for x in (layer.feats, layer.w, layer.bias))
    r = torch_storage(res, "bf16")
    tiles = sv.submconv3d(f, nm, ww, bb, residual=r, activation="silu")
    out = r.clone()
    sv.submconv3d_xrun(f, nm, slots, count, ww, bb, out=out, residual=out, activation="silu")
    sv.device_status()
    assert_near_plain(out, tiles)
    rows = sample_rows(wl.N, 1500, seed=8)
    ref, scale = oracle_mod.conv_fused(layer.feats, nm.cpu().numpy(), layer.w, layer.bias, "bf16", residual=res,
                                       act="silu", rows=rows, threads=oracle_mod.host_threads())
    assert_within(to_f64(out[torch.from_numpy(rows).cuda()]), ref, scale, "bf16")
