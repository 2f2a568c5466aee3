"""Input gradient (spconv_submconv3d_dgrad) on the GPU against the oracle's
exact sums: |gpu - exact| <= tol * sum|terms|, tol 1e-5 (f32) / 4e-3 (bf16).
The oracle's dgrad is the scatter sum over map entries (no symmetry used);
the GPU computes the forward convolution of dout with w[K-1-k]^T, which
equals it for the point-symmetric mirrored offset lists used here."""
import numpy as np
import pytest

import workloads as W
from helpers import assert_within, sample_rows, to_f64, torch_storage

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


def run_dgrad(sv, dout, nmap, w, dtype):
    import torch
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    got = sv.submconv3d_dgrad(torch_storage(dout, dtype), nm, torch_storage(w, dtype),
                              dtype=("tf32" if dtype == "tf32" else None))
    sv.device_status()
    return to_f64(got)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "tf32"])
@pytest.mark.parametrize("ci,co", [(16, 16), (64, 64), (128, 128), (32, 80), (272, 64), (64, 256), (96, 384)])
def test_dgrad_matches_oracle(sv, oracle_mod, dtype, ci, co):
    """Forward Ci (the dgrad output width) above 256 needs two launches; Co
    (the dgrad reduction width) not a multiple of 64 leaves a partial chunk."""
    coords = W.random_occupancy(14, 0.3, ci * 3 + co)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    dout = W.values(ci + co, 21, (n, co), dtype)
    w = W.values(ci + co, 22, (27, ci, co), dtype, 1.0 / np.sqrt(27 * co))
    ref, dabs = oracle_mod.dgrad(dout, nmap, w, dtype, threads=oracle_mod.host_threads())
    assert_within(run_dgrad(sv, dout, nmap, w, dtype), ref, dabs, dtype)


def test_dgrad_wide_offsets_medium_sample(sv, oracle_mod):
    """125 offsets (5x5x5 cube, also mirrored) on a shuffled occupancy, and
    the medium workload's map checked on sampled rows."""
    coords = W.random_occupancy(20, 0.2, 5)
    coords = coords[W.permutation(len(coords), 5)]
    n = len(coords)
    offs = W.offsets_cube(2)
    assert np.array_equal(offs[::-1], -offs)
    nmap = oracle_mod.build_nmap(coords, offs)
    dout = W.values(7, 21, (n, 64), "bf16")
    w = W.values(7, 22, (125, 32, 64), "bf16", 0.05)
    ref, dabs = oracle_mod.dgrad(dout, nmap, w, "bf16", threads=oracle_mod.host_threads())
    assert_within(run_dgrad(sv, dout, nmap, w, "bf16"), ref, dabs, "bf16")

    wl = W.make("medium")
    layer = wl.layers[0]
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    dout = W.values(8, 21, (wl.N, layer.Co), "bf16")
    got = run_dgrad(sv, dout, nmap, layer.w, "bf16")
    rows = sample_rows(wl.N, 1500, 8)
    ref, dabs = oracle_mod.dgrad(dout, nmap, layer.w, "bf16", rows=rows,
                                 threads=oracle_mod.host_threads())
    assert_within(got[rows], ref, dabs, "bf16")


def test_dgrad_isolated_voxels_get_centre_term_only(sv, oracle_mod):
    """Voxels with no neighbour: dfeats = w[13] dout (centre offset only)."""
    coords = np.array([[2, 2, 2], [2, 2, 9], [9, 2, 2], [9, 9, 9]], dtype=np.int32)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    dout = W.values(9, 21, (4, 32), "f32")
    w = W.values(9, 22, (27, 16, 32), "f32")
    got = run_dgrad(sv, dout, nmap, w, "f32")
    exact = dout.astype(np.float64) @ w[13].astype(np.float64).T
    np.testing.assert_allclose(got, exact, rtol=1e-5, atol=1e-5 * np.abs(exact).max())


# ---------------------------------------------------------------- weight grad
def run_wgrad(sv, feats, dout, nmap, dtype):
    import torch
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    dw, db = sv.submconv3d_wgrad(torch_storage(feats, dtype), torch_storage(dout, dtype), nm)
    sv.device_status()
    return dw.double().cpu().numpy(), db.double().cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ci,co", [(16, 16), (64, 64), (48, 80), (128, 128)])
def test_wgrad_matches_oracle(sv, oracle_mod, dtype, ci, co):
    """fp32 sums of widened inputs: |gpu - exact| <= 1e-5 * sum|terms| for
    both storage types (the result is fp32, not rounded to the storage
    type).  dbias against the plain column sum."""
    coords = W.random_occupancy(15, 0.3, ci * 5 + co)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(ci + co, 31, (n, ci), dtype)
    dout = W.values(ci + co, 32, (n, co), dtype)
    ref, dabs = oracle_mod.wgrad(feats, dout, nmap, dtype)
    dw, db = run_wgrad(sv, feats, dout, nmap, dtype)
    assert_within(dw, ref, dabs, "f32")
    d64 = oracle_mod.widen(dout, dtype)
    assert_within(db, d64.sum(axis=0), np.abs(d64).sum(axis=0), "f32")


def test_wgrad_many_slices_and_wide_offsets(sv, oracle_mod):
    """More voxels than one CTA slice (several atomic partial sums per
    output) on the small workload, 27 offsets; a shuffled 5x5x5 case."""
    wl = W.make("small")
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    feats = W.values(41, 31, (wl.N, 32), "bf16")
    dout = W.values(41, 32, (wl.N, 16), "bf16")
    ref, dabs = oracle_mod.wgrad(feats, dout, nmap, "bf16")
    dw, _ = run_wgrad(sv, feats, dout, nmap, "bf16")
    assert_within(dw, ref, dabs, "f32")

    coords = W.random_occupancy(18, 0.2, 43)
    coords = coords[W.permutation(len(coords), 43)]
    nmap = oracle_mod.build_nmap(coords, W.offsets_cube(2))
    feats = W.values(43, 31, (len(coords), 16), "f32")
    dout = W.values(43, 32, (len(coords), 32), "f32")
    ref, dabs = oracle_mod.wgrad(feats, dout, nmap, "f32")
    dw, _ = run_wgrad(sv, feats, dout, nmap, "f32")
    assert_within(dw, ref, dabs, "f32")


def test_backward_adjoint_on_gpu(sv, oracle_mod):
    """<y, conv(x; w)> = <dgrad(y), x> = <wgrad(x, y), w>, all three computed
    on the GPU in fp32 (exact kernels), within fp32 accumulation error."""
    import torch
    coords = W.random_occupancy(16, 0.3, 51)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    x = W.values(51, 1, (n, 32), "f32")
    w = W.values(51, 2, (27, 32, 48), "f32", 0.1)
    y = W.values(51, 3, (n, 48), "f32")
    nm = torch.from_numpy(nmap).cuda()
    xt, wt, yt = torch_storage(x, "f32"), torch_storage(w, "f32"), torch_storage(y, "f32")
    fwd = sv.submconv3d(xt, nm, wt)
    dx = sv.submconv3d_dgrad(yt, nm, wt)
    dw, _ = sv.submconv3d_wgrad(xt, yt, nm)
    a = float((yt.double() * fwd.double()).sum())
    b = float((dx.double() * xt.double()).sum())
    c = float((dw.double() * wt.double()).sum())
    scale = float((yt.double().abs() * fwd.double().abs()).sum()) + 1.0
    assert abs(a - b) <= 1e-5 * scale and abs(a - c) <= 1e-5 * scale
