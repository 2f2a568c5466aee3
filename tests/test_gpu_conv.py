"""Fused convolution on the GPU against the oracle's exact result:
|gpu - exact| <= tol * sum|terms| with tol = 1e-5 (f32) and 4e-3 (bf16, tf32)."""
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


def run_gpu(sv, feats, nmap, w, bias, dtype):
    import torch
    f = torch_storage(feats, dtype)
    ww = torch_storage(w, dtype)
    b = None if bias is None else torch_storage(bias, dtype)
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    out = sv.submconv3d(f, nm, ww, b, dtype=("tf32" if dtype == "tf32" else None))
    sv.device_status()
    return to_f64(out)


def layer_values(seed, n, k, ci, co, dtype, bias=True):
    feats = W.values(seed, 11, (n, ci), dtype)
    w = W.values(seed, 12, (k, ci, co), dtype, 1.0 / np.sqrt(k * ci))
    b = W.values(seed, 13, (co,), dtype, 0.1) if bias else None
    return feats, w, b


@pytest.mark.parametrize("name", ["tiny", "tiny_shell1"])
def test_tiny_f32_full(sv, oracle_mod, name):
    wl = W.make(name)
    layer = wl.layers[0]
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    ref, sabs = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "f32")
    got = run_gpu(sv, layer.feats, nmap, layer.w, layer.bias, "f32")
    assert_within(got, ref, sabs, "f32")


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
@pytest.mark.parametrize("name", ["tiny", "tiny_shell1"])
def test_tiny_tensor_core(sv, oracle_mod, name, dtype):
    wl = W.make(name)
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    feats, w, b = layer_values(3, wl.N, 27, 16, 16, dtype)
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, dtype)
    assert_within(run_gpu(sv, feats, nmap, w, b, dtype), ref, sabs, dtype)


def test_small_bf16_full(sv, oracle_mod):
    wl = W.make("small")
    layer = wl.layers[0]
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    ref, sabs = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "bf16",
                                threads=oracle_mod.host_threads())
    assert_within(run_gpu(sv, layer.feats, nmap, layer.w, layer.bias, "bf16"), ref, sabs, "bf16")


@pytest.mark.parametrize("ci,co", [(16, 16), (32, 48), (48, 80), (64, 64), (80, 128), (128, 256),
                                   (256, 128), (384, 96), (64, 272), (16, 512)])
@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
def test_channel_shapes(sv, oracle_mod, ci, co, dtype):
    """Ci / Co not multiples of the 64-element (bf16) or 32-element (tf32)
    chunk, Co above 256 (several launches) and a ragged last tile.  In bf16,
    Ci = 256 and 384 with Co <= 128 take two-chunk stages with per-chunk
    barriers (two and three stages per offset)."""
    coords = W.random_occupancy(14, 0.25, ci + co)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats, w, b = layer_values(ci * 7 + co, len(coords), 27, ci, co, dtype)
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, dtype, threads=oracle_mod.host_threads())
    assert_within(run_gpu(sv, feats, nmap, w, b, dtype), ref, sabs, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "tf32"])
@pytest.mark.parametrize("n", [1, 127, 128, 129, 300])
def test_edge_sizes(sv, oracle_mod, n, dtype):
    coords = W.random_occupancy(12, 0.5, 77)[:n]
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats, w, b = layer_values(n, n, 27, 32, 64, dtype)
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, dtype)
    assert_within(run_gpu(sv, feats, nmap, w, b, dtype), ref, sabs, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "tf32"])
def test_all_sentinel_gives_bias_exactly(sv, oracle_mod, dtype):
    n, k = 300, 27
    feats, w, b = layer_values(8, n, k, 32, 48, dtype)
    for fill in (n, -1, n + 100, -(1 << 31), (1 << 31) - 1):
        nmap = np.full((k, n), fill, dtype=np.int64).astype(np.int32)
        got = run_gpu(sv, feats, nmap, w, b, dtype)
        expect = np.broadcast_to(W.storage_to_f64(b, dtype), (n, 48))
        np.testing.assert_array_equal(got, expect)
        nobias = run_gpu(sv, feats, nmap, w, None, dtype)
        np.testing.assert_array_equal(nobias, np.zeros((n, 48)))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "tf32"])
def test_garbage_invalid_entries_and_no_bias(sv, oracle_mod, dtype):
    coords = W.random_occupancy(12, 0.3, 91)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    d = W.draws_u64(91, 5, 0, nmap.size).reshape(nmap.shape)
    junk = np.array([-1, n + 1, -(1 << 30), (1 << 31) - 1], dtype=np.int64)[(d % np.uint64(4)).astype(np.int64)]
    nmap = np.where(nmap == n, junk, nmap).astype(np.int32)
    feats, w, _ = layer_values(91, n, 27, 48, 32, dtype)
    ref, sabs = oracle_mod.conv(feats, nmap, w, None, dtype)
    assert_within(run_gpu(sv, feats, nmap, w, None, dtype), ref, sabs, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "tf32"])
@pytest.mark.parametrize("k", [1, 8, 33, 64])
def test_other_offset_counts(sv, oracle_mod, k, dtype):
    """K = 1 (centre only: a dense GEMM), and K above one 32-offset slot."""
    coords = W.random_occupancy(12, 0.4, 50 + k)
    n = len(coords)
    offs = W.offsets_3x3x3() if k <= 27 else W.offsets_cube(2)
    offs = offs[13:14] if k == 1 else offs[:k]
    nmap = oracle_mod.build_nmap(coords, offs)
    feats, w, b = layer_values(k, n, k, 32, 32, dtype)
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, dtype)
    assert_within(run_gpu(sv, feats, nmap, w, b, dtype), ref, sabs, dtype)


@pytest.mark.parametrize("ci,co", [(32, 32), (64, 128), (128, 128), (96, 208)])
def test_tf32_runs_tensor_core_products(sv, oracle_mod, ci, co):
    """SPCONV_TF32 takes the tensor-core kernel (kind::tf32): its products use
    operands with 10 mantissa bits, so on inputs whose low mantissa bits are
    set its output differs from the exact-fp32 kernel's (SPCONV_F32) by at
    most what that operand rounding allows (2 * 2^-10 relative per product,
    plus fp32 accumulation), while staying within the tf32 tolerance of the
    oracle.  It also matches the oracle evaluated on the inputs rounded to 10
    mantissa bits (toward zero or to nearest) within the fp32 bound."""
    import torch
    coords = W.random_occupancy(16, 0.3, ci + 3 * co)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats, w, b = layer_values(ci + co, len(coords), 27, ci, co, "f32")
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, "f32", threads=oracle_mod.host_threads())
    got_tf32 = run_gpu(sv, feats, nmap, w, b, "tf32")
    got_f32 = run_gpu(sv, feats, nmap, w, b, "f32")
    assert_within(got_tf32, ref, sabs, "tf32")
    assert_within(got_f32, ref, sabs, "f32")
    assert not np.array_equal(got_tf32, got_f32)
    assert (np.abs(got_tf32 - got_f32) <= (2 * 2.0 ** -10 + 1e-5) * sabs).all()

    def to_tf32(a, nearest):
        bits = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
        if nearest:
            bits = bits + 0x1000 + ((bits >> 13) & 1) - 1   # round half to even at bit 13
        return (bits & np.uint64(0xFFFFE000)).astype(np.uint32).view(np.float32)

    fits = []
    for nearest in (False, True):
        ref_t, sabs_t = oracle_mod.conv(to_tf32(feats, nearest), nmap, to_tf32(w, nearest), b, "f32",
                                        threads=oracle_mod.host_threads())
        fits.append(bool((np.abs(got_tf32 - ref_t) <= 1e-5 * sabs_t).all()))
    assert any(fits), "tf32 output matches neither truncated nor rounded tf32 operands"


def test_isolated_voxels_reduce_to_centre_gemm(sv, oracle_mod):
    """Voxels with no neighbour: out = feats @ w[13] + bias."""
    g = np.arange(0, 40, 3)
    coords = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3).astype(np.int32)[:1000]
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    assert (nmap[np.arange(27) != 13] == len(coords)).all()
    feats, w, b = layer_values(4, len(coords), 27, 64, 64, "bf16")
    got = run_gpu(sv, feats, nmap, w, b, "bf16")
    f = W.storage_to_f64(feats, "bf16")
    ref = f @ W.storage_to_f64(w, "bf16")[13] + W.storage_to_f64(b, "bf16")
    sabs = np.abs(f) @ np.abs(W.storage_to_f64(w, "bf16")[13]) + np.abs(W.storage_to_f64(b, "bf16"))
    assert_within(got, ref, sabs, "bf16")


def test_repeat_calls_are_identical(sv, oracle_mod):
    import torch
    wl = W.make("small")
    layer = wl.layers[0]
    c = torch.from_numpy(wl.coords).cuda()
    nm = sv.build_nmap(c)
    f, w, b = (torch_storage(a, "bf16") for a in (layer.feats, layer.w, layer.bias))
    o1 = sv.submconv3d(f, nm, w, b)
    o2 = sv.submconv3d(f, nm, w, b)
    assert torch.equal(o1, o2)


def _large(sv, oracle_mod, name, li, sample):
    """The product path on the GPU (map build, then the conv, in the bench's
    launch configuration) against the oracle's own path on the host (its map
    by sort + binary search, then its fp64 loop nest), on ``sample`` seeded
    rows plus the first and last 160 (all rows when ``sample`` is None).
    The two paths share no intermediate: the maps are compared in full by
    test_gpu_nmap.py."""
    import torch
    from helpers import oracle_full_map
    wl = W.make(name)
    layer = wl.layers[li]
    c = torch.from_numpy(wl.coords).cuda()
    nm = sv.build_nmap(c)
    f, w, b = (torch_storage(a, layer.dtype) for a in (layer.feats, layer.w, layer.bias))
    out = sv.submconv3d(f, nm, w, b)
    sv.device_status()
    assert torch.isfinite(out.float()).all()
    del nm
    _, ref_map = oracle_full_map(name)
    rows = np.arange(wl.N, dtype=np.int64) if sample is None else sample_rows(wl.N, sample, li + 17)
    ref, sabs = oracle_mod.conv(layer.feats, ref_map, layer.w, layer.bias, layer.dtype, rows=rows,
                                threads=oracle_mod.host_threads())
    got = to_f64(out[torch.from_numpy(rows).cuda()])
    return assert_within(got, ref, sabs, layer.dtype)


def test_medium_bf16_all_rows(sv, oracle_mod):
    _large(sv, oracle_mod, "medium", 0, None)


@pytest.mark.parametrize("li", [0, 1])
def test_channel_bf16_sampled(sv, oracle_mod, li):
    _large(sv, oracle_mod, "channel", li, 1 << 18)


def test_decoder_bf16_sampled(sv, oracle_mod):
    _large(sv, oracle_mod, "decoder", 0, 1 << 20)
