"""Pins for the CPU oracle: every check compares it with something other than
itself (brute force, a library dense 3-D cross-correlation, a dense GEMM,
closed forms, invariants and hand-worked numbers).

The formula is the one in the module docstring of the page
"sparse_conv_metal.py" (trellis-2-mrp-mlx, mlx_backend); the sentinel rule is
the kernel body's skip of entries that are not valid rows; the bias is the
one the wrapper adds.  The last group of tests plants plausible mistakes in
the oracle's inputs and checks that a pin catches each one.
"""
import json
import os

import numpy as np
import pytest

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


# ---------------------------------------------------------------- helpers
def brute_force_nmap(coords, offsets):
    """O(N^2 K): compare every shifted coordinate with every voxel."""
    coords = np.asarray(coords, dtype=np.int64)
    N = coords.shape[0]
    nmap = np.full((len(offsets), N), N, dtype=np.int32)
    for k, off in enumerate(np.asarray(offsets, dtype=np.int64)):
        target = coords + off
        eq = (target[:, None, :] == coords[None, :, :]).all(axis=2)  # (N, N)
        hit = eq.any(axis=1)
        nmap[k, hit] = np.argmax(eq, axis=1)[hit]
    return nmap


def dense_xcorr_at_sites(coords, side, feats64, w64, bias64):
    """Scatter features into a zero dense grid, run torch's conv3d (a
    cross-correlation) in float64 with zero padding 1, read the active sites."""
    torch = pytest.importorskip("torch")
    N, Ci = feats64.shape
    K, _, Co = w64.shape
    assert K == 27
    grid = np.zeros((Ci, side, side, side), dtype=np.float64)
    grid[:, coords[:, 0], coords[:, 1], coords[:, 2]] = feats64.T
    weight = np.zeros((Co, Ci, 3, 3, 3), dtype=np.float64)
    for k, (dz, dy, dx) in enumerate(W.offsets_3x3x3()):
        weight[:, :, dz + 1, dy + 1, dx + 1] = w64[k].T
    out = torch.nn.functional.conv3d(torch.from_numpy(grid)[None], torch.from_numpy(weight),
                                     torch.from_numpy(bias64), padding=1)[0].numpy()
    return out[:, coords[:, 0], coords[:, 1], coords[:, 2]].T


def f64(a, dtype):
    return W.storage_to_f64(a, dtype)


def load_golden():
    with open(GOLDEN) as fh:
        return json.load(fh)["examples"]


def golden_arrays(ex):
    coords = np.asarray(ex["coords"], dtype=np.int32)
    K, Ci, Co = 27, ex["Ci"], ex["Co"]
    feats = np.asarray(ex["feats"], dtype=np.float32)
    if "w_listed" in ex:
        w = np.full((K, Ci, Co), 100.0, dtype=np.float32)
        for k, m in ex["w_listed"].items():
            w[int(k)] = np.asarray(m, dtype=np.float32)
    else:
        w = (np.arange(K, dtype=np.float32) + 1.0).reshape(K, 1, 1) * np.ones((K, Ci, Co), np.float32)
    bias = np.asarray(ex["bias"], dtype=np.float32)
    return coords, feats, w, bias


# ---------------------------------------------------------------- nmap pins
@pytest.mark.parametrize("side,frac,seed", [(6, 0.3, 1), (8, 0.6, 2), (10, 0.05, 3), (7, 1.0, 4)])
def test_nmap_matches_brute_force_random(oracle_mod, side, frac, seed):
    coords = W.random_occupancy(side, frac, seed)
    offs = W.offsets_3x3x3()
    np.testing.assert_array_equal(oracle_mod.build_nmap(coords, offs), brute_force_nmap(coords, offs))


def test_nmap_matches_brute_force_tiny_shell(oracle_mod):
    coords = W.coords_only("tiny_shell1")
    assert coords.shape[0] == 1814
    offs = W.offsets_3x3x3()
    np.testing.assert_array_equal(oracle_mod.build_nmap(coords, offs), brute_force_nmap(coords, offs))


def test_nmap_brute_force_shuffled_and_wide_offsets(oracle_mod):
    coords = W.random_occupancy(9, 0.4, 7)
    perm = W.permutation(len(coords), 7)
    coords = coords[perm]
    offs = W.offsets_cube(2)  # 125 offsets
    np.testing.assert_array_equal(oracle_mod.build_nmap(coords, offs), brute_force_nmap(coords, offs))


def test_nmap_invariants_tiny(oracle_mod):
    coords = W.coords_only("tiny")
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    N = coords.shape[0]
    np.testing.assert_array_equal(nmap[13], np.arange(N))           # centre offset is the identity
    for k in range(27):                                             # nmap[k,n]=m  =>  nmap[26-k,m]=n
        n = np.nonzero(nmap[k] < N)[0]
        np.testing.assert_array_equal(nmap[26 - k, nmap[k, n]], n)


@pytest.mark.parametrize("L", [1, 2, 3, 5])
def test_valid_pairs_closed_form_full_cube(oracle_mod, L):
    # Every cell of an L^3 cube active: offset (dz,dy,dx) has (L-|dz|)(L-|dy|)(L-|dx|)
    # valid pairs; summed over {-1,0,1}^3 that is (L + 2(L-1))^3 = (3L-2)^3.
    g = np.arange(L)
    coords = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3).astype(np.int32)
    nmap = oracle_mod.build_nmap(coords + 3, W.offsets_3x3x3())
    assert oracle_mod.count_valid_pairs(nmap) == (3 * L - 2) ** 3


@pytest.mark.parametrize("L", [1, 4, 9])
def test_valid_pairs_closed_form_line(oracle_mod, L):
    # A run of L voxels along x: L centre pairs + 2(L-1) x-neighbour pairs.
    coords = np.stack([np.full(L, 4), np.full(L, 4), np.arange(L) + 4], 1).astype(np.int32)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    assert oracle_mod.count_valid_pairs(nmap) == 3 * L - 2


def test_nmap_grid_edges_and_empty(oracle_mod):
    # Neighbours below 0 or at 2^20 are absent, never wrapped.
    hi = (1 << 20) - 1
    coords = np.array([[0, 0, 0], [hi, hi, hi], [0, hi, 0]], dtype=np.int32)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    expect = np.full((27, 3), 3, dtype=np.int32)
    expect[13] = [0, 1, 2]
    np.testing.assert_array_equal(nmap, expect)
    assert oracle_mod.build_nmap(np.zeros((0, 3), np.int32), W.offsets_3x3x3()).shape == (27, 0)


def test_nmap_rejects_duplicates_and_range(oracle_mod):
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_nmap(np.array([[1, 2, 3], [4, 5, 6], [1, 2, 3]], np.int32), W.offsets_3x3x3())
    assert e.value.code == oracle_mod.ERR_DUPLICATE_COORD
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_nmap(np.array([[1, -2, 3]], np.int32), W.offsets_3x3x3())
    assert e.value.code == oracle_mod.ERR_INVALID_ARG
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.build_nmap(np.array([[1, 1 << 20, 3]], np.int32), W.offsets_3x3x3())


# ---------------------------------------------------------------- conv pins
def test_hand_worked_examples(oracle_mod):
    for ex in load_golden():
        coords, feats, w, bias = golden_arrays(ex)
        nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
        N = coords.shape[0]
        expect_map = np.full((27, N), N, dtype=np.int32)
        for k, row in ex["nonsentinel_entries"].items():
            expect_map[int(k)] = row
        np.testing.assert_array_equal(nmap, expect_map)
        assert oracle_mod.count_valid_pairs(nmap) == ex["valid_pairs"]
        for dtype in ("f32", "bf16"):
            st = lambda a: W.to_storage(a, dtype)
            out, sabs = oracle_mod.conv(st(feats), nmap, st(w), st(bias), dtype)
            np.testing.assert_array_equal(out, np.asarray(ex["out"], np.float64))
            np.testing.assert_array_equal(sabs, np.asarray(ex["sabs"], np.float64))


@pytest.mark.parametrize("side,frac,seed,Ci,Co", [
    (8, 0.3, 11, 4, 5), (10, 0.6, 12, 3, 2), (12, 0.05, 13, 8, 8), (9, 0.95, 14, 2, 6)])
def test_conv_equals_dense_xcorr_random(oracle_mod, side, frac, seed, Ci, Co):
    coords = W.random_occupancy(side, frac, seed)
    N = coords.shape[0]
    feats = W.values(seed, 1, (N, Ci), "f32")
    w = W.values(seed, 2, (27, Ci, Co), "f32", 0.2)
    bias = W.values(seed, 3, (Co,), "f32", 0.1)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    out, sabs = oracle_mod.conv(feats, nmap, w, bias, "f32")
    ref = dense_xcorr_at_sites(coords, side, f64(feats, "f32"), f64(w, "f32"), f64(bias, "f32"))
    assert np.all(np.abs(out - ref) <= 1e-12 * sabs)
    assert np.all(sabs >= np.abs(out) - 1e-12 * sabs)


@pytest.mark.parametrize("name", ["tiny", "tiny_shell1"])
def test_conv_equals_dense_xcorr_tiny_configs(oracle_mod, name):
    wl = W.make(name)
    layer = wl.layers[0]
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    out, sabs = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, layer.dtype)
    ref = dense_xcorr_at_sites(wl.coords, wl.side, f64(layer.feats, "f32"), f64(layer.w, "f32"),
                               f64(layer.bias, "f32"))
    assert np.all(np.abs(out - ref) <= 1e-12 * sabs)


def test_conv_bf16_widening_equals_dense_xcorr(oracle_mod):
    coords = W.random_occupancy(8, 0.5, 21)
    N = coords.shape[0]
    feats = W.values(21, 1, (N, 16), "bf16")
    w = W.values(21, 2, (27, 16, 16), "bf16", 0.1)
    bias = W.values(21, 3, (16,), "bf16", 0.1)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    out, sabs = oracle_mod.conv(feats, nmap, w, bias, "bf16")
    ref = dense_xcorr_at_sites(coords, 8, f64(feats, "bf16"), f64(w, "bf16"), f64(bias, "bf16"))
    assert np.all(np.abs(out - ref) <= 1e-12 * sabs)


def test_centre_offset_only_is_dense_gemm(oracle_mod):
    N, Ci, Co = 300, 24, 40
    feats = W.values(5, 1, (N, Ci), "f32")
    w = W.values(5, 2, (1, Ci, Co), "f32")
    bias = W.values(5, 3, (Co,), "f32")
    nmap = np.arange(N, dtype=np.int32)[None, :]
    out, sabs = oracle_mod.conv(feats, nmap, w, bias, "f32")
    ref = f64(feats, "f32") @ f64(w, "f32")[0] + f64(bias, "f32")
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * sabs.max())
    mag = np.abs(f64(feats, "f32")) @ np.abs(f64(w, "f32")[0]) + np.abs(f64(bias, "f32"))
    np.testing.assert_allclose(sabs, mag, rtol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_sentinel_map_gives_bias_exactly(oracle_mod, dtype):
    N, K, Ci, Co = 50, 27, 16, 32
    feats = W.values(6, 1, (N, Ci), dtype)
    w = W.values(6, 2, (K, Ci, Co), dtype)
    bias = W.values(6, 3, (Co,), dtype)
    for fill in (N, -1, N + 7, np.iinfo(np.int32).max, np.iinfo(np.int32).min):
        nmap = np.full((K, N), fill, dtype=np.int32)
        out, sabs = oracle_mod.conv(feats, nmap, w, bias, dtype)
        np.testing.assert_array_equal(out, np.broadcast_to(f64(bias, dtype), (N, Co)))
        np.testing.assert_array_equal(sabs, np.broadcast_to(np.abs(f64(bias, dtype)), (N, Co)))


def test_invalid_entries_of_any_value_contribute_nothing(oracle_mod):
    coords = W.random_occupancy(8, 0.4, 31)
    N = coords.shape[0]
    feats = W.values(31, 1, (N, 4), "f32")
    w = W.values(31, 2, (27, 4, 3), "f32")
    bias = W.values(31, 3, (3,), "f32")
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    ref, _ = oracle_mod.conv(feats, nmap, w, bias, "f32")
    garbage = nmap.copy()
    bad = garbage == N
    rng = W.draws_u64(31, 9, 0, int(bad.sum()))
    choices = np.array([-1, N + 1, -(1 << 30), 1 << 30], dtype=np.int64)
    garbage[bad] = choices[(rng % np.uint64(4)).astype(np.int64)]
    out, _ = oracle_mod.conv(feats, garbage, w, bias, "f32")
    np.testing.assert_array_equal(out, ref)


def test_linearity_in_feats_and_weights(oracle_mod):
    # Inputs are small integers times powers of two, so a*x + b*y is exact in
    # float32 and both sides are exact sums up to fp64 rounding.
    coords = W.random_occupancy(9, 0.35, 41)
    N = coords.shape[0]
    Ci, Co = 5, 4
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())

    def ints(sid, shape, scale):
        d = W.draws_u64(41, sid, 0, int(np.prod(shape)))
        return ((d % np.uint64(17)).astype(np.float32) - 8.0).reshape(shape) * np.float32(scale)

    f1, f2 = ints(1, (N, Ci), 1.0), ints(2, (N, Ci), 1.0)
    w1, w2 = ints(3, (27, Ci, Co), 0.0625), ints(4, (27, Ci, Co), 0.0625)
    a, b = 3.0, -2.0
    o1, s1 = oracle_mod.conv(f1, nmap, w1, None, "f32")
    o2, s2 = oracle_mod.conv(f2, nmap, w1, None, "f32")
    o12, _ = oracle_mod.conv((a * f1 + b * f2).astype(np.float32), nmap, w1, None, "f32")
    assert np.all(np.abs(o12 - (a * o1 + b * o2)) <= 1e-12 * (abs(a) * s1 + abs(b) * s2))
    p2, t2 = oracle_mod.conv(f1, nmap, w2, None, "f32")
    p12, _ = oracle_mod.conv(f1, nmap, (a * w1 + b * w2).astype(np.float32), None, "f32")
    assert np.all(np.abs(p12 - (a * o1 + b * p2)) <= 1e-12 * (abs(a) * s1 + abs(b) * t2))
    assert np.abs(o1).max() > 1.0  # the check is not vacuous


def test_permutation_equivariance(oracle_mod):
    coords = W.random_occupancy(10, 0.3, 51)
    N = coords.shape[0]
    feats = W.values(51, 1, (N, 6), "bf16")
    w = W.values(51, 2, (27, 6, 7), "bf16")
    bias = W.values(51, 3, (7,), "bf16")
    offs = W.offsets_3x3x3()
    nmap = oracle_mod.build_nmap(coords, offs)
    out, sabs = oracle_mod.conv(feats, nmap, w, bias, "bf16")
    perm = W.permutation(N, 51)
    inv = np.argsort(perm)
    nmap_p = oracle_mod.build_nmap(coords[perm], offs)
    # entries permute as indices: nmap_p[k, i] = inv[nmap[k, perm[i]]] (sentinel stays N)
    expect = nmap[:, perm]
    valid = expect < N
    expect = np.where(valid, inv[np.minimum(expect, N - 1)], N)
    np.testing.assert_array_equal(nmap_p, expect)
    out_p, _ = oracle_mod.conv(feats[perm], nmap_p, w, bias, "bf16")
    np.testing.assert_allclose(out_p, out[perm], rtol=0, atol=1e-12 * sabs.max())


def test_row_selection_and_threads_match_full(oracle_mod):
    wl = W.make("tiny")
    layer = wl.layers[0]
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    full, fs = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "f32")
    rows = np.array([4095, 0, 17, 17, 2048], dtype=np.int64)
    part, ps = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "f32", rows=rows)
    np.testing.assert_array_equal(part, full[rows])
    par, _ = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "f32", threads=4)
    np.testing.assert_array_equal(par, full)


# ------------------------------------------------- planted mistakes are caught
def _dense_pin_holds(oracle_mod, coords, side, feats, w, bias, nmap, w_oracle=None):
    """The dense pin with the oracle fed ``nmap`` (and ``w_oracle``, which
    stands for an oracle that reads the weights wrongly)."""
    out, sabs = oracle_mod.conv(feats, nmap, w if w_oracle is None else w_oracle, bias, "f32")
    ref = dense_xcorr_at_sites(coords, side, f64(feats, "f32"), f64(w, "f32"), f64(bias, "f32"))
    return bool(np.all(np.abs(out - ref) <= 1e-12 * sabs))


def test_planted_mistakes_fail_a_pin(oracle_mod):
    side = 8
    coords = W.random_occupancy(side, 0.4, 61)
    N, C = coords.shape[0], 4
    feats = W.values(61, 1, (N, C), "f32")
    w = W.values(61, 2, (27, C, C), "f32")
    bias = W.values(61, 3, (C,), "f32")
    offs = W.offsets_3x3x3()
    good = oracle_mod.build_nmap(coords, offs)
    assert _dense_pin_holds(oracle_mod, coords, side, feats, w, bias, good)
    # neighbour direction flipped (coords - offset)
    flipped = oracle_mod.build_nmap(coords, -offs)
    assert not _dense_pin_holds(oracle_mod, coords, side, feats, w, bias, flipped)
    # weights read transposed within an offset
    wt = np.ascontiguousarray(np.transpose(w, (0, 2, 1)))
    assert not _dense_pin_holds(oracle_mod, coords, side, feats, w, bias, good, w_oracle=wt)
    # one offset dropped
    dropped = good.copy()
    dropped[5] = N
    assert not _dense_pin_holds(oracle_mod, coords, side, feats, w, bias, dropped)
    # offsets enumerated in (dx, dy, dz) order instead of (dz, dy, dx)
    swapped = oracle_mod.build_nmap(coords, offs[:, ::-1].copy())
    assert not _dense_pin_holds(oracle_mod, coords, side, feats, w, bias, swapped)
    # bias dropped: the hand-worked example catches it
    ex = load_golden()[1]
    gc, gf, gw, gb = golden_arrays(ex)
    gmap = oracle_mod.build_nmap(gc, offs)
    out, _ = oracle_mod.conv(gf, gmap, gw, None, "f32")
    assert not np.array_equal(out, np.asarray(ex["out"], np.float64))


@pytest.mark.parametrize("threads", [2, 3, 7])
def test_threaded_nmap_equals_brute_force(oracle_mod, threads):
    """The threaded build (one sort, voxels split over threads) gives the
    brute-force map, shuffled input and 125 offsets included, and raises the
    same errors."""
    coords = W.random_occupancy(9, 0.45, 13)
    coords = coords[W.permutation(len(coords), 13)]
    for offs in (W.offsets_3x3x3(), W.offsets_cube(2)):
        np.testing.assert_array_equal(oracle_mod.build_nmap(coords, offs, threads=threads),
                                      brute_force_nmap(coords, offs))
    tiny = coords[:threads - 1]  # fewer voxels than threads
    np.testing.assert_array_equal(oracle_mod.build_nmap(tiny, W.offsets_3x3x3(), threads=threads),
                                  brute_force_nmap(tiny, W.offsets_3x3x3()))
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_nmap(np.array([[1, 2, 3], [4, 5, 6], [1, 2, 3]], np.int32), W.offsets_3x3x3(),
                              threads=threads)
    assert e.value.code == oracle_mod.ERR_DUPLICATE_COORD
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_nmap(np.array([[1, 2, 3], [1, 1 << 20, 3]], np.int32), W.offsets_3x3x3(),
                              threads=threads)
    assert e.value.code == oracle_mod.ERR_INVALID_ARG


def test_nmap_rows_equals_full_map_columns(oracle_mod):
    coords = W.random_occupancy(9, 0.5, 71)
    offs = W.offsets_3x3x3()
    full = brute_force_nmap(coords, offs)
    rows = np.array([0, len(coords) - 1, 5, 5, len(coords) // 2], dtype=np.int64)
    np.testing.assert_array_equal(oracle_mod.nmap_rows(coords, offs, rows), full[:, rows])


# ---------------------------------------------------------------- fused epilogue
# conv_fused = act(conv + bias + residual).  Pinned by values of the two
# activations fixed by their definitions, by a library logistic function
# (scipy.special.expit, an independent formula for SiLU = x * logistic(x)),
# and by the library dense cross-correlation with the residual and torch's
# own activations applied.

def test_activation_closed_form_values(oracle_mod):
    # centre offset only, w = identity, no bias: conv = feats exactly
    feats = np.array([[0.0, 1.0, -1.0, 2.5], [-30.0, 40.0, 0.5, -0.25]], dtype=np.float32)
    nmap = np.array([[0, 1]], dtype=np.int32)
    w = np.eye(4, dtype=np.float32)[None]
    out, _ = oracle_mod.conv_fused(feats, nmap, w, None, "f32", act="silu")
    assert out[0, 0] == 0.0
    assert abs(out[0, 1] - 0.7310585786300049) < 1e-15   # 1 / (1 + e^-1)
    assert abs(out[0, 2] + 0.2689414213699951) < 1e-15   # -1 / (1 + e)
    assert abs(out[1, 0]) < 1e-11 and abs(out[1, 1] - 40.0) < 1e-15
    out, _ = oracle_mod.conv_fused(feats, nmap, w, None, "f32", act="relu")
    np.testing.assert_array_equal(out, np.maximum(feats, 0).astype(np.float64))


def test_fused_epilogue_matches_library_logistic(oracle_mod):
    special = pytest.importorskip("scipy.special")
    coords = W.random_occupancy(10, 0.3, 21)
    N = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(51, 1, (N, 16), "f32")
    w = W.values(51, 2, (27, 16, 8), "f32", 0.1)
    bias = W.values(51, 3, (8,), "f32")
    res = W.values(51, 4, (N, 8), "f32")
    pre, _ = oracle_mod.conv(feats, nmap, w, bias, "f32")
    pre = pre + res.astype(np.float64)
    out, scale = oracle_mod.conv_fused(feats, nmap, w, bias, "f32", residual=res, act="silu")
    np.testing.assert_allclose(out, pre * special.expit(pre), rtol=1e-13, atol=1e-13)
    out, _ = oracle_mod.conv_fused(feats, nmap, w, bias, "f32", residual=res, act="relu")
    np.testing.assert_array_equal(out, np.where(pre > 0, pre, 0.0))
    assert np.all(scale >= 1.1 * np.abs(res) - 1e-12)


@pytest.mark.parametrize("act", ["relu", "silu"])
def test_fused_epilogue_equals_dense_xcorr(oracle_mod, act):
    torch = pytest.importorskip("torch")
    side = 9
    coords = W.random_occupancy(side, 0.35, 31)
    N = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(52, 1, (N, 8), "f32")
    w = W.values(52, 2, (27, 8, 16), "f32", 0.2)
    bias = W.values(52, 3, (16,), "f32")
    res = W.values(52, 4, (N, 16), "f32")
    dense = dense_xcorr_at_sites(coords, side, f64(feats, "f32"), f64(w, "f32"), f64(bias, "f32"))
    pre = torch.from_numpy(dense + res.astype(np.float64))
    ref = (torch.nn.functional.silu(pre) if act == "silu" else torch.nn.functional.relu(pre)).numpy()
    out, _ = oracle_mod.conv_fused(feats, nmap, w, bias, "f32", residual=res, act=act)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # activation before the residual add is a different (wrong) order
    wrong = (torch.nn.functional.silu(torch.from_numpy(dense)) if act == "silu"
             else torch.nn.functional.relu(torch.from_numpy(dense))).numpy() + res
    assert not np.allclose(out, wrong, rtol=1e-6, atol=1e-6)


def test_fused_epilogue_without_extras_is_conv(oracle_mod):
    coords = W.random_occupancy(8, 0.4, 41)
    N = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(53, 1, (N, 16), "f32")
    w = W.values(53, 2, (27, 16, 16), "f32")
    a, sa = oracle_mod.conv(feats, nmap, w, None, "f32")
    b, sb = oracle_mod.conv_fused(feats, nmap, w, None, "f32")
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(sa, sb)


# ---------------------------------------------------------------- backward
# dgrad / wgrad are the chain rule applied to the forward formula.  Pinned by
# torch autograd through the library dense cross-correlation (gradients read
# at the active sites, with the output gradient zero off them), and by the
# exact adjoint identities against the (already pinned) forward sum:
#   <y, conv(x; w)> = <dgrad(y; w), x> = <wgrad(x, y), w>   (no bias).

def _backward_case(oracle_mod, side, frac, seed, ci, co, dtype="f32"):
    coords = W.random_occupancy(side, frac, seed)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    x = W.values(seed, 1, (n, ci), dtype)
    w = W.values(seed, 2, (27, ci, co), dtype, 0.3)
    y = W.values(seed, 3, (n, co), dtype)
    return coords, nmap, x, w, y


def test_backward_equals_dense_autograd(oracle_mod):
    torch = pytest.importorskip("torch")
    side = 8
    coords, nmap, x, w, y = _backward_case(oracle_mod, side, 0.4, 101, 6, 5)
    ci, co = x.shape[1], y.shape[1]
    grid = torch.zeros((1, ci, side, side, side), dtype=torch.float64)
    grid[0, :, coords[:, 0], coords[:, 1], coords[:, 2]] = torch.from_numpy(f64(x, "f32").T)
    grid.requires_grad_(True)
    weight = torch.zeros((co, ci, 3, 3, 3), dtype=torch.float64)
    for k, (dz, dy, dx) in enumerate(W.offsets_3x3x3()):
        weight[:, :, dz + 1, dy + 1, dx + 1] = torch.from_numpy(f64(w, "f32")[k].T)
    weight.requires_grad_(True)
    out = torch.nn.functional.conv3d(grid, weight, padding=1)
    ymask = torch.zeros_like(out)
    ymask[0, :, coords[:, 0], coords[:, 1], coords[:, 2]] = torch.from_numpy(f64(y, "f32").T)
    gx, gw = torch.autograd.grad((out * ymask).sum(), (grid, weight))
    ref_dx = gx[0, :, coords[:, 0], coords[:, 1], coords[:, 2]].T.numpy()
    ref_dw = np.stack([gw[:, :, dz + 1, dy + 1, dx + 1].T.numpy()
                       for dz, dy, dx in W.offsets_3x3x3()])
    dx_, _ = oracle_mod.dgrad(y, nmap, w, "f32")
    dw_, _ = oracle_mod.wgrad(x, y, nmap, "f32")
    np.testing.assert_allclose(dx_, ref_dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw_, ref_dw, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_adjoint_identities(oracle_mod, dtype):
    coords, nmap, x, w, y = _backward_case(oracle_mod, 11, 0.3, 102, 16, 24, dtype)
    fwd, _ = oracle_mod.conv(x, nmap, w, None, dtype)
    dx_, _ = oracle_mod.dgrad(y, nmap, w, dtype)
    dw_, _ = oracle_mod.wgrad(x, y, nmap, dtype)
    lhs = float(np.sum(f64(y, dtype) * fwd))
    assert abs(lhs - float(np.sum(dx_ * f64(x, dtype)))) <= 1e-9 * max(1.0, abs(lhs))
    assert abs(lhs - float(np.sum(dw_ * f64(w, dtype)))) <= 1e-9 * max(1.0, abs(lhs))


def test_dgrad_is_flipped_transposed_conv_on_symmetric_offsets(oracle_mod):
    """With offsets[K-1-k] = -offsets[k] the input gradient is a forward
    convolution of dout with weights w[K-1-k]^T (the form the GPU uses)."""
    _, nmap, _, w, y = _backward_case(oracle_mod, 10, 0.35, 103, 8, 12)
    offs = W.offsets_3x3x3()
    assert np.array_equal(offs[::-1], -offs)
    dx_, _ = oracle_mod.dgrad(y, nmap, w, "f32")
    wt = np.ascontiguousarray(np.transpose(w[::-1], (0, 2, 1)))
    via_fwd, _ = oracle_mod.conv(y, nmap, wt, None, "f32")
    np.testing.assert_allclose(dx_, via_fwd, rtol=1e-12, atol=1e-12)


def test_backward_row_and_entry_selection(oracle_mod):
    _, nmap, x, w, y = _backward_case(oracle_mod, 9, 0.4, 104, 16, 16)
    n = x.shape[0]
    rows = np.array([0, 3, n // 2, n - 1], dtype=np.int64)
    full, fabs_ = oracle_mod.dgrad(y, nmap, w, "f32")
    part, pabs = oracle_mod.dgrad(y, nmap, w, "f32", rows=rows, threads=2)
    np.testing.assert_array_equal(part, full[rows])
    np.testing.assert_array_equal(pabs, fabs_[rows])
    dw_full, _ = oracle_mod.wgrad(x, y, nmap, "f32")
    entries = np.array([0, 17, 27 * 16 * 16 - 1, 5 * 256 + 3 * 16 + 9], dtype=np.int64)
    dw_part, _ = oracle_mod.wgrad(x, y, nmap, "f32", entries=entries)
    np.testing.assert_allclose(dw_part, dw_full.reshape(-1)[entries], rtol=1e-13, atol=1e-13)


def test_backward_planted_mistake_fails_adjoint(oracle_mod):
    """Feeding dgrad the unflipped map direction (nmap rows reversed) breaks
    the adjoint identity, so that pin would catch an offset-order slip."""
    _, nmap, x, w, y = _backward_case(oracle_mod, 10, 0.35, 105, 8, 8)
    fwd, _ = oracle_mod.conv(x, nmap, w, None, "f32")
    bad, _ = oracle_mod.dgrad(y, np.ascontiguousarray(nmap[::-1]), w, "f32")
    lhs = float(np.sum(f64(y, "f32") * fwd))
    assert abs(lhs - float(np.sum(bad * f64(x, "f32")))) > 1e-6 * max(1.0, abs(lhs))
