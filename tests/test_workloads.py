"""The seeded input generator: determinism, geometry and value recipes."""
import numpy as np
import pytest

import workloads as W


def _brute_shell(side, c, r, h):
    g = np.stack(np.meshgrid(*[np.arange(side)] * 3, indexing="ij"), -1).reshape(-1, 3)
    d = np.sqrt(((g - np.asarray(c, np.float64)) ** 2).sum(1))
    return g[np.abs(d - r) < h].astype(np.int32)


@pytest.mark.parametrize("c,r,h", [((16.0, 16.0, 16.0), 12.0, 0.5), ((16.0, 16.0, 16.0), 12.0, 1.5),
                                   ((20.3, 10.7, 13.1), 9.3, 1.0), ((5.5, 25.2, 14.9), 17.7, 1.5)])
def test_shell_cells_equal_brute_force(c, r, h):
    np.testing.assert_array_equal(W.sorted_unique(W.shell_cells(32, c, r, h), 32), _brute_shell(32, c, r, h))


def test_tiny_configs_sizes_and_order():
    for name, n in (("tiny", 4096), ("tiny_shell1", 1814)):
        wl = W.make(name)
        assert wl.N == n and wl.K == 27
        keys = W.pack_keys(wl.coords, wl.side)
        assert np.all(np.diff(keys) > 0)  # sorted, unique
        layer = wl.layers[0]
        assert (layer.Ci, layer.Co, layer.dtype) == (16, 16, "f32")
        assert layer.feats.min() >= -1.0 and layer.feats.max() < 1.0


def test_small_config():
    wl = W.make("small")
    assert 10_000 < wl.N < 200_000
    keys = W.pack_keys(wl.coords, wl.side)
    assert np.all(np.diff(keys) > 0)
    assert wl.coords.min() >= 0 and wl.coords.max() < 128
    layer = wl.layers[0]
    assert layer.feats.dtype == np.uint16 and layer.feats.shape == (wl.N, 64)
    f = W.bf16_bits_to_f32(layer.feats)
    assert abs(float(f.mean())) < 0.01 and abs(float(f.std()) - 1.0) < 0.01
    wv = W.bf16_bits_to_f32(layer.w)
    assert abs(float(wv.std()) * np.sqrt(27 * 64) - 1.0) < 0.05


def test_determinism_and_chunk_independence():
    a = W.normal(3, 5, 0, 1000)
    b = np.concatenate([W.normal(3, 5, 0, 400), W.normal(3, 5, 400, 600)])
    np.testing.assert_array_equal(a, b)
    x = W._chunked(W.normal, 9, 9, 100_000, "bf16", chunk=7_001)
    y = W._chunked(W.normal, 9, 9, 100_000, "bf16")
    np.testing.assert_array_equal(x, y)
    assert not np.array_equal(W.normal(3, 5, 0, 100), W.normal(4, 5, 0, 100))


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator.
    z = np.uint64(0) + np.arange(1, 4, dtype=np.uint64) * W._GAMMA
    out = W._mix64(z)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = (W.normal(1, 2, 0, 10_000) * 3.0).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]  # ties to even
    ours = W.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)


def test_offsets_order():
    offs = W.offsets_3x3x3()
    for k, (dz, dy, dx) in enumerate(offs):
        assert k == 9 * (dz + 1) + 3 * (dy + 1) + (dx + 1)
    np.testing.assert_array_equal(offs[13], [0, 0, 0])
