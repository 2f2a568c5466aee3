"""The materialising comparison path (bench.materialized_forward: the
(K, N, Ci) gather written out by torch index_select and contracted by cuBLAS
GEMMs, chunk by chunk) against the oracle.  This is the stock path the page
replaces (module docstring: the gather is materialised and contracted one or
two offsets at a time); the benchmark times it beside the fused call, so its
result is held to the same acceptance rule: |out - exact| <= 4e-3 * sum|terms|."""
import numpy as np
import pytest

import workloads as W
from helpers import assert_within, to_f64, torch_storage

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    return torch, bench


@pytest.mark.parametrize("chunk", [1, 2, 27])
def test_materialized_small_matches_oracle(env, oracle_mod, chunk):
    torch, bench = env
    wl = W.make("small")
    layer = wl.layers[0]
    nmap = oracle_mod.build_nmap(wl.coords, wl.offsets)
    ref, sabs = oracle_mod.conv(layer.feats, nmap, layer.w, layer.bias, "bf16",
                                threads=oracle_mod.host_threads())
    f, w, b = (torch_storage(a, "bf16") for a in (layer.feats, layer.w, layer.bias))
    got = bench.materialized_forward(torch, f, torch.from_numpy(nmap).cuda(), w, b, chunk)
    assert got.dtype == torch.bfloat16 and got.shape == (wl.N, layer.Co)
    assert_within(to_f64(got), ref, sabs, "bf16")


def test_materialized_invalid_entries_select_zero_rows(env, oracle_mod):
    """Entries outside [0, N) (the sentinel and garbage values) contribute
    nothing, as in the fused call."""
    torch, bench = env
    coords = W.random_occupancy(12, 0.3, 93)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    junk = np.where((np.arange(nmap.size).reshape(nmap.shape) % 3) == 0, -5, n + 9)
    nmap = np.where(nmap == n, junk, nmap).astype(np.int32)
    feats = W.values(93, 11, (n, 64), "bf16")
    w = W.values(93, 12, (27, 64, 32), "bf16", 1.0 / np.sqrt(27 * 64))
    b = W.values(93, 13, (32,), "bf16", 0.1)
    ref, sabs = oracle_mod.conv(feats, nmap, w, b, "bf16")
    got = bench.materialized_forward(torch, torch_storage(feats, "bf16"), torch.from_numpy(nmap).cuda(),
                                     torch_storage(w, "bf16"), torch_storage(b, "bf16"), 2)
    assert_within(to_f64(got), ref, sabs, "bf16")
