"""Fused epilogue (spconv_submconv3d_ex): out = act(conv + bias + residual),
on the GPU against the oracle's exact fp64 result.  Acceptance as for the
plain convolution, |gpu - exact| <= tol * scale, where scale = (slope bound
of the activation) x (sum |terms| + |bias| + |residual|) and tol = 1e-5
(f32) or 4e-3 (bf16)."""
import numpy as np
import pytest

import workloads as W
from helpers import assert_within, to_f64, torch_storage

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


def case(oracle_mod, side, frac, seed, ci, co, dtype):
    coords = W.random_occupancy(side, frac, seed)
    n = len(coords)
    nmap = oracle_mod.build_nmap(coords, W.offsets_3x3x3())
    feats = W.values(seed, 11, (n, ci), dtype)
    w = W.values(seed, 12, (27, ci, co), dtype, 1.0 / np.sqrt(27 * ci))
    b = W.values(seed, 13, (co,), dtype, 0.1)
    res = W.values(seed, 14, (n, co), dtype)
    return nmap, feats, w, b, res


def run_ex(sv, nmap, feats, w, b, res, dtype, act, in_place=False):
    import torch
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    f, ww, bb = torch_storage(feats, dtype), torch_storage(w, dtype), torch_storage(b, dtype)
    r = None if res is None else torch_storage(res, dtype)
    out = r if in_place else None
    got = sv.submconv3d(f, nm, ww, bb, out=out, residual=r, activation=act,
                        dtype=("tf32" if dtype == "tf32" else None))
    sv.device_status()
    if in_place:
        assert got.data_ptr() == r.data_ptr()
    return to_f64(got)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "tf32"])
@pytest.mark.parametrize("act", ["relu", "silu", None])
@pytest.mark.parametrize("with_res", [True, False])
def test_epilogue_matches_oracle(sv, oracle_mod, dtype, act, with_res):
    """Several 256-voxel tiles and a ragged last one (N = 1,420)."""
    nmap, feats, w, b, res = case(oracle_mod, 16, 0.35, 61, 64, 64, dtype)
    res = res if with_res else None
    ref, scale = oracle_mod.conv_fused(feats, nmap, w, b, dtype, residual=res, act=act or "none")
    got = run_ex(sv, nmap, feats, w, b, res, dtype, act)
    assert_within(got, ref, scale, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
@pytest.mark.parametrize("ci,co", [(128, 128), (64, 256), (32, 272)])
def test_epilogue_channel_shapes(sv, oracle_mod, ci, co, dtype):
    """One and two M blocks, and Co > 256 (two launches, the second with a
    16-channel remainder): each launch adds its own channel range of the
    residual."""
    nmap, feats, w, b, res = case(oracle_mod, 14, 0.3, ci + co, ci, co, dtype)
    ref, scale = oracle_mod.conv_fused(feats, nmap, w, b, dtype, residual=res, act="silu",
                                       threads=oracle_mod.host_threads())
    assert_within(run_ex(sv, nmap, feats, w, b, res, dtype, "silu"), ref, scale, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "tf32"])
def test_epilogue_in_place_residual(sv, oracle_mod, dtype):
    """out is the residual buffer itself (x <- act(conv(x') + b + x))."""
    nmap, feats, w, b, res = case(oracle_mod, 15, 0.3, 71, 64, 128, dtype)
    ref, scale = oracle_mod.conv_fused(feats, nmap, w, b, dtype, residual=res, act="relu")
    assert_within(run_ex(sv, nmap, feats, w, b, res, dtype, "relu", in_place=True), ref, scale, dtype)


def test_epilogue_none_equals_plain_call_bitwise(sv, oracle_mod):
    import torch
    nmap, feats, w, b, _ = case(oracle_mod, 14, 0.3, 81, 64, 64, "bf16")
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    f, ww, bb = torch_storage(feats, "bf16"), torch_storage(w, "bf16"), torch_storage(b, "bf16")
    plain = sv.submconv3d(f, nm, ww, bb)
    zero = torch.zeros_like(plain)
    fused = sv.submconv3d(f, nm, ww, bb, residual=zero, activation="none")
    assert torch.equal(plain, fused)


def test_chained_layers_on_one_map(sv, oracle_mod):
    """Two layers back to back on one neighbour map, the second consuming the
    first's bf16 output (a decoder block: x1 = silu(conv1(x) + b1);
    y = relu(conv2(x1) + b2 + x)).  Each layer is checked against the oracle
    on the exact input it received."""
    import torch
    nmap, feats, w1, b1, _ = case(oracle_mod, 16, 0.3, 91, 64, 64, "bf16")
    w2 = W.values(92, 12, (27, 64, 64), "bf16", 1.0 / np.sqrt(27 * 64))
    b2 = W.values(92, 13, (64,), "bf16", 0.1)
    nm = torch.from_numpy(np.ascontiguousarray(nmap, dtype=np.int32)).cuda()
    x = torch_storage(feats, "bf16")
    x1 = sv.submconv3d(x, nm, torch_storage(w1, "bf16"), torch_storage(b1, "bf16"), activation="silu")
    y = sv.submconv3d(x1, nm, torch_storage(w2, "bf16"), torch_storage(b2, "bf16"), residual=x,
                      activation="relu")
    sv.device_status()
    x1_bits = x1.cpu().view(torch.int16).numpy().view(np.uint16)
    ref1, s1 = oracle_mod.conv_fused(feats, nmap, w1, b1, "bf16", act="silu")
    assert_within(to_f64(x1), ref1, s1, "bf16")
    ref2, s2 = oracle_mod.conv_fused(x1_bits, nmap, w2, b2, "bf16", residual=feats, act="relu")
    assert_within(to_f64(y), ref2, s2, "bf16")


def test_epilogue_rejects_unknown_activation(sv):
    import torch
    f = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    nm = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    w = torch.zeros((1, 16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        sv.submconv3d(f, nm, w, activation="gelu")
