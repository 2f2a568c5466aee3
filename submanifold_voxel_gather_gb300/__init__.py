"""GB300-native fused submanifold sparse 3-D convolution.

Thin Python binding over the C ABI in ``include/spconv.h`` (``libspconv.so``,
built in-tree by ``python -m submanifold_voxel_gather_gb300.build``).  PyTorch
provides device memory and streams only; every step of the computation runs
in the library's CUDA kernels.  There is no fallback: if the library is
missing or the GPU is not an sm_103a part, calls raise.

The operation (page "sparse_conv_metal.py", trellis-2-mrp-mlx, mlx_backend)::

    out[n, co] = bias[co] + sum_k sum_ci feats[nmap[k, n], ci] * w[k, ci, co]

with ``nmap`` the (K, N) int32 neighbour map in which N marks a missing
neighbour; ``build_nmap`` builds it from voxel coordinates.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

__all__ = [
    "SpconvError", "load_library", "library_path", "version", "workspace_size", "build_nmap",
    "submconv3d", "submconv3d_dgrad", "submconv3d_wgrad", "tile_order", "count_valid_pairs",
    "xrun_layout", "submconv3d_xrun", "submconv3d_dgrad_xrun",
    "device_status",
    "default_offsets", "ACTIVATIONS",
    "F32", "TF32", "BF16",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libspconv.so")

# spconv_dtype
F32, TF32, BF16 = 0, 1, 2
_DTYPE_NAMES = {"f32": F32, "tf32": TF32, "bf16": BF16}

STATUS_NAMES = {
    0: "SPCONV_OK", -1: "SPCONV_ERR_INVALID_ARG", -2: "SPCONV_ERR_UNSUPPORTED",
    -3: "SPCONV_ERR_WORKSPACE", -4: "SPCONV_ERR_DUPLICATE_COORD", -5: "SPCONV_ERR_CUDA",
    -6: "SPCONV_ERR_DEVICE",
}


class SpconvError(RuntimeError):
    """A library call returned a non-zero spconv_status."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libspconv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built; run `python -m submanifold_voxel_gather_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.spconv_version.argtypes = []
        lib.spconv_version.restype = ctypes.c_int
        lib.spconv_last_error.argtypes = []
        lib.spconv_last_error.restype = ctypes.c_char_p
        lib.spconv_build_nmap_workspace_size.argtypes = [i64]
        lib.spconv_build_nmap_workspace_size.restype = ctypes.c_size_t
        lib.spconv_build_nmap.argtypes = [vp, i64, vp, i32, vp, vp, ctypes.c_size_t, vp]
        lib.spconv_build_nmap.restype = ctypes.c_int
        lib.spconv_build_nmap_async.argtypes = [vp, i64, vp, i32, vp, vp, ctypes.c_size_t, vp, vp]
        lib.spconv_build_nmap_async.restype = ctypes.c_int
        lib.spconv_submconv3d.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int, vp]
        lib.spconv_submconv3d.restype = ctypes.c_int
        lib.spconv_submconv3d_ex.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int,
                                             ctypes.c_int, vp]
        lib.spconv_submconv3d_ex.restype = ctypes.c_int
        lib.spconv_submconv3d_dgrad.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int, vp]
        lib.spconv_submconv3d_dgrad.restype = ctypes.c_int
        lib.spconv_submconv3d_wgrad.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int, vp]
        lib.spconv_submconv3d_wgrad.restype = ctypes.c_int
        lib.spconv_submconv3d_ordered.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int,
                                                  vp]
        lib.spconv_submconv3d_ordered.restype = ctypes.c_int
        lib.spconv_tile_order.argtypes = [vp, i64, i32, vp, vp]
        lib.spconv_tile_order.restype = ctypes.c_int
        lib.spconv_xrun_workspace_size.argtypes = [i64]
        lib.spconv_xrun_workspace_size.restype = ctypes.c_size_t
        lib.spconv_xrun_slot_capacity.argtypes = [i64]
        lib.spconv_xrun_slot_capacity.restype = i64
        lib.spconv_xrun_layout.argtypes = [vp, vp, i64, i32, vp, i64, vp, vp, ctypes.c_size_t, vp]
        lib.spconv_xrun_layout.restype = ctypes.c_int
        lib.spconv_build_nmap_xrun_workspace_size.argtypes = [i64]
        lib.spconv_build_nmap_xrun_workspace_size.restype = ctypes.c_size_t
        lib.spconv_build_nmap_xrun.argtypes = [vp, i64, vp, vp, i64, vp, vp, ctypes.c_size_t, vp, vp]
        lib.spconv_build_nmap_xrun.restype = ctypes.c_int
        lib.spconv_submconv3d_xrun.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, i64, i32, i32, i32,
                                               ctypes.c_int, vp]
        lib.spconv_submconv3d_xrun.restype = ctypes.c_int
        lib.spconv_submconv3d_xrun_ex.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                                  ctypes.c_int, ctypes.c_int, vp]
        lib.spconv_submconv3d_xrun_ex.restype = ctypes.c_int
        lib.spconv_submconv3d_dgrad_xrun.argtypes = [vp, vp, vp, i64, vp, vp, vp, i64, i32, i32, i32,
                                                     ctypes.c_int, vp]
        lib.spconv_submconv3d_dgrad_xrun.restype = ctypes.c_int
        lib.spconv_count_valid_pairs.argtypes = [vp, i64, i32, vp, vp]
        lib.spconv_count_valid_pairs.restype = ctypes.c_int
        lib.spconv_device_status.argtypes = [vp]
        lib.spconv_device_status.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(code: int) -> None:
    if code != 0:
        msg = load_library().spconv_last_error().decode(errors="replace")
        raise SpconvError(code, msg)


def version() -> int:
    return load_library().spconv_version()


def workspace_size(n: int) -> int:
    """Device bytes spconv_build_nmap needs for ``n`` voxels."""
    return int(load_library().spconv_build_nmap_workspace_size(int(n)))


def default_offsets() -> np.ndarray:
    """The 27 offsets of {-1,0,1}^3 in lexicographic (dz, dy, dx) order
    (k = 9(dz+1) + 3(dy+1) + (dx+1); k = 13 is the centre)."""
    r = np.arange(-1, 2, dtype=np.int32)
    dz, dy, dx = np.meshgrid(r, r, r, indexing="ij")
    return np.ascontiguousarray(np.stack([dz.ravel(), dy.ravel(), dx.ravel()], 1), dtype=np.int32)


def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _require_cuda(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")


def build_nmap(coords, offsets=None, workspace=None, stream=None, out=None, status=None):
    """Neighbour map (K, N) int32 of ``coords`` ((N, 3) int32 CUDA tensor,
    (z, y, x), distinct, components in [0, 2^20)).  ``offsets`` is a host
    (K, 3) integer array (default: ``default_offsets()``).  ``workspace`` is an
    optional uint8 CUDA tensor of at least ``workspace_size(N)`` bytes; if
    omitted one is taken from torch's allocator.  ``out`` is an optional
    (K, N) int32 CUDA tensor to write.  Waits for the stream once (to read
    the duplicate/range flags), unless ``status`` (a one-element int32 CUDA
    tensor) is given: then the verdict (0 = OK, else a negative status code)
    is written there on the stream and the call does not wait
    (spconv_build_nmap_async)."""
    torch = _torch()
    _require_cuda(coords, "coords", torch.int32)
    if coords.dim() != 2 or coords.shape[1] != 3:
        raise ValueError("coords must have shape (N, 3)")
    offs = default_offsets() if offsets is None else np.ascontiguousarray(
        np.asarray(offsets.cpu() if hasattr(offsets, "cpu") else offsets), dtype=np.int32).reshape(-1, 3)
    n, k = coords.shape[0], offs.shape[0]
    if out is None:
        nmap = torch.empty((k, n), dtype=torch.int32, device=coords.device)
    else:
        _require_cuda(out, "out", torch.int32)
        if tuple(out.shape) != (k, n):
            raise ValueError("out must have shape (K, N)")
        nmap = out
    need = workspace_size(n)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=coords.device)
    _require_cuda(workspace, "workspace", torch.uint8)
    lib = load_library()
    if status is None:
        _check(lib.spconv_build_nmap(_ptr(coords), n, offs.ctypes.data_as(ctypes.c_void_p), k,
                                     _ptr(nmap), _ptr(workspace), workspace.numel(),
                                     _stream_handle(stream)))
    else:
        _require_cuda(status, "status", torch.int32)
        if status.numel() != 1:
            raise ValueError("status must have one element")
        _check(lib.spconv_build_nmap_async(_ptr(coords), n, offs.ctypes.data_as(ctypes.c_void_p), k,
                                           _ptr(nmap), _ptr(workspace), workspace.numel(), _ptr(status),
                                           _stream_handle(stream)))
    return nmap


def _dtype_code(t, dtype):
    torch = _torch()
    if dtype is None:
        if t.dtype == torch.float32:
            return F32
        if t.dtype == torch.bfloat16:
            return BF16
        raise TypeError(f"unsupported feature dtype {t.dtype}")
    code = _DTYPE_NAMES[dtype] if isinstance(dtype, str) else int(dtype)
    want = torch.bfloat16 if code == BF16 else torch.float32
    if t.dtype != want:
        raise TypeError(f"dtype {dtype} needs {want} storage, got {t.dtype}")
    return code


ACTIVATIONS = {None: 0, "none": 0, "relu": 1, "silu": 2}


def submconv3d(feats, nmap, w, bias=None, out=None, dtype=None, stream=None, residual=None,
               activation=None, order=None):
    """Fused submanifold convolution.  feats (N, Ci), w (K, Ci, Co), bias (Co,)
    or None, all in one storage dtype (float32 or bfloat16); nmap (K, N) int32.
    ``dtype``: None (float32 -> exact "f32", bfloat16 -> "bf16") or "tf32"
    for float32 storage with tf32 tensor-core products.  Returns out (N, Co).

    ``residual`` (N, Co) and ``activation`` ("relu" or "silu") select the
    fused epilogue out = act(conv + bias + residual) (spconv_submconv3d_ex);
    ``out`` may be the residual tensor itself.

    ``order`` (N,) int32, a permutation from ``tile_order``, forms the tiles
    along it (spconv_submconv3d_ordered): the same result, fewer empty rows
    gathered for scattered inputs.  Not combined with the fused epilogue."""
    torch = _torch()
    code = _dtype_code(feats, dtype)
    _require_cuda(feats, "feats", feats.dtype)
    _require_cuda(nmap, "nmap", torch.int32)
    _require_cuda(w, "w", feats.dtype)
    if bias is not None:
        _require_cuda(bias, "bias", feats.dtype)
    if feats.dim() != 2 or w.dim() != 3 or nmap.dim() != 2:
        raise ValueError("expected feats (N, Ci), nmap (K, N), w (K, Ci, Co)")
    n, ci = feats.shape
    k, co = w.shape[0], w.shape[2]
    if tuple(nmap.shape) != (k, n) or w.shape[1] != ci:
        raise ValueError("inconsistent shapes")
    if bias is not None and tuple(bias.shape) != (co,):
        raise ValueError("bias must have shape (Co,)")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(a for a in ACTIVATIONS if a)}")
    if residual is not None:
        _require_cuda(residual, "residual", feats.dtype)
        if tuple(residual.shape) != (n, co):
            raise ValueError("residual must have shape (N, Co)")
    if out is None:
        out = torch.empty((n, co), dtype=feats.dtype, device=feats.device)
    else:
        _require_cuda(out, "out", feats.dtype)
        if tuple(out.shape) != (n, co):
            raise ValueError("out must have shape (N, Co)")
    lib = load_library()
    act = ACTIVATIONS[activation]
    if order is not None:
        _require_cuda(order, "order", torch.int32)
        if tuple(order.shape) != (n,):
            raise ValueError("order must have shape (N,)")
        if residual is not None or act != 0:
            raise ValueError("order is not combined with the fused epilogue")
        _check(lib.spconv_submconv3d_ordered(_ptr(feats), _ptr(nmap), _ptr(order), _ptr(w), _ptr(bias),
                                             _ptr(out), n, k, ci, co, code, _stream_handle(stream)))
    elif residual is None and act == 0:
        _check(lib.spconv_submconv3d(_ptr(feats), _ptr(nmap), _ptr(w), _ptr(bias), _ptr(out), n, k,
                                     ci, co, code, _stream_handle(stream)))
    else:
        _check(lib.spconv_submconv3d_ex(_ptr(feats), _ptr(nmap), _ptr(w), _ptr(bias), _ptr(residual),
                                        _ptr(out), n, k, ci, co, code, act, _stream_handle(stream)))
    return out


def submconv3d_dgrad(dout, nmap, w, out=None, dtype=None, stream=None):
    """Input gradient of submconv3d: dfeats (N, Ci) from dout (N, Co), the
    forward weights w (K, Ci, Co) and a map built from a point-symmetric,
    mirrored offset list (such as the default 3x3x3 list)."""
    torch = _torch()
    code = _dtype_code(dout, dtype)
    _require_cuda(dout, "dout", dout.dtype)
    _require_cuda(nmap, "nmap", torch.int32)
    _require_cuda(w, "w", dout.dtype)
    if dout.dim() != 2 or w.dim() != 3 or nmap.dim() != 2:
        raise ValueError("expected dout (N, Co), nmap (K, N), w (K, Ci, Co)")
    n, co = dout.shape
    k, ci = w.shape[0], w.shape[1]
    if tuple(nmap.shape) != (k, n) or w.shape[2] != co:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((n, ci), dtype=dout.dtype, device=dout.device)
    else:
        _require_cuda(out, "out", dout.dtype)
        if tuple(out.shape) != (n, ci):
            raise ValueError("out must have shape (N, Ci)")
    _check(load_library().spconv_submconv3d_dgrad(_ptr(dout), _ptr(nmap), _ptr(w), _ptr(out), n, k, ci,
                                                   co, code, _stream_handle(stream)))
    return out


def submconv3d_wgrad(feats, dout, nmap, k=None, with_bias=True, stream=None):
    """Weight (and bias) gradients of submconv3d: returns dw (K, Ci, Co) and,
    if ``with_bias``, dbias (Co,), both float32, from the forward input feats
    (N, Ci), dout (N, Co) and the map (K, N)."""
    torch = _torch()
    code = _dtype_code(feats, None)
    _require_cuda(feats, "feats", feats.dtype)
    _require_cuda(dout, "dout", feats.dtype)
    _require_cuda(nmap, "nmap", torch.int32)
    n, ci = feats.shape
    kk, n2 = nmap.shape
    if dout.dim() != 2 or dout.shape[0] != n or n2 != n:
        raise ValueError("expected feats (N, Ci), dout (N, Co), nmap (K, N)")
    co = dout.shape[1]
    dw = torch.empty((kk, ci, co), dtype=torch.float32, device=feats.device)
    db = torch.empty((co,), dtype=torch.float32, device=feats.device) if with_bias else None
    _check(load_library().spconv_submconv3d_wgrad(_ptr(feats), _ptr(dout), _ptr(nmap), _ptr(dw), _ptr(db),
                                                   n, kk, ci, co, code, _stream_handle(stream)))
    return (dw, db) if with_bias else dw


def tile_order(nmap, out=None, stream=None):
    """A tile order for ``submconv3d(..., order=...)``: (N,) int32, a
    permutation of the voxels; within chunks of 4096 consecutive voxels they
    are sorted by neighbour mask (spconv_tile_order)."""
    torch = _torch()
    _require_cuda(nmap, "nmap", torch.int32)
    k, n = nmap.shape
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=nmap.device)
    else:
        _require_cuda(out, "out", torch.int32)
        if tuple(out.shape) != (n,):
            raise ValueError("out must have shape (N,)")
    _check(load_library().spconv_tile_order(_ptr(nmap), n, k, _ptr(out), _stream_handle(stream)))
    return out


def xrun_layout(coords, nmap, slots=None, slot_count=None, workspace=None, stream=None):
    """x-run slot layout for ``submconv3d_xrun`` (spconv_xrun_layout): returns
    (slots, slot_count), an int32 CUDA tensor of spconv_xrun_slot_capacity(N)
    entries whose first S hold the slot codes, and a (1,) int64 CUDA tensor
    holding S.  ``nmap`` must come from the default 3x3x3 offsets."""
    torch = _torch()
    _require_cuda(coords, "coords", torch.int32)
    _require_cuda(nmap, "nmap", torch.int32)
    k, n = nmap.shape
    if tuple(coords.shape) != (n, 3):
        raise ValueError("coords must have shape (N, 3) matching nmap (K, N)")
    lib = load_library()
    cap = int(lib.spconv_xrun_slot_capacity(n))
    if slots is None:
        slots = torch.empty(cap, dtype=torch.int32, device=nmap.device)
    else:
        _require_cuda(slots, "slots", torch.int32)
    if slot_count is None:
        slot_count = torch.empty(1, dtype=torch.int64, device=nmap.device)
    else:
        _require_cuda(slot_count, "slot_count", torch.int64)
    wbytes = int(lib.spconv_xrun_workspace_size(n))
    if workspace is None:
        workspace = torch.empty(wbytes, dtype=torch.uint8, device=nmap.device)
    else:
        _require_cuda(workspace, "workspace", torch.uint8)
    _check(lib.spconv_xrun_layout(_ptr(coords), _ptr(nmap), n, k, _ptr(slots), slots.numel(), _ptr(slot_count),
                                  _ptr(workspace), workspace.numel(), _stream_handle(stream)))
    return slots, slot_count


def build_nmap_xrun(coords, out=None, slots=None, slot_count=None, workspace=None, status=None, stream=None):
    """The map (default 3x3x3 offsets) and the x-run slot layout in one call
    (spconv_build_nmap_xrun): returns (nmap, slots, slot_count) as
    ``build_nmap`` and ``xrun_layout`` would.  ``status``: an int32 CUDA
    tensor of one element that receives the verdict without a host wait;
    None waits and raises on a bad input."""
    torch = _torch()
    _require_cuda(coords, "coords", torch.int32)
    if coords.dim() != 2 or coords.shape[1] != 3:
        raise ValueError("coords must have shape (N, 3)")
    n = coords.shape[0]
    lib = load_library()
    dev = coords.device
    if out is None:
        out = torch.empty((27, n), dtype=torch.int32, device=dev)
    else:
        _require_cuda(out, "out", torch.int32)
        if tuple(out.shape) != (27, n):
            raise ValueError("out must have shape (27, N)")
    cap = int(lib.spconv_xrun_slot_capacity(n))
    if slots is None:
        slots = torch.empty(cap, dtype=torch.int32, device=dev)
    else:
        _require_cuda(slots, "slots", torch.int32)
    if slot_count is None:
        slot_count = torch.empty(1, dtype=torch.int64, device=dev)
    else:
        _require_cuda(slot_count, "slot_count", torch.int64)
    wbytes = int(lib.spconv_build_nmap_xrun_workspace_size(n))
    if workspace is None:
        workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    else:
        _require_cuda(workspace, "workspace", torch.uint8)
    if status is not None:
        _require_cuda(status, "status", torch.int32)
    _check(lib.spconv_build_nmap_xrun(_ptr(coords), n, _ptr(out), _ptr(slots), slots.numel(), _ptr(slot_count),
                                      _ptr(workspace), workspace.numel(),
                                      None if status is None else _ptr(status), _stream_handle(stream)))
    return out, slots, slot_count


def submconv3d_xrun(feats, nmap, slots, slot_count, w, bias=None, out=None, stream=None, residual=None,
                    activation=None):
    """``submconv3d`` over an x-run slot layout from ``xrun_layout``
    (spconv_submconv3d_xrun): bf16, K = 27, Ci = 128, Co <= 128.  Returns out
    (N, Co).

    ``residual`` (N, Co) and ``activation`` ("relu" or "silu") select the
    fused epilogue out = act(conv + bias + residual)
    (spconv_submconv3d_xrun_ex); ``out`` may be the residual tensor itself."""
    torch = _torch()
    _require_cuda(feats, "feats", torch.bfloat16)
    _require_cuda(nmap, "nmap", torch.int32)
    _require_cuda(slots, "slots", torch.int32)
    _require_cuda(slot_count, "slot_count", torch.int64)
    _require_cuda(w, "w", torch.bfloat16)
    if feats.dim() != 2 or w.dim() != 3 or nmap.dim() != 2:
        raise ValueError("expected feats (N, Ci), nmap (K, N), w (K, Ci, Co)")
    n, ci = feats.shape
    k, co = w.shape[0], w.shape[2]
    if tuple(nmap.shape) != (k, n) or w.shape[1] != ci:
        raise ValueError("shapes of feats, nmap and w do not agree")
    if bias is not None:
        _require_cuda(bias, "bias", torch.bfloat16)
    if out is None:
        out = torch.empty((n, co), dtype=feats.dtype, device=feats.device)
    else:
        _require_cuda(out, "out", feats.dtype)
        if tuple(out.shape) != (n, co):
            raise ValueError("out must have shape (N, Co)")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(a for a in ACTIVATIONS if a)}")
    if residual is not None:
        _require_cuda(residual, "residual", torch.bfloat16)
        if tuple(residual.shape) != (n, co):
            raise ValueError("residual must have shape (N, Co)")
    act = ACTIVATIONS[activation]
    lib = load_library()
    if residual is None and act == 0:
        _check(lib.spconv_submconv3d_xrun(_ptr(feats), _ptr(nmap), _ptr(slots), slots.numel(), _ptr(slot_count),
                                          _ptr(w), _ptr(bias), _ptr(out), n, k, ci, co, BF16,
                                          _stream_handle(stream)))
    else:
        _check(lib.spconv_submconv3d_xrun_ex(_ptr(feats), _ptr(nmap), _ptr(slots), slots.numel(),
                                             _ptr(slot_count), _ptr(w), _ptr(bias), _ptr(residual), _ptr(out), n,
                                             k, ci, co, BF16, act, _stream_handle(stream)))
    return out


def submconv3d_dgrad_xrun(dout, nmap, slots, slot_count, w, out=None, stream=None):
    """``submconv3d_dgrad`` over an x-run slot layout from ``xrun_layout``
    (spconv_submconv3d_dgrad_xrun): bf16, K = 27, Co = 128, Ci <= 128.
    Returns dfeats (N, Ci)."""
    torch = _torch()
    _require_cuda(dout, "dout", torch.bfloat16)
    _require_cuda(nmap, "nmap", torch.int32)
    _require_cuda(slots, "slots", torch.int32)
    _require_cuda(slot_count, "slot_count", torch.int64)
    _require_cuda(w, "w", torch.bfloat16)
    if dout.dim() != 2 or w.dim() != 3 or nmap.dim() != 2:
        raise ValueError("expected dout (N, Co), nmap (K, N), w (K, Ci, Co)")
    n, co = dout.shape
    k, ci = w.shape[0], w.shape[1]
    if tuple(nmap.shape) != (k, n) or w.shape[2] != co:
        raise ValueError("shapes of dout, nmap and w do not agree")
    if out is None:
        out = torch.empty((n, ci), dtype=dout.dtype, device=dout.device)
    else:
        _require_cuda(out, "out", dout.dtype)
        if tuple(out.shape) != (n, ci):
            raise ValueError("out must have shape (N, Ci)")
    _check(load_library().spconv_submconv3d_dgrad_xrun(_ptr(dout), _ptr(nmap), _ptr(slots), slots.numel(),
                                                       _ptr(slot_count), _ptr(w), _ptr(out), n, k, ci, co, BF16,
                                                       _stream_handle(stream)))
    return out


def count_valid_pairs(nmap, stream=None) -> int:
    """Number of entries v of nmap with 0 <= v < N (waits for the stream)."""
    torch = _torch()
    _require_cuda(nmap, "nmap", torch.int32)
    k, n = nmap.shape
    count = torch.empty(1, dtype=torch.int64, device=nmap.device)
    _check(load_library().spconv_count_valid_pairs(_ptr(nmap), n, k, _ptr(count),
                                                   _stream_handle(stream)))
    if stream is not None:
        stream.synchronize()
    return int(count.item())


def device_status(stream=None) -> None:
    """Raise SpconvError if a kernel has reported an internal error."""
    _check(load_library().spconv_device_status(_stream_handle(stream)))
