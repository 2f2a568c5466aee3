"""CPU oracle for the fused submanifold sparse 3-D convolution.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product package never
imports this module, and this module imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation), compiled
with gcc on first use.  What it follows on the page "sparse_conv_metal.py"
(trellis-2-mrp-mlx, mlx_backend):

* ``build_nmap`` - the (K, N) int32 neighbour map the wrapper docstring
  describes, missing neighbours marked with N; neighbour of voxel n under
  offset k is the voxel at coords[n] + offsets[k].
* ``conv`` - the module-docstring formula, with the kernel body's rule that
  an entry that is not a valid row contributes nothing, plus the bias the
  wrapper adds.  Returns the exact (fp64) result and the per-output scale
  sum |terms| that the acceptance tolerance is measured against.
* ``dgrad`` / ``wgrad`` - gradients of ``conv`` with respect to the features
  and the weights (the chain rule applied to the formula; the page has no
  backward pass), plain sums in fp64.
* ``conv_fused`` - ``conv`` followed by the library's fused epilogue,
  act(conv + bias + residual) with act ReLU or SiLU.  The page defines no
  epilogue beyond the bias (the conv runs layer after layer inside decoders,
  module docstring); this is the plain definition of the extension, in fp64.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
things other than itself: a brute-force neighbour search, a library dense
3-D cross-correlation read back at the active sites, a dense GEMM for the
centre offset alone, exact bias for an empty map, linearity, permutation
equivariance, closed-form pair counts and a hand-worked example.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", f"liboracle-{platform.machine()}.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_DUPLICATE_COORD = -4
ERR_NOMEM = -6

DTYPE_CODE = {"f32": 0, "tf32": 0, "bf16": 1}

# Acceptance rule for feature outputs: |gpu - exact| <= TOL[dtype] * sabs.
TOL = {"f32": 1e-5, "tf32": 4e-3, "bf16": 4e-3}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with status {code}")
        self.code = code


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if force or not fresh:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            lib.oracle_build_nmap.argtypes = [vp, i64, vp, i32, vp]
            lib.oracle_build_nmap.restype = ctypes.c_int
            lib.oracle_nmap_rows.argtypes = [vp, i64, vp, i32, vp, i64, vp]
            lib.oracle_nmap_rows.restype = ctypes.c_int
            lib.oracle_conv.argtypes = [vp, i32, vp, vp, vp, i64, i32, i32, i32, vp, i64, vp, vp]
            lib.oracle_conv.restype = ctypes.c_int
            lib.oracle_dgrad.argtypes = [vp, i32, vp, vp, i64, i32, i32, i32, vp, i64, vp, vp]
            lib.oracle_dgrad.restype = ctypes.c_int
            lib.oracle_wgrad.argtypes = [vp, vp, i32, vp, i64, i32, i32, i32, vp, i64, vp, vp]
            lib.oracle_wgrad.restype = ctypes.c_int
            lib.oracle_count_valid_pairs.argtypes = [vp, i64, i32]
            lib.oracle_count_valid_pairs.restype = ctypes.c_int64
            lib.oracle_table_new.argtypes = [vp, i64, ctypes.POINTER(ctypes.c_int)]
            lib.oracle_table_new.restype = vp
            lib.oracle_table_query.argtypes = [vp, vp, i64, vp, i32, i64, i64, vp]
            lib.oracle_table_query.restype = ctypes.c_int
            lib.oracle_table_free.argtypes = [vp]
            lib.oracle_table_free.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def build_nmap(coords: np.ndarray, offsets: np.ndarray, threads: int = 1) -> np.ndarray:
    """(K, N) int32 neighbour map; entry N marks a missing neighbour.

    ``threads`` > 1 sorts the coordinates once and splits the voxels over
    that many threads; every entry is the same binary search either way."""
    lib = _load()
    coords = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, 3)
    offsets = np.ascontiguousarray(offsets, dtype=np.int32).reshape(-1, 3)
    N, K = coords.shape[0], offsets.shape[0]
    nmap = np.empty((K, N), dtype=np.int32)
    threads = max(1, min(int(threads), N))
    if threads == 1 or N == 0:
        rc = lib.oracle_build_nmap(_ptr(coords), N, _ptr(offsets), K, _ptr(nmap))
        if rc != OK:
            raise OracleError(rc, "build_nmap")
        return nmap
    if K < 1:
        raise OracleError(ERR_INVALID_ARG, "build_nmap")
    status = ctypes.c_int(0)
    table = lib.oracle_table_new(_ptr(coords), N, ctypes.byref(status))
    if not table:
        raise OracleError(status.value, "build_nmap")
    try:
        bounds = np.linspace(0, N, threads + 1).astype(np.int64)

        def run(i):
            rc = lib.oracle_table_query(table, _ptr(coords), N, _ptr(offsets), K,
                                        int(bounds[i]), int(bounds[i + 1]), _ptr(nmap))
            if rc != OK:
                raise OracleError(rc, "build_nmap")

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, range(threads)))
    finally:
        lib.oracle_table_free(table)
    return nmap


def nmap_rows(coords: np.ndarray, offsets: np.ndarray, rows) -> np.ndarray:
    """Columns ``rows`` of the neighbour map: (K, len(rows)) int32, entry
    [k, r] = nmap[k, rows[r]] (the full table is still sorted)."""
    lib = _load()
    coords = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, 3)
    offsets = np.ascontiguousarray(offsets, dtype=np.int32).reshape(-1, 3)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    N, K = coords.shape[0], offsets.shape[0]
    out = np.empty((K, rows.shape[0]), dtype=np.int32)
    rc = lib.oracle_nmap_rows(_ptr(coords), N, _ptr(offsets), K, _ptr(rows), rows.shape[0], _ptr(out))
    if rc != OK:
        raise OracleError(rc, "nmap_rows")
    return out


def conv(feats: np.ndarray, nmap: np.ndarray, w: np.ndarray, bias, dtype: str,
         rows=None, threads: int = 1):
    """Exact convolution (fp64) of stored values.

    feats (N, Ci), w (K, Ci, Co) and bias (Co,) hold the stored values: float32
    for "f32"/"tf32", uint16 bf16 bit patterns for "bf16".  ``rows`` selects
    output rows (default all).  Returns ``(out, sabs)``, both float64 of shape
    (len(rows), Co).  ``threads`` splits the rows over that many threads; the
    per-output arithmetic is the same loop nest either way.
    """
    lib = _load()
    code = DTYPE_CODE[dtype]
    sdt = np.uint16 if dtype == "bf16" else np.float32
    feats = np.ascontiguousarray(feats, dtype=sdt)
    w = np.ascontiguousarray(w, dtype=sdt)
    nmap = np.ascontiguousarray(nmap, dtype=np.int32)
    K, N = nmap.shape
    Ci = feats.shape[1]
    Co = w.shape[2]
    if feats.shape[0] != N or w.shape[:2] != (K, Ci):
        raise ValueError("oracle.conv: inconsistent shapes")
    bias_arr = None if bias is None else np.ascontiguousarray(bias, dtype=sdt)
    if rows is None:
        rows = np.arange(N, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.empty((R, Co), dtype=np.float64)
    sabs = np.empty((R, Co), dtype=np.float64)
    if R == 0:
        return out, sabs

    def run(a, b):
        rc = lib.oracle_conv(_ptr(feats), code, _ptr(nmap), _ptr(w),
                             None if bias_arr is None else _ptr(bias_arr),
                             N, K, Ci, Co, _ptr(rows[a:b]), b - a,
                             _ptr(out[a:b]), _ptr(sabs[a:b]))
        if rc != OK:
            raise OracleError(rc, "conv")

    threads = max(1, min(int(threads), R))
    if threads == 1:
        run(0, R)
    else:
        bounds = np.linspace(0, R, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return out, sabs


# Largest slope of each activation: the error of the pre-activation value is
# multiplied by at most this much.  SiLU's derivative peaks at ~1.0998
# (x ~ 2.40).
ACT_LIPSCHITZ = {"none": 1.0, "relu": 1.0, "silu": 1.1}


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values (float32, or uint16 bf16 bit patterns) as exact float64."""
    a = np.asarray(a)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float32).astype(np.float64)


def conv_fused(feats: np.ndarray, nmap: np.ndarray, w: np.ndarray, bias, dtype: str,
               residual=None, act: str = "none", rows=None, threads: int = 1):
    """act(conv + bias + residual), exact in fp64.

    ``residual`` (N, Co) holds stored values like ``feats`` (or None);
    ``act`` is "none", "relu" (max(x, 0)) or "silu" (x / (1 + exp(-x))).
    Returns ``(out, scale)``: scale = slope bound of ``act`` x (sum |terms| +
    |bias| + |residual|), the size the acceptance tolerance multiplies.
    """
    if act not in ACT_LIPSCHITZ:
        raise ValueError(f"unknown activation {act!r}")
    pre, sabs = conv(feats, nmap, w, bias, dtype, rows=rows, threads=threads)
    if residual is not None:
        res = widen(residual, dtype)
        if rows is not None:
            res = res[np.asarray(rows, dtype=np.int64)]
        pre = pre + res
        sabs = sabs + np.abs(res)
    if act == "relu":
        out = np.maximum(pre, 0.0)
    elif act == "silu":
        with np.errstate(over="ignore"):
            out = pre / (1.0 + np.exp(-pre))
    else:
        out = pre
    return out, ACT_LIPSCHITZ[act] * sabs


def dgrad(dout: np.ndarray, nmap: np.ndarray, w: np.ndarray, dtype: str, rows=None,
          threads: int = 1):
    """dfeats[m, ci] = sum over valid entries m = nmap[k, n] of
    sum_co dout[n, co] * w[k, ci, co], exact (fp64).  ``rows`` selects rows of
    dfeats (default all).  Returns ``(dfeats, sum |terms|)``."""
    lib = _load()
    code = DTYPE_CODE[dtype]
    sdt = np.uint16 if dtype == "bf16" else np.float32
    dout = np.ascontiguousarray(dout, dtype=sdt)
    w = np.ascontiguousarray(w, dtype=sdt)
    nmap = np.ascontiguousarray(nmap, dtype=np.int32)
    K, N = nmap.shape
    Ci, Co = w.shape[1], w.shape[2]
    if dout.shape != (N, Co) or w.shape[0] != K:
        raise ValueError("oracle.dgrad: inconsistent shapes")
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.empty((R, Ci), dtype=np.float64)
    dabs = np.empty((R, Ci), dtype=np.float64)
    if R == 0:
        return out, dabs

    def run(a, b):
        rc = lib.oracle_dgrad(_ptr(dout), code, _ptr(nmap), _ptr(w), N, K, Ci, Co, _ptr(rows[a:b]),
                              b - a, _ptr(out[a:b]), _ptr(dabs[a:b]))
        if rc != OK:
            raise OracleError(rc, "dgrad")

    threads = max(1, min(int(threads), R))
    if threads == 1:
        run(0, R)
    else:
        bounds = np.linspace(0, R, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return out, dabs


def wgrad(feats: np.ndarray, dout: np.ndarray, nmap: np.ndarray, dtype: str, entries=None):
    """dw[k, ci, co] = sum over valid entries of feats[nmap[k, n], ci] *
    dout[n, co], exact (fp64).  With ``entries`` (flat indices into (K, Ci,
    Co)) only those values are computed.  Returns ``(dw, sum |terms|)``, of
    shape (K, Ci, Co) or (len(entries),)."""
    lib = _load()
    code = DTYPE_CODE[dtype]
    sdt = np.uint16 if dtype == "bf16" else np.float32
    feats = np.ascontiguousarray(feats, dtype=sdt)
    dout = np.ascontiguousarray(dout, dtype=sdt)
    nmap = np.ascontiguousarray(nmap, dtype=np.int32)
    K, N = nmap.shape
    Ci, Co = feats.shape[1], dout.shape[1]
    if feats.shape[0] != N or dout.shape[0] != N:
        raise ValueError("oracle.wgrad: inconsistent shapes")
    if entries is None:
        out = np.empty((K, Ci, Co), dtype=np.float64)
        dabs = np.empty((K, Ci, Co), dtype=np.float64)
        rc = lib.oracle_wgrad(_ptr(feats), _ptr(dout), code, _ptr(nmap), N, K, Ci, Co, None, 0,
                              _ptr(out), _ptr(dabs))
    else:
        entries = np.ascontiguousarray(entries, dtype=np.int64)
        out = np.empty(entries.shape[0], dtype=np.float64)
        dabs = np.empty(entries.shape[0], dtype=np.float64)
        rc = lib.oracle_wgrad(_ptr(feats), _ptr(dout), code, _ptr(nmap), N, K, Ci, Co, _ptr(entries),
                              entries.shape[0], _ptr(out), _ptr(dabs))
    if rc != OK:
        raise OracleError(rc, "wgrad")
    return out, dabs


def count_valid_pairs(nmap: np.ndarray) -> int:
    """Number of map entries v with 0 <= v < N."""
    lib = _load()
    nmap = np.ascontiguousarray(nmap, dtype=np.int32)
    K, N = nmap.shape
    return int(lib.oracle_count_valid_pairs(_ptr(nmap), N, K))


def host_threads() -> int:
    """Host threads available to the oracle."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1
