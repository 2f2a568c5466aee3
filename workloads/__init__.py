"""Seeded synthetic voxel workloads: inputs only.

This module is shared by the CPU oracle's tests and by the GPU path's tests
and benchmark.  It draws coordinates, features, weights and biases and holds
none of the neighbour-map or convolution arithmetic.

Random numbers come from one counter-based generator written out here from
its published definition: SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014).  Draw ``i`` of the
stream ``(seed, sid)`` is ``mix64(key(seed, sid) + (i + 1) * GAMMA)``, so any
chunk of a stream can be drawn independently and in parallel with the same
result.  Normals use the Box-Muller transform (one normal from two uniforms).

Geometry follows the five workload recipes of the fused submanifold-conv
benchmark (sphere shells, a Gaussian-blob level band with isolated voxels, a
shell-plus-sprinkle mix and a decoder-scale shell set); every cell membership
test is a float64 comparison, so a workload is bit-identical on any IEEE-754
host given the same seed.

Coordinates are ``(z, y, x)`` int32, unique, sorted lexicographically.
Offsets are the 27 cells of ``{-1,0,1}^3`` in lexicographic ``(dz, dy, dx)``
order, so ``k = 9*(dz+1) + 3*(dy+1) + (dx+1)`` and the centre is ``k = 13``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_MASK64 = (1 << 64) - 1
_GAMMA_INT = 0x9E3779B97F4A7C15
_GAMMA = np.uint64(_GAMMA_INT)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30 = np.uint64(30)
_S27 = np.uint64(27)
_S31 = np.uint64(31)
_S11 = np.uint64(11)
_TWO_M53 = float(2.0 ** -53)

# Distinct stream ids, one per kind of draw.
SID_GEOMETRY = 1
SID_SPRINKLE = 2
SID_ISOLATED = 3
SID_FEATS = 100
SID_W = 200
SID_BIAS = 300
SID_TEST = 900


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> _S30)) * _M1
    z = (z ^ (z >> _S27)) * _M2
    return z ^ (z >> _S31)


def stream_key(seed: int, sid: int) -> int:
    """Starting state of stream ``sid`` under ``seed`` (two SplitMix64 steps)."""
    return _mix64_int(_mix64_int(seed * _GAMMA_INT + 0x632BE59BD9B4E019) + sid * _GAMMA_INT)


def draws_u64(seed: int, sid: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream ``(seed, sid)`` as uint64."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    return _mix64(np.uint64(stream_key(seed, sid)) + i * _GAMMA)


def uniform(seed: int, sid: int, start: int, count: int) -> np.ndarray:
    """float64 uniforms in [0, 1) from the top 53 bits of each draw."""
    return (draws_u64(seed, sid, start, count) >> _S11).astype(np.float64) * _TWO_M53


def normal(seed: int, sid: int, start: int, count: int) -> np.ndarray:
    """float64 standard normals; normal ``j`` uses draws ``2j`` and ``2j+1``."""
    d = draws_u64(seed, sid, 2 * start, 2 * count)
    u1 = ((d[0::2] >> _S11).astype(np.float64) + 1.0) * _TWO_M53  # (0, 1]
    u2 = (d[1::2] >> _S11).astype(np.float64) * _TWO_M53          # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos((2.0 * np.pi) * u2)


# --------------------------------------------------------------------------
# Storage types.  bf16 values are held as their uint16 bit patterns.
# --------------------------------------------------------------------------
DTYPES = ("f32", "tf32", "bf16")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, to nearest with ties to even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def storage_dtype(dtype: str):
    return np.uint16 if dtype == "bf16" else np.float32


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = np.asarray(x64, dtype=np.float32)
    return f32_to_bf16_bits(x32) if dtype == "bf16" else x32


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunked(fn, seed: int, sid: int, count: int, dtype: str, chunk: int = 1 << 22) -> np.ndarray:
    """Draw ``count`` values with ``fn`` in parallel chunks into storage dtype."""
    out = np.empty(count, dtype=storage_dtype(dtype))

    def work(s):
        end = min(s + chunk, count)
        for a in range(s, end, 1 << 15):  # cache-sized pieces
            b = min(a + (1 << 15), end)
            out[a:b] = to_storage(fn(seed, sid, a, b - a), dtype)

    starts = range(0, count, chunk)
    if count <= chunk:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    return out


# --------------------------------------------------------------------------
# Offsets and geometry.
# --------------------------------------------------------------------------
def offsets_cube(radius: int = 1) -> np.ndarray:
    """All offsets of ``{-r..r}^3`` in lexicographic (dz, dy, dx) order."""
    r = np.arange(-radius, radius + 1, dtype=np.int32)
    dz, dy, dx = np.meshgrid(r, r, r, indexing="ij")
    return np.stack([dz.ravel(), dy.ravel(), dx.ravel()], axis=1).astype(np.int32)


def offsets_3x3x3() -> np.ndarray:
    return offsets_cube(1)


def pack_keys(coords: np.ndarray, side: int) -> np.ndarray:
    c = coords.astype(np.int64)
    return (c[:, 0] * side + c[:, 1]) * side + c[:, 2]


def unpack_keys(keys: np.ndarray, side: int) -> np.ndarray:
    out = np.empty((keys.size, 3), dtype=np.int32)
    out[:, 2] = keys % side
    out[:, 1] = (keys // side) % side
    out[:, 0] = keys // (side * side)
    return out


def unique_sorted_keys(keys: np.ndarray) -> np.ndarray:
    """Sorted distinct values (sort + adjacent-difference, no hashing)."""
    k = np.sort(keys)
    if k.size == 0:
        return k
    keep = np.empty(k.size, dtype=bool)
    keep[0] = True
    np.not_equal(k[1:], k[:-1], out=keep[1:])
    return k[keep]


def sorted_unique(coords: np.ndarray, side: int) -> np.ndarray:
    return unpack_keys(unique_sorted_keys(pack_keys(coords, side)), side)


def shell_keys(side: int, centre, radius: float, half: float) -> np.ndarray:
    """Packed keys ``(z*side + y)*side + x`` of the integer cells p in
    [0, side)^3 with | |p - c| - radius | < half (unsorted, distinct)."""
    cz, cy, cx = (float(v) for v in centre)
    r_out = radius + half
    r_in = radius - half
    z0, z1 = max(0, int(np.floor(cz - r_out)) - 1), min(side - 1, int(np.ceil(cz + r_out)) + 1)
    y0, y1 = max(0, int(np.floor(cy - r_out)) - 1), min(side - 1, int(np.ceil(cy + r_out)) + 1)
    zz, yy = np.meshgrid(np.arange(z0, z1 + 1), np.arange(y0, y1 + 1), indexing="ij")
    zz = zz.ravel()
    yy = yy.ravel()
    q = (zz - cz) ** 2 + (yy - cy) ** 2
    ro2 = r_out * r_out - q
    keep = ro2 > 0
    zz, yy, q, ro2 = zz[keep], yy[keep], q[keep], ro2[keep]
    so = np.sqrt(ro2)
    si = np.sqrt(np.maximum(r_in * r_in - q, 0.0)) if r_in > 0 else np.zeros_like(so)
    # Candidate x intervals (widened by one cell; the exact test below decides).
    lo_a = np.floor(cx - so).astype(np.int64) - 1
    hi_a = np.ceil(cx - si).astype(np.int64) + 1
    lo_b = np.floor(cx + si).astype(np.int64) - 1
    hi_b = np.ceil(cx + so).astype(np.int64) + 1
    merged = lo_b <= hi_a
    hi_a = np.where(merged, hi_b, hi_a)
    starts = np.concatenate([lo_a, lo_b[~merged]])
    stops = np.concatenate([hi_a, hi_b[~merged]]) + 1
    zs = np.concatenate([zz, zz[~merged]])
    ys = np.concatenate([yy, yy[~merged]])
    lens = stops - starts
    total = int(lens.sum())
    rows = np.repeat(np.arange(len(lens)), lens)
    x = starts[rows] + (np.arange(total) - np.repeat(np.cumsum(lens) - lens, lens))
    z = zs[rows]
    y = ys[rows]
    inside = (x >= 0) & (x < side)
    x, y, z = x[inside], y[inside], z[inside]
    d = np.sqrt((z - cz) ** 2 + (y - cy) ** 2 + (x - cx) ** 2)
    hit = np.abs(d - radius) < half
    return (z[hit] * side + y[hit]) * side + x[hit]


def shell_cells(side: int, centre, radius: float, half: float) -> np.ndarray:
    """Integer cells p in [0, side)^3 with | |p - c| - radius | < half."""
    return unpack_keys(shell_keys(side, centre, radius, half), side)


def random_spheres(seed: int, count: int, side: int, r_lo: float, r_hi: float, margin: float,
                   half: float):
    """``count`` spheres: radius ~ U(r_lo, r_hi), centre uniform so that the
    shell plus ``margin`` cells stays inside the grid."""
    u = uniform(seed, SID_GEOMETRY, 0, 4 * count).reshape(count, 4)
    out = []
    for i in range(count):
        r = r_lo + (r_hi - r_lo) * u[i, 0]
        lo = r + half + margin
        hi = (side - 1) - lo
        c = tuple(lo + (hi - lo) * u[i, 1 + j] for j in range(3))
        out.append((c, r))
    return out


def shells_of_spheres(seed, count, side, r_lo, r_hi, half, margin=2.0) -> np.ndarray:
    parts = [shell_keys(side, c, r, half)
             for c, r in random_spheres(seed, count, side, r_lo, r_hi, margin, half)]
    return unpack_keys(unique_sorted_keys(np.concatenate(parts)), side)


def add_sprinkle(coords: np.ndarray, side: int, seed: int, n_add: int) -> np.ndarray:
    """Add ``n_add`` distinct uniformly random cells not already active."""
    occ = np.zeros(side ** 3, dtype=bool)
    occ[pack_keys(coords, side)] = True
    got = []
    start = 0
    need = n_add
    while need > 0:
        batch = max(2 * need, 1024)
        cand = (draws_u64(seed, SID_SPRINKLE, start, batch) % np.uint64(side ** 3)).astype(np.int64)
        start += batch
        order = np.argsort(cand, kind="stable")
        sc = cand[order]
        dup = np.zeros(sc.size, dtype=bool)
        dup[1:] = sc[1:] == sc[:-1]
        first = np.sort(order[~dup])
        cand = cand[first]
        cand = cand[~occ[cand]]
        cand = cand[:need]
        occ[cand] = True
        got.append(cand)
        need -= len(cand)
    keys = np.concatenate([pack_keys(coords, side)] + got)
    return unpack_keys(np.sort(keys), side)


def add_isolated(coords: np.ndarray, side: int, seed: int, n_add: int) -> np.ndarray:
    """Add ``n_add`` voxels whose 26 neighbours are all inactive, by rejection
    sampling cells of [1, side-2]^3 in draw order."""
    occ = np.zeros((side, side, side), dtype=bool)
    occ[coords[:, 0], coords[:, 1], coords[:, 2]] = True
    added = []
    start = 0
    inner = side - 2
    while len(added) < n_add:
        batch = 4096
        d = draws_u64(seed, SID_ISOLATED, start, 3 * batch).reshape(batch, 3)
        start += 3 * batch
        cells = (d % np.uint64(inner)).astype(np.int64) + 1
        for z, y, x in cells:
            if occ[z - 1:z + 2, y - 1:y + 2, x - 1:x + 2].any():
                continue
            occ[z, y, x] = True
            added.append((z, y, x))
            if len(added) == n_add:
                break
    keys = np.concatenate([pack_keys(coords, side),
                           pack_keys(np.asarray(added, dtype=np.int64).reshape(-1, 3), side)])
    return unpack_keys(np.sort(keys), side)


def blob_band(seed: int, side: int, n_blobs: int, eps: float) -> np.ndarray:
    """Cells with |f - 0.5| < eps, f = sum of n_blobs isotropic Gaussians with
    centres ~ U(48, 208)^3 (scaled to the grid) and sigma ~ U(12, 32)."""
    u = uniform(seed, SID_GEOMETRY, 0, 4 * n_blobs).reshape(n_blobs, 4)
    scale = side / 256.0
    cen = (48.0 + 160.0 * u[:, :3]) * scale
    sig = (12.0 + 20.0 * u[:, 3]) * scale
    g = np.arange(side, dtype=np.float64)
    found = []
    for z in range(side):
        dz2 = (z - cen[:, 0]) ** 2                                   # (B,)
        dy2 = (g[None, :] - cen[:, 1:2]) ** 2                         # (B, side)
        dx2 = (g[None, :] - cen[:, 2:3]) ** 2                         # (B, side)
        f = np.zeros((side, side), dtype=np.float64)
        for b in range(n_blobs):
            e = -(dz2[b] + dy2[b][:, None] + dx2[b][None, :]) / (2.0 * sig[b] * sig[b])
            f += np.exp(e)
        yy, xx = np.nonzero(np.abs(f - 0.5) < eps)
        found.append(np.stack([np.full_like(yy, z), yy, xx], axis=1))
    return np.concatenate(found).astype(np.int32)


# --------------------------------------------------------------------------
# Workloads.
# --------------------------------------------------------------------------
@dataclass
class Layer:
    """One convolution: stored feats (N,Ci), w (K,Ci,Co), bias (Co,).

    ``dtype`` is the storage/compute type: "f32" (fp32 storage, exact fp32
    arithmetic), "tf32" (fp32 storage, tf32 products) or "bf16" (bf16
    storage as uint16 bits, fp32 accumulation)."""
    Ci: int
    Co: int
    dtype: str
    feats: np.ndarray
    w: np.ndarray
    bias: np.ndarray


@dataclass
class Workload:
    name: str
    seed: int
    side: int
    coords: np.ndarray
    offsets: np.ndarray
    layers: list = field(default_factory=list)
    note: str = ""

    @property
    def N(self) -> int:
        return int(self.coords.shape[0])

    @property
    def K(self) -> int:
        return int(self.offsets.shape[0])


def make_layer(seed: int, li: int, N: int, K: int, Ci: int, Co: int, dtype: str,
               feat_dist: str = "normal", bias_std: float = 0.1) -> Layer:
    """Seeded values: feats N(0,1) or U(-1,1); w ~ N(0, std = 1/sqrt(K*Ci));
    bias ~ N(0, std = bias_std); all rounded to the storage type."""
    if feat_dist == "uniform":
        feats = _chunked(lambda s, sid, a, n: 2.0 * uniform(s, sid, a, n) - 1.0,
                         seed, SID_FEATS + li, N * Ci, dtype)
    else:
        feats = _chunked(normal, seed, SID_FEATS + li, N * Ci, dtype)
    std = 1.0 / np.sqrt(K * Ci)
    w = _chunked(lambda s, sid, a, n: std * normal(s, sid, a, n), seed, SID_W + li, K * Ci * Co, dtype)
    bias = _chunked(lambda s, sid, a, n: bias_std * normal(s, sid, a, n), seed, SID_BIAS + li, Co, dtype)
    return Layer(Ci, Co, dtype, feats.reshape(N, Ci), w.reshape(K, Ci, Co), bias)


# Frozen level-band half-width for the medium workload: chosen once so the
# band of the seed-2 blob field holds about 0.95 M cells.
MEDIUM_EPS = 0.208


def _tiny(literal_shell: bool) -> Workload:
    side, c = 32, (16.0, 16.0, 16.0)
    if literal_shell:
        coords = sorted_unique(shell_cells(side, c, 12.0, 0.5), side)
        name, note = "tiny_shell1", "all cells of the 1-thick r=12 shell in 32^3"
    else:
        coords = sorted_unique(shell_cells(side, c, 12.0, 1.5), side)[:4096]
        name, note = "tiny", "first 4096 (z,y,x) cells of the 3-thick r=12 shell in 32^3"
    wl = Workload(name, 0, side, coords, offsets_3x3x3(), note=note)
    wl.layers.append(make_layer(0, 0, wl.N, wl.K, 16, 16, "f32", feat_dist="uniform"))
    return wl


def _small() -> Workload:
    side = 128
    coords = shells_of_spheres(1, 3, side, 20.0, 50.0, 1.0)
    wl = Workload("small", 1, side, coords, offsets_3x3x3(),
                  note="2-thick shells of 3 spheres r~U(20,50) in 128^3")
    wl.layers.append(make_layer(1, 0, wl.N, wl.K, 64, 64, "bf16"))
    return wl


def _medium() -> Workload:
    side = 256
    band = blob_band(2, side, 8, MEDIUM_EPS)
    band = sorted_unique(band, side)
    n_iso = int(round(len(band) * 0.05 / 0.95))
    coords = add_isolated(band, side, 2, n_iso)
    wl = Workload("medium", 2, side, coords, offsets_3x3x3(),
                  note=f"|f-0.5|<{MEDIUM_EPS} band of 8 Gaussian blobs in 256^3 + {n_iso} isolated voxels")
    wl.layers.append(make_layer(2, 0, wl.N, wl.K, 128, 128, "bf16"))
    return wl


def _channel() -> Workload:
    side = 512
    shells = shells_of_spheres(3, 6, side, 60.0, 120.0, 1.0)
    n_s = int(round(len(shells) * 0.3 / 0.7))
    coords = add_sprinkle(shells, side, 3, n_s)
    wl = Workload("channel", 3, side, coords, offsets_3x3x3(),
                  note=f"2-thick shells of 6 spheres r~U(60,120) in 512^3 + {n_s} random cells (30%)")
    wl.layers.append(make_layer(3, 0, wl.N, wl.K, 256, 128, "bf16"))
    wl.layers.append(make_layer(3, 1, wl.N, wl.K, 64, 256, "bf16"))
    return wl


def _decoder() -> Workload:
    side = 1024
    coords = shells_of_spheres(4, 12, side, 100.0, 210.0, 1.5)
    wl = Workload("decoder", 4, side, coords, offsets_3x3x3(),
                  note="3-thick shells of 12 spheres r~U(100,210) in 1024^3")
    wl.layers.append(make_layer(4, 0, wl.N, wl.K, 128, 128, "bf16"))
    return wl


_BUILDERS = {
    "tiny": lambda: _tiny(False),
    "tiny_shell1": lambda: _tiny(True),
    "small": _small,
    "medium": _medium,
    "channel": _channel,
    "decoder": _decoder,
}

CONFIGS = tuple(_BUILDERS)


def make(name: str) -> Workload:
    """Build the named workload (deterministic)."""
    return _BUILDERS[name]()


def coords_only(name: str) -> np.ndarray:
    """Coordinates of a named workload without drawing any values."""
    wl = {
        "tiny": lambda: sorted_unique(shell_cells(32, (16.0,) * 3, 12.0, 1.5), 32)[:4096],
        "tiny_shell1": lambda: sorted_unique(shell_cells(32, (16.0,) * 3, 12.0, 0.5), 32),
    }
    if name in wl:
        return wl[name]()
    return make(name).coords


# --------------------------------------------------------------------------
# Small generic cases for tests.
# --------------------------------------------------------------------------
def random_occupancy(side: int, frac: float, seed: int) -> np.ndarray:
    """Cells of a side^3 grid kept with probability ``frac`` (sorted)."""
    u = uniform(seed, SID_TEST, 0, side ** 3)
    keys = np.nonzero(u < frac)[0].astype(np.int64)
    return unpack_keys(keys, side)


def permutation(n: int, seed: int, sid: int = SID_TEST + 1) -> np.ndarray:
    """A seeded permutation of range(n) (argsort of uniform draws)."""
    return np.argsort(draws_u64(seed, sid, 0, n), kind="stable").astype(np.int64)


def values(seed: int, sid: int, shape, dtype: str, scale: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return _chunked(lambda s, i, a, c: scale * normal(s, i, a, c), seed, sid, n, dtype).reshape(shape)
