"""Shared test helpers: moving generator outputs to torch and checking GPU
results against the oracle's acceptance rule."""
import numpy as np

import workloads as W


def torch_storage(arr, dtype, device="cuda"):
    """Stored values (float32, or uint16 bf16 bits) -> torch tensor on device."""
    import torch
    a = np.ascontiguousarray(arr)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a.astype(np.float32, copy=False)).to(device)


def to_f64(t):
    """GPU output tensor -> float64 numpy (exact widening)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def assert_within(gpu64, ref64, sabs, dtype, tol=None):
    """|gpu - exact| <= tol * sum|terms| elementwise; returns the worst ratio."""
    from oracle import TOL
    tol = TOL[dtype] if tol is None else tol
    err = np.abs(gpu64 - ref64)
    bound = tol * sabs
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} outputs outside {tol}*sum|terms| "
            f"(first at {tuple(i)}: gpu={gpu64[tuple(i)]!r} exact={ref64[tuple(i)]!r} "
            f"sabs={sabs[tuple(i)]!r})")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sabs > 0, err / sabs, 0.0)
    return float(r.max()) if r.size else 0.0


def sample_rows(n, count, seed):
    """First and last 160 rows (covers the first and the ragged last tile)
    plus ``count`` seeded random rows, sorted and distinct."""
    head = np.arange(min(n, 160))
    tail = np.arange(max(0, n - 160), n)
    rnd = (W.draws_u64(seed, W.SID_TEST + 7, 0, count) % np.uint64(max(n, 1))).astype(np.int64)
    return np.unique(np.concatenate([head, tail, rnd])).astype(np.int64)


_ORACLE_MAPS = {}


def oracle_full_map(name):
    """(coords, the oracle's whole (K, N) map) of a named workload, computed
    once per test session (threaded: one sort, voxels split over the host's
    threads)."""
    import oracle
    if name not in _ORACLE_MAPS:
        coords = W.coords_only(name)
        _ORACLE_MAPS[name] = (coords, oracle.build_nmap(coords, W.offsets_3x3x3(),
                                                        threads=oracle.host_threads()))
    return _ORACLE_MAPS[name]
