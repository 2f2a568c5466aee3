#!/usr/bin/env python
"""Benchmark of the fused submanifold sparse 3-D convolution hot path.

One step = one pass of the whole hot path over one batch of synthetic input:
the neighbour-map build from voxel coordinates (hash clear / insert / query)
followed by the fused gather-GEMM-accumulate convolution, on the decoder-scale
workload (3-thick shells of 12 random spheres in a 1024^3 grid, ~11.8 M
voxels, K = 27, Ci = Co = 128, bf16 in/out, fp32 accumulation).

Metric: TFLOP/s = 2 * valid_pairs * Ci * Co / time (whole job, all ranks).
Inputs are resident in HBM when the timed region starts; they are larger
than L2 (129 MB), so no flush is needed between steps.  ``e2e`` repeats the
measurement through the public API with pinned host buffers, host<->device
copies inside the timed region.  ``roofline`` reports the convolution
kernel's achieved FLOP/s against the measured dense bf16 tensor peak.
``cpu_baseline`` times the CPU oracle on a bounded sample of the workload.

``--impl reference`` times the CPU oracle alone (the reference arm: there is
no runnable reference implementation of this path on these machines).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "submconv3d TFLOP/s (2·valid_pairs·Ci·Co) & voxels/s; % of bf16 tensor roofline"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
DOMINANT_KERNEL = "submconv_tc_kernel<256, 1, 1, 0, 0, 0>"
XRUN_KERNEL = "submconv_xrun_kernel"
KERNEL_SOURCES = ("submanifold_voxel_gather_gb300/csrc/conv_tc.cu",
                  "submanifold_voxel_gather_gb300/csrc/ptx.cuh")
XRUN_SOURCES = ("submanifold_voxel_gather_gb300/csrc/conv_xrun.cu",
                "submanifold_voxel_gather_gb300/csrc/ptx.cuh")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decoder")
    ap.add_argument("--layer", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--path", choices=["auto", "tiles", "xrun"], default="auto",
                    help="conv path: 'tiles' = spconv_submconv3d (voxel tiles); 'xrun' = the x-run "
                         "slot layout (built in each step after the map) and the row-shifted conv; "
                         "'auto' = xrun where the layer's shape allows it (bf16, Ci = 128, Co <= 128, "
                         "the 27 lexicographic offsets), else tiles")
    ap.add_argument("--xrun", action="store_true", help="same as --path xrun")
    ap.add_argument("--no-numa-bind", action="store_true",
                    help="allocate the end-to-end pinned buffers without placing them near the GPU")
    ap.add_argument("--e2e-slots", type=int, default=3,
                    help="end-to-end steps in flight (one stream and buffer set each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-epilogue", action="store_true",
                    help="skip timing the fused residual + SiLU epilogue against the plain conv")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip timing the input and weight gradients on the same map")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="approximate CPU work of the oracle baseline sample")
    ap.add_argument("--materialized", action="store_true",
                    help="also time the materialising gather + GEMM path on the headline workload")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload lines (and the materialising comparison on medium)")
    return ap.parse_args()


def materialized_forward(torch, feats, nmap, w, bias, chunk):
    """The path the page replaces, on this GPU, with torch ops only: the
    (K, N, Ci) gather is materialised ``chunk`` offsets at a time
    (index_select over feats with a zero pad row appended, so the sentinel N
    selects zeros), each chunk is contracted by one cuBLAS GEMM with bf16
    inputs and an fp32 result, the chunk results are summed in fp32, the
    bias is added and the sum is rounded once.  Not part of the library."""
    k, n = nmap.shape
    ci, co = w.shape[1], w.shape[2]
    dev = feats.device
    padded = torch.cat([feats, torch.zeros((1, ci), dtype=feats.dtype, device=dev)])
    idx = torch.where((nmap >= 0) & (nmap < n), nmap, torch.full_like(nmap, n)).long()
    acc = torch.zeros((n, co), dtype=torch.float32, device=dev)
    for k0 in range(0, k, chunk):
        k1 = min(k, k0 + chunk)
        # voxel-major index order: the gather lands as (N, chunk * Ci) directly
        g = padded.index_select(0, idx[k0:k1].t().reshape(-1)).view(n, (k1 - k0) * ci)
        acc += torch.mm(g, w[k0:k1].reshape((k1 - k0) * ci, co), out_dtype=torch.float32)
        del g
    if bias is not None:
        acc += bias.float()
    return acc.to(feats.dtype)


def materialized_baseline(torch, sv, feats, nmap, w, bias, out_fused, reps=3):
    """Time and peak device memory of the materialising path (chunks of two
    offsets, as the page describes the stock layer, and the whole gather at
    once) next to the fused call, on the same inputs.  Peak memory is what
    each path allocates beyond its inputs and output."""
    k = nmap.shape[0]
    dev = feats.device
    res = {}
    for name, chunk in (("chunks_of_2_offsets", 2), ("whole_gather", k)):
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        got = materialized_forward(torch, feats, nmap, w, bias, chunk)
        torch.cuda.synchronize(dev)
        peak = torch.cuda.max_memory_allocated(dev) - base
        diff = float((got.float() - out_fused.float()).abs().max() / out_fused.float().abs().max())
        del got
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            r = materialized_forward(torch, feats, nmap, w, bias, chunk)
            del r
        e1.record()
        torch.cuda.synchronize(dev)
        res[name] = {"ms": e0.elapsed_time(e1) / reps, "peak_extra_gb": peak / 1e9,
                     "max_rel_diff_vs_fused": diff}
    # the fused call's own working set beyond its inputs and output: none
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        sv.submconv3d(feats, nmap, w, bias, out=out_fused)
    e1.record()
    torch.cuda.synchronize(dev)
    res["fused"] = {"ms": e0.elapsed_time(e1) / reps,
                    "peak_extra_gb": (torch.cuda.max_memory_allocated(dev) - base) / 1e9}
    return res


def max_over_ranks(torch, value, pg, device):
    """The job's clock: the largest per-rank time (ms) over the process group
    (the value itself on a single process)."""
    if pg is None:
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank, ms_per_step):
    """Whole-job throughput: every rank runs the same step (replicas), so the
    job does world x the per-rank FLOPs in the slowest rank's step time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel=DOMINANT_KERNEL):
    h = hashlib.sha256()
    for rel in (XRUN_SOURCES if kernel == XRUN_KERNEL else KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(workload, kernel=DOMINANT_KERNEL):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(kernel, {})
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash(kernel) or rec.get("workload") != workload:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_id):
        self.device_id = device_id
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.device_id is not None:
            cmd += ["-i", str(self.device_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def smi_device_id(torch, dev):
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return None


def build_workload(name, layer_index):
    import workloads as W
    t0 = time.time()
    wl = W.make(name)
    return wl, wl.layers[layer_index], time.time() - t0


def to_device(torch, arr, dtype, dev):
    a = np.ascontiguousarray(arr)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def parse_cpulist(text):
    """CPU ids of a Linux cpulist string such as "0-71,144-215"."""
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def gpu_local_cpus(torch, dev):
    """(NUMA node, CPU ids) of the host node nearest to `dev`, read from the
    PCI device's sysfs entry, or None where that is not readable."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        bdf = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        base = os.path.join("/sys/bus/pci/devices", bdf)
        with open(os.path.join(base, "numa_node")) as fh:
            node = int(fh.read())
        with open(os.path.join(base, "local_cpulist")) as fh:
            cpus = parse_cpulist(fh.read())
        return node, cpus
    except (AttributeError, OSError, ValueError):
        return None


def host_pinned(torch, arr, dtype):
    a = np.ascontiguousarray(arr)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dtype == "bf16" else torch.from_numpy(a)
    return t.pin_memory()


# --------------------------------------------------------------------- oracle
_PER_ROW_S = None


def oracle_step(wl, layer, seconds, threads, seed, keep=False):
    """One bounded oracle pass over a seeded sample of output rows: the
    neighbour-map rows (sort of all N voxels + binary searches) and the fp64
    conv loop nest of those rows, sized for about ``seconds`` of work on
    ``threads`` threads.  Returns (flops, timed seconds, rows), plus
    (rows, exact out, sum |terms|) when ``keep``."""
    global _PER_ROW_S
    import oracle
    import workloads as W
    n = wl.N

    def conv_rows(sub, rows, nthreads):
        full = np.full((wl.K, n), n, dtype=np.int32)   # untimed: sampled columns only
        full[:, rows] = sub
        t0 = time.perf_counter()
        res = oracle.conv(layer.feats, full, layer.w, layer.bias, layer.dtype, rows=rows, threads=nthreads)
        return time.perf_counter() - t0, res

    if _PER_ROW_S is None:   # untimed calibration
        cal = np.unique((W.draws_u64(7, 1, 0, 64) % np.uint64(n)).astype(np.int64))
        _PER_ROW_S = max(conv_rows(oracle.nmap_rows(wl.coords, wl.offsets, cal), cal, 1)[0] / len(cal),
                         1e-6)
    count = int(max(256, min(n, seconds * threads / _PER_ROW_S)))
    rows = np.unique((W.draws_u64(seed, 2, 0, count) % np.uint64(n)).astype(np.int64))
    t0 = time.perf_counter()
    sub = oracle.nmap_rows(wl.coords, wl.offsets, rows)
    t_map = time.perf_counter() - t0
    t_conv, (ref, sabs) = conv_rows(sub, rows, threads)
    pairs = int(((sub >= 0) & (sub < n)).sum())
    res = (2.0 * pairs * layer.Ci * layer.Co, t_map + t_conv, len(rows))
    return res + ((rows, ref, sabs),) if keep else res


def err_over_s(torch, out, rows, ref, sabs):
    """max over the listed rows of |gpu - exact| / sum|terms| (the quantity
    the acceptance tolerance bounds)."""
    got = out[torch.from_numpy(rows).to(out.device)].float().cpu().numpy().astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sabs > 0, np.abs(got - ref) / sabs, np.where(got == ref, 0.0, np.inf))
    return float(r.max()) if r.size else 0.0


def sampled_rows(n, count, seed):
    """First and last 160 rows plus ``count`` seeded rows, sorted, distinct."""
    import workloads as W
    rnd = (W.draws_u64(seed, 3, 0, count) % np.uint64(max(n, 1))).astype(np.int64)
    return np.unique(np.concatenate([np.arange(min(n, 160)), np.arange(max(0, n - 160), n), rnd]))


# Every workload of the benchmark suite other than the headline one: the
# per-config lines of the bench record.
PER_CONFIG = (("tiny", 0), ("small", 0), ("medium", 0), ("channel", 0), ("channel", 1))


def fp32_alu_tflops(torch, dev, sm_mhz):
    """CUDA-core fp32 peak: SMs x 128 fp32 lanes x 2 FLOP (FMA) x SM clock."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def per_config_lines(torch, sv, dev, bf16_peak, hbm_peak, sm_max_mhz, reps=10, check_rows=2048,
                     materialized_on="medium"):
    """Build + conv time, throughput, roofline fraction and parity (max
    |gpu - exact| / sum|terms| on sampled rows against the oracle's own map
    and loop nest) for each workload of PER_CONFIG.  L2 is flushed before
    every timed launch (a 256 MB write), since the small workloads fit in
    it.  Times are CUDA events on the launching stream, averaged over reps.
    Returns (lines, the materialising comparison on ``materialized_on``)."""
    import oracle
    import workloads as W
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    alu_peak = fp32_alu_tflops(torch, dev, sm_max_mhz)
    lines = {}
    mat = None
    wl = None
    for name, li in PER_CONFIG:
        if wl is None or wl.name != name:
            wl = None
            wl = W.make(name)
        layer = wl.layers[li]
        n, k, ci, co, dt = wl.N, wl.K, layer.Ci, layer.Co, layer.dtype
        coords = torch.from_numpy(wl.coords).to(dev)
        feats = to_device(torch, layer.feats, dt, dev)
        w = to_device(torch, layer.w, dt, dev)
        bias = to_device(torch, layer.bias, dt, dev)
        nmap = torch.empty((k, n), dtype=torch.int32, device=dev)
        out = torch.empty((n, co), dtype=feats.dtype, device=dev)
        ws = torch.empty(sv.workspace_size(n), dtype=torch.uint8, device=dev)
        tf = "tf32" if dt == "tf32" else None
        for _ in range(3):
            sv.build_nmap(coords, workspace=ws, out=nmap)
            sv.submconv3d(feats, nmap, w, bias, out=out, dtype=tf)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            sv.build_nmap(coords, workspace=ws, out=nmap)
            e[1].record(stream)
            flush.zero_()
            e[2].record(stream)
            sv.submconv3d(feats, nmap, w, bias, out=out, dtype=tf)
            e[3].record(stream)
        torch.cuda.synchronize(dev)
        sv.device_status()
        build_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / reps
        conv_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / reps
        pairs = sv.count_valid_pairs(nmap)
        flops = 2.0 * pairs * ci * co
        tflops = flops / (conv_ms * 1e-3) / 1e12
        elem = 2 if dt == "bf16" else 4
        comp = n * ci * elem + n * co * elem + 4 * k * n + k * ci * co * elem + co * elem
        if dt == "bf16":
            bound, peak, peak_src = "tensor", bf16_peak, "measured bf16 dense (burst)"
        else:
            bound, peak, peak_src = "alu", alu_peak, "fp32 CUDA-core peak (SMs x 128 lanes x 2 x max SM clock)"
        t_roof = max(flops / (peak * 1e12), comp / (hbm_peak * 1e9)) * 1e3
        rows = sampled_rows(n, check_rows, 40 + li)
        sub = oracle.nmap_rows(wl.coords, wl.offsets, rows)
        full = np.full((k, n), n, dtype=np.int32)
        full[:, rows] = sub
        ref, sabs = oracle.conv(layer.feats, full, layer.w, layer.bias, dt, rows=rows,
                                threads=oracle.host_threads())
        key = name if len(wl.layers) == 1 else f"{name}_layer{'AB'[li]}"
        lines[key] = {
            "N": n, "K": k, "Ci": ci, "Co": co, "dtype": dt, "valid_pairs": pairs,
            "conv_ms": conv_ms, "tflops": tflops, "voxels_per_s": n / (conv_ms * 1e-3),
            "bound": bound, "peak": peak, "peak_source": peak_src, "frac": tflops / peak,
            "t_roof_ms": t_roof, "frac_of_roofline": t_roof / conv_ms, "build_ms": build_ms,
            "build_voxels_per_s": n / (build_ms * 1e-3),
            "max_err_over_S": err_over_s(torch, out, rows, ref, sabs),
            "tol": oracle.TOL[dt], "rows_checked": int(len(rows)),
            "l2": "flushed before every timed launch"}
        if xrun_supported(layer, wl):
            # the row-shifted conv over the x-run slot layout, same inputs
            lib = sv.load_library()
            slots = torch.empty(int(lib.spconv_xrun_slot_capacity(n)), dtype=torch.int32, device=dev)
            count = torch.empty(1, dtype=torch.int64, device=dev)
            xws = torch.empty(int(lib.spconv_build_nmap_xrun_workspace_size(n)), dtype=torch.uint8, device=dev)
            for _ in range(3):
                sv.build_nmap_xrun(coords, out=nmap, slots=slots, slot_count=count, workspace=xws)
                sv.submconv3d_xrun(feats, nmap, slots, count, w, bias, out=out)
            for e in ev:
                flush.zero_()
                e[0].record(stream)
                sv.build_nmap_xrun(coords, out=nmap, slots=slots, slot_count=count, workspace=xws)
                e[1].record(stream)
                flush.zero_()
                e[2].record(stream)
                sv.submconv3d_xrun(feats, nmap, slots, count, w, bias, out=out)
                e[3].record(stream)
            torch.cuda.synchronize(dev)
            sv.device_status()
            xbuild_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / reps  # map + layout
            xconv_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / reps
            xt = flops / (xconv_ms * 1e-3) / 1e12
            lines[key]["xrun"] = {
                "conv_ms": xconv_ms, "build_ms": xbuild_ms, "tflops": xt, "frac": xt / peak,
                "frac_of_roofline": t_roof / xconv_ms, "slots": int(count.item()),
                "max_err_over_S": err_over_s(torch, out, rows, ref, sabs)}
            del slots, count, xws
        if name == materialized_on and dt == "bf16":
            mat = materialized_baseline(torch, sv, feats, nmap, w, bias, out)
            mat["workload"] = f"{name}: N={n}, {ci}->{co} {dt}"
        del coords, feats, w, bias, nmap, out, ws
    del flush
    return lines, mat


# --------------------------------------------------------------------- arms
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl, layer, _ = build_workload(args.workload, args.layer)
    threads = oracle.host_threads()
    step_seconds = max(2.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_step(wl, layer, step_seconds, threads, seed=500 + i)
    flops = secs = 0.0
    rows_total = 0
    for i in range(args.steps):
        f, s, r = oracle_step(wl, layer, step_seconds, threads, seed=1000 + i)
        flops += f
        secs += s
        rows_total += r
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": layer.dtype,
        "data": "synthetic (seeded generator)",
        "config": workload_config(wl, layer, xrun=use_xrun(args, layer, wl)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows_total // args.steps} seeded output rows per step "
                                   f"(neighbour map by sort + binary search, fp64 conv loop nest)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, layer, pairs=None, xrun=False):
    cfg = {"workload": f"decoder-scale: {wl.note}" if wl.name == "decoder" else f"{wl.name}: {wl.note}",
           "N": wl.N, "K": wl.K, "Ci": layer.Ci, "Co": layer.Co, "seed": wl.seed,
           "step": ("build_nmap + xrun_layout + submconv3d_xrun" if xrun else "build_nmap + submconv3d"),
           "l2": "inputs larger than L2 (no flush between steps)"}
    if pairs is not None:
        cfg["valid_pairs"] = pairs
    return cfg


def copy_bandwidths(torch, dev, d_in, h_in, d_out, h_out, streams, reps=3):
    """Pinned host<->device copy rates (GB/s) measured with CUDA events:
    host->device alone (h_in -> d_in), device->host alone (d_out -> h_out),
    and both at once on two streams."""
    h2d = h_in.numel() * h_in.element_size()
    d2h = d_out.numel() * d_out.element_size()
    main = torch.cuda.current_stream(dev)

    def timed(fn):
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for st in streams:
            st.wait_event(e0)
        for _ in range(reps):
            fn()
        for st in streams:
            main.wait_stream(st)
        e1.record(main)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    def up():
        with torch.cuda.stream(streams[0]):
            d_in.copy_(h_in, non_blocking=True)

    def down():
        with torch.cuda.stream(streams[1]):
            h_out.copy_(d_out, non_blocking=True)

    up()      # untimed first use of each path (the first copy of a process can be slow)
    down()
    t_up = timed(up)
    t_down = timed(down)
    t_both = timed(lambda: (up(), down()))
    return {"h2d_gbs": h2d / t_up / 1e6, "d2h_gbs": d2h / t_down / 1e6,
            "both_gbs": (h2d + d2h) / t_both / 1e6}


def time_calls(torch, fn, stream, reps=5, warmup=2):
    """Mean device time of fn() over reps calls (CUDA events on `stream`)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def time_pair(torch, fa, fb, stream, rounds=4, reps=2):
    """Median device times of fa() and fb(), measured in alternation (a
    clock that drifts during the run then biases neither)."""
    ta, tb = [], []
    for _ in range(rounds):
        ta.append(time_calls(torch, fa, stream, reps=reps, warmup=1))
        tb.append(time_calls(torch, fb, stream, reps=reps, warmup=1))
    return float(np.median(ta)), float(np.median(tb))


def xrun_supported(layer, wl):
    """Shapes the row-shifted conv takes: bf16, Ci = 128, Co <= 128, the 27
    lexicographic 3x3x3 offsets."""
    import workloads as W
    return (layer.dtype == "bf16" and layer.Ci == 128 and layer.Co <= 128 and
            np.array_equal(np.asarray(wl.offsets), W.offsets_3x3x3()))


def use_xrun(args, layer, wl):
    if args.xrun or args.path == "xrun":
        if not xrun_supported(layer, wl):
            raise SystemExit("the x-run path takes bf16, Ci = 128, Co <= 128 and the 27 lexicographic offsets")
        return True
    return args.path == "auto" and xrun_supported(layer, wl)


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    import submanifold_voxel_gather_gb300 as sv
    sv.load_library()
    wl, layer, gen_s = build_workload(args.workload, args.layer)
    n, k, ci, co = wl.N, wl.K, layer.Ci, layer.Co
    dtype = layer.dtype

    coords = torch.from_numpy(wl.coords).to(dev)
    feats = to_device(torch, layer.feats, dtype, dev)
    w = to_device(torch, layer.w, dtype, dev)
    bias = to_device(torch, layer.bias, dtype, dev)
    nmap = torch.empty((k, n), dtype=torch.int32, device=dev)
    out = torch.empty((n, co), dtype=feats.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    tf = "tf32" if dtype == "tf32" else None

    args.xrun = use_xrun(args, layer, wl)
    xrun = None
    lib = sv.load_library()
    if args.xrun:
        # the map and the x-run slot layout come from one call (one workspace)
        xrun = {"slots": torch.empty(int(lib.spconv_xrun_slot_capacity(n)), dtype=torch.int32, device=dev),
                "count": torch.empty(1, dtype=torch.int64, device=dev)}
        ws = torch.empty(int(lib.spconv_build_nmap_xrun_workspace_size(n)), dtype=torch.uint8, device=dev)
    else:
        ws = torch.empty(sv.workspace_size(n), dtype=torch.uint8, device=dev)

    def build(c, nm, w_s, x, status=None, stream=None):
        if x is not None:
            sv.build_nmap_xrun(c, out=nm, slots=x["slots"], slot_count=x["count"], workspace=w_s, status=status,
                               stream=stream)
        else:
            sv.build_nmap(c, workspace=w_s, out=nm, status=status, stream=stream)

    def conv(f, nm, ww, b, o, x, stream=None):
        if x is not None:
            sv.submconv3d_xrun(f, nm, x["slots"], x["count"], ww, b, out=o, stream=stream)
        else:
            sv.submconv3d(f, nm, ww, b, out=o, dtype=tf, stream=stream)

    def step():
        build(coords, nmap, ws, xrun)
        conv(feats, nmap, w, bias, out, xrun)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    sv.device_status()
    pairs = sv.count_valid_pairs(nmap)
    flops = 2.0 * pairs * ci * co

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(smi_device_id(torch, dev))
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(args.steps):
        build(coords, nmap, ws, xrun)
        ev[i][0].record(stream)
        conv(feats, nmap, w, bias, out, xrun)
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    conv_ms = [a.elapsed_time(b) for a, b in ev]
    conv_avg_ms = sum(conv_ms) / len(conv_ms)
    if pg is not None:
        total_ms = max_over_ranks(torch, total_ms, pg, dev)
        pg.barrier()
    sv.device_status()
    ms_per_step = total_ms / args.steps

    # ---- device memory the step uses beyond its inputs (coords, feats, w,
    # bias) and outputs (nmap, out): the map build's workspace, which the
    # caller allocates once, plus anything allocated during a step (the
    # library allocates nothing; the conv needs no workspace)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    build(coords, nmap, ws, xrun)
    torch.cuda.synchronize(dev)
    during_build = torch.cuda.max_memory_allocated(dev) - base
    torch.cuda.reset_peak_memory_stats(dev)
    conv(feats, nmap, w, bias, out, xrun)
    torch.cuda.synchronize(dev)
    during_conv = torch.cuda.max_memory_allocated(dev) - base
    ws_bytes = ws.numel() * ws.element_size()
    if xrun is not None:  # the slot layout's buffers are scratch of the step too
        ws_bytes += sum(v.numel() * v.element_size() for v in xrun.values())
    peak_extra = {"bytes": ws_bytes + max(during_build, during_conv), "build_workspace_bytes": ws_bytes,
                  "allocated_during_build": during_build, "allocated_during_conv": during_conv,
                  "gather_materialised_bytes": 0,
                  "note": "nmap (4*K*N bytes) is the build's output and the conv's input, not counted"}

    # ---- the fused epilogue out = SiLU(conv + bias + residual) against the
    # plain conv, on the same map and the same conv kernel
    epilogue = None
    if not args.no_epilogue:
        res = out.clone()
        out2 = torch.empty_like(out)

        def fused_conv():
            if xrun is not None:
                sv.submconv3d_xrun(feats, nmap, xrun["slots"], xrun["count"], w, bias, out=out2, residual=res,
                                   activation="silu")
            else:
                sv.submconv3d(feats, nmap, w, bias, out=out2, residual=res, activation="silu", dtype=tf)

        plain_ms, fused_ms = time_pair(torch, lambda: conv(feats, nmap, w, bias, out2, xrun), fused_conv, stream)
        epilogue = {"plain_ms": plain_ms, "fused_ms": fused_ms, "ratio": fused_ms / plain_ms,
                    "act": "silu", "residual": True, "kernel": XRUN_KERNEL if xrun is not None else DOMINANT_KERNEL}
        if xrun is not None:
            # the voxel-tile kernel's fused epilogue on the same inputs
            tp, tf_ms = time_pair(torch, lambda: sv.submconv3d(feats, nmap, w, bias, out=out2, dtype=tf),
                                  lambda: sv.submconv3d(feats, nmap, w, bias, out=out2, residual=res,
                                                        activation="silu", dtype=tf), stream)
            epilogue["tiles"] = {"plain_ms": tp, "fused_ms": tf_ms, "ratio": tf_ms / tp, "kernel": DOMINANT_KERNEL}
        sv.device_status()
        del res, out2
        torch.cuda.empty_cache()

    # ---- backward on the same map, outside the timed region: the input
    # gradient (over the x-run layout when the step uses it) and the weight
    # gradient, with this step's output standing in for dout
    backward = None
    if not args.no_backward and dtype == "bf16":
        dout = out.clone()
        din = torch.empty_like(feats)

        xrun_dgrad = xrun is not None and co == 128  # the x-run input gradient reduces 128 channels

        def dgrad():
            if xrun_dgrad:
                sv.submconv3d_dgrad_xrun(dout, nmap, xrun["slots"], xrun["count"], w, out=din)
            else:
                sv.submconv3d_dgrad(dout, nmap, w, out=din)

        dg_ms = time_calls(torch, dgrad, stream, reps=3, warmup=1)
        wg_ms = time_calls(torch, lambda: sv.submconv3d_wgrad(feats, dout, nmap), stream, reps=3, warmup=1)
        sv.device_status()
        backward = {"dgrad_ms": dg_ms, "dgrad_tflops": flops / (dg_ms * 1e-3) / 1e12,
                    "dgrad_kernel": XRUN_KERNEL if xrun_dgrad else DOMINANT_KERNEL,
                    "wgrad_ms": wg_ms, "wgrad_tflops": flops / (wg_ms * 1e-3) / 1e12,
                    "wgrad_kernel": "wgrad_tc_kernel", "note": "2*valid_pairs*Ci*Co FLOPs each"}
        del dout, din
        torch.cuda.empty_cache()

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        # Pinned buffers are placed in the host memory nearest the GPU: the
        # process runs on that node's CPUs while they are allocated (the
        # kernel places their pages on the allocating CPU's node), then
        # returns to its previous CPU set.
        host_node = None
        prev_cpus = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
        local = gpu_local_cpus(torch, dev) if not args.no_numa_bind else None
        if local is not None and prev_cpus is not None:
            node, cpus = local
            cpus &= prev_cpus
            bind = bool(cpus) and cpus != prev_cpus
            if bind:
                os.sched_setaffinity(0, cpus)
            host_node = {"node": node, "local_cpus": len(cpus), "bound": bind}
        h_coords = torch.from_numpy(wl.coords).pin_memory()
        h_feats = host_pinned(torch, layer.feats, dtype)
        h_w = host_pinned(torch, layer.w, dtype)
        h_bias = host_pinned(torch, layer.bias, dtype)
        # Several steps in flight: step i runs on stream i % S with its own
        # device and pinned output buffers, so its host->device copies overlap
        # the kernels and device->host reads of the steps before it (the map
        # build reports its verdict on the device instead of waiting).  With
        # S = 3 each stream's chain (copy in, build, conv, copy out) spans
        # three steps, so both copy directions stay busy: measured on GB300,
        # pinned copies reach ~210 GB/s one way and ~340 GB/s both ways at
        # once, and a step moves ~6.2 GB.  Every step still copies all its
        # inputs from pinned host memory and reads its whole output back; the
        # verdicts are checked after the timed region.
        nslots = args.e2e_slots
        streams = [torch.cuda.Stream(dev) for _ in range(nslots)]
        slots = []
        for _ in range(nslots):
            slots.append({
                "coords": torch.empty_like(coords), "feats": torch.empty_like(feats),
                "w": torch.empty_like(w), "bias": torch.empty_like(bias),
                "nmap": torch.empty_like(nmap), "ws": torch.empty_like(ws), "out": torch.empty_like(out),
                "status": torch.full((1,), -99, dtype=torch.int32, device=dev),
                "xrun": None if xrun is None else {k: torch.empty_like(v) for k, v in xrun.items()},
                "h_out": torch.empty((n, co), dtype=feats.dtype).pin_memory()})
        if host_node is not None and host_node["bound"]:
            os.sched_setaffinity(0, prev_cpus)

        def e2e_step(i):
            sl, st = slots[i % nslots], streams[i % nslots]
            with torch.cuda.stream(st):
                sl["coords"].copy_(h_coords, non_blocking=True)
                sl["feats"].copy_(h_feats, non_blocking=True)
                sl["w"].copy_(h_w, non_blocking=True)
                sl["bias"].copy_(h_bias, non_blocking=True)
                build(sl["coords"], sl["nmap"], sl["ws"], sl["xrun"], status=sl["status"], stream=st)
                conv(sl["feats"], sl["nmap"], sl["w"], sl["bias"], sl["out"], sl["xrun"], stream=st)
                sl["h_out"].copy_(sl["out"], non_blocking=True)

        main = torch.cuda.current_stream(dev)
        for i in range(nslots):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for st in streams:
            st.wait_event(e0)
        for i in range(args.steps):
            e2e_step(i)
        for st in streams:
            main.wait_stream(st)
        e1.record(main)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1)
        e2e_ms = max_over_ranks(torch, e2e_ms, pg, dev)
        bad = [int(sl["status"].item()) for sl in slots if int(sl["status"].item()) != 0]
        if bad:
            raise RuntimeError(f"map build reported status {bad} in the end-to-end loop")
        h2d = sum(t.numel() * t.element_size() for t in (h_coords, h_feats, h_w, h_bias))
        d2h = slots[0]["h_out"].numel() * slots[0]["h_out"].element_size()

        # The copies' own floor on this machine: each direction's bytes at that
        # direction's measured one-way rate, the two directions fully
        # overlapped.  No schedule of the loop above can move its bytes
        # faster.  (both_gbs, one large copy each way on two streams at
        # once, is reported beside it: how much the copy engines overlap
        # the two directions depends on the streams they are given.)
        bw = copy_bandwidths(torch, dev, slots[0]["feats"], h_feats, slots[0]["out"], slots[0]["h_out"],
                             streams[:2])
        floor_ms = max(h2d / bw["h2d_gbs"], d2h / bw["d2h_gbs"]) / 1e6
        e2e = {"value": job_tflops(world, flops, e2e_ms / args.steps), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / args.steps, "steps_in_flight": nslots, "host_node": host_node,
               "achieved_copy_gbs": (h2d + d2h) / (e2e_ms / args.steps) / 1e6,
               "copy_floor": dict(bw, floor_ms_per_step=floor_ms)}
        del e2e_step, slots, streams, h_coords, h_feats, h_w, h_bias
        torch.cuda.empty_cache()

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0

    materialized = None
    if args.materialized and dtype == "bf16":
        materialized = materialized_baseline(torch, sv, feats, nmap, w, bias, out)

    bf16_peak, hbm_peak, peak_kind = peaks()
    achieved = flops / (conv_avg_ms * 1e-3) / 1e12
    elem = 2 if dtype == "bf16" else 4
    comp_bytes = n * ci * elem + n * co * elem + 4 * k * n + k * ci * co * elem + co * elem
    t_roof_ms = max(flops / (bf16_peak * 1e12), comp_bytes / (hbm_peak * 1e9)) * 1e3
    roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak,
                "traffic": recorded_traffic(args.workload, XRUN_KERNEL if args.xrun else DOMINANT_KERNEL),
                "kernel": XRUN_KERNEL if args.xrun else DOMINANT_KERNEL, "peak_source": f"{peak_kind} bf16 dense (burst)",
                "algorithmic_flops_per_launch": flops, "conv_ms": conv_avg_ms,
                "compulsory_bytes": comp_bytes, "t_roof_ms": t_roof_ms,
                "frac_of_roofline": t_roof_ms / conv_avg_ms}

    cpu = None
    import oracle
    threads = oracle.host_threads()
    if not args.no_cpu_baseline and world == 1:
        f, s, r, (rows, ref, sabs) = oracle_step(wl, layer, args.cpu_seconds, threads, seed=99, keep=True)
        cpu = {"value": f / s / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{r} seeded output rows of the same workload: neighbour map by sort + "
                         f"binary search over all N voxels, fp64 conv loop nest over the sample; "
                         f"{s:.1f} s"}
    else:
        _, _, _, (rows, ref, sabs) = oracle_step(wl, layer, 1.0, threads, seed=99, keep=True)
    # parity of this run's output on the oracle's sampled rows (its own map rows)
    parity = {"max_err_over_S": err_over_s(torch, out, rows, ref, sabs), "tol": oracle.TOL[dtype],
              "rows_checked": int(len(rows))}

    per_config, mat_medium = None, None
    if not args.no_per_config:
        del coords, feats, w, bias, nmap, ws
        torch.cuda.empty_cache()
        per_config, mat_medium = per_config_lines(torch, sv, dev, bf16_peak, hbm_peak,
                                                  clocks.get("sm_max_mhz") or 2070.0)
    if materialized is None:
        materialized = mat_medium

    line = {
        "metric": METRIC, "value": job_tflops(world, flops, ms_per_step), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded generator; decoder-scale voxel shells, random-init weights)",
        "config": workload_config(wl, layer, pairs, xrun=args.xrun),
        "voxels_per_s": world * n / (ms_per_step * 1e-3),
        "conv_tflops": achieved,
        "build_ms": ms_per_step - conv_avg_ms,
        "roofline": roofline,
        "max_err_over_S": parity["max_err_over_S"],
        "parity": parity,
        "peak_extra_bytes": peak_extra["bytes"],
        "peak_extra": peak_extra,
        "cpu_baseline": cpu,
        "e2e": e2e,
        **({"epilogue": epilogue} if epilogue is not None else {}),
        **({"backward": backward} if backward is not None else {}),
        # per step: the map build's seven kernels (flag reset, range/order/box
        # check, clear, insert, dense-row query, row-hash query, voxel-hash
        # query: the paths not taken return at once) and one conv launch
        # (Co <= 256) (on the x-run path: three layout kernels and one conv
        # launch)
        "gpu_launches": ((7 + 3 + 1) if args.xrun else (7 + (co + 255) // 256)) * args.steps,
        "clocks": clocks,
        "generation_s": gen_s,
        **({"per_config": per_config} if per_config is not None else {}),
        **({"materialized": materialized} if materialized is not None else {}),
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
