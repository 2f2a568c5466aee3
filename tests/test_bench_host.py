"""bench.py's host-side helpers on CPU: the Linux cpulist parser used to
place the end-to-end pinned buffers on the GPU's NUMA node."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_cpulist_ranges_and_singles():
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}


def test_cpulist_single_cpu_and_empty():
    assert bench.parse_cpulist("5") == {5}
    assert bench.parse_cpulist("") == set()
    assert bench.parse_cpulist("\n") == set()


def test_cpulist_matches_this_host():
    # the running process's own cpulist, where Linux exposes it
    path = "/sys/devices/system/cpu/online"
    if not os.path.exists(path):
        return
    with open(path) as fh:
        online = bench.parse_cpulist(fh.read())
    assert os.sched_getaffinity(0) <= online


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference (the CPU oracle arm) on a small workload:
    one JSON line with the contract's keys, the same metric and unit as the
    GPU arm, and a cpu_baseline / e2e describing this run."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "small", "--steps", "1", "--warmup", "1", "--cpu-seconds", "0.5"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["N"] > 0 and "workload" in d["config"]
