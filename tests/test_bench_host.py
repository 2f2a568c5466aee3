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
