"""CPU checks of bench.py's bookkeeping (no GPU, nothing timed).

The DRAM traffic a bench line reports comes from committed ncu captures and
is only used while the kernel's sources are unchanged; the source list of
each operator must therefore include every header its .cu file includes.
"""
import os
import re

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "point_cloud_neighbor_gb300", "csrc")


def includes(name, seen=None):
    seen = set() if seen is None else seen
    text = open(os.path.join(CSRC, name)).read()
    for inc in re.findall(r'#include "(pc_[a-z_]+[.]cuh)"', text):
        if inc not in seen:
            seen.add(inc)
            includes(inc, seen)
    return seen


def test_kernel_source_lists_cover_their_includes():
    for op, files in bench.KERNEL_SOURCES.items():
        missing = includes(files[0]) - set(files)
        assert not missing, f"{op}: {sorted(missing)} not hashed"


def test_recorded_traffic_lines_parse():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    n = 0
    for line in open(path):
        if line.startswith("#") or not line.strip():   # the header: command, notes
            continue
        kv = dict(p.split("=", 1) for p in line.split())
        assert kv["op"] in bench.KERNEL_SOURCES
        assert float(kv["dram_bytes_per_launch"]) > 0
        n += 1
    assert n > 0


def test_warmup_below_three_is_rejected():
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"),
                        "--warmup", "2"], capture_output=True, text=True)
    assert r.returncode != 0 and "warmup" in r.stderr
