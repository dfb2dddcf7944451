"""Host-side checks of bench.py's bookkeeping (no GPU).

`roofline.traffic` is read from profiles/traffic.txt only while a kernel's
source hash matches the one its DRAM capture was taken at, so the hash must
cover every file the kernel's translation unit includes from the library's
sources; and every committed row must parse and name a known kernel."""
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "chunked_causal_gqa_gb300", "csrc")


def _local_includes(path):
    with open(path) as f:
        names = re.findall(r'^#include "([^"]+)"', f.read(), flags=re.M)
    return [n for n in names if os.path.isfile(os.path.join(CSRC, n))]


def test_source_hash_covers_every_included_kernel_header():
    for kernel, src in bench.KERNEL_SOURCES.items():
        hashed = {"pfa_ptx.cuh"} | {os.path.basename(h) for h in bench.KERNEL_HEADERS.get(kernel, ())}
        # the host-side header pfa_internal.h holds declarations only
        needed = {n for n in _local_includes(os.path.join(ROOT, src)) if n.endswith(".cuh")}
        assert needed <= hashed, (kernel, needed - hashed)
        assert len(bench.source_hash(kernel)) == 16


def test_traffic_rows_parse_and_name_known_kernels():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert rows
    for r in rows:
        assert len(r) == 4, r
        kernel, workload, h, nbytes = r
        assert kernel in bench.KERNEL_SOURCES, r
        assert re.fullmatch(r"[0-9a-f]{16}", h), r
        assert int(nbytes) > 0
