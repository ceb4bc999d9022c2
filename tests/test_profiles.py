"""The committed ncu summaries under profiles/ (no GPU).

Each summary named <kernel>_<workload>.md carries the stamp of the kernel sources it profiled and
the DRAM bytes of one launch, which bench.py reports as ``roofline.traffic`` only while the stamp
still matches the sources.  Every ncu command recorded there leaves the GPU clocks alone.
"""

import os
import re

import pytest

import bench
from persistent_warp_specialized_gb300 import _build

PROFILES = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
FILES = sorted(os.listdir(PROFILES))


def kernel_of(name):
    """The kernel a summary file is named for (longest matching prefix), or None."""
    hits = [k for k in _build.KERNEL_SOURCES if name.startswith(k + "_")]
    return max(hits, key=len) if hits else None


def test_profiles_hold_text_summaries_only():
    assert FILES
    for name in FILES:
        assert name.endswith((".md", ".txt")), name


@pytest.mark.parametrize("name", FILES)
def test_every_ncu_command_keeps_the_clocks(name):
    # an ncu invocation, possibly continued over backslash-newlines
    text = open(os.path.join(PROFILES, name)).read().replace("\\\n", " ")
    for cmd in re.findall(r"^\s*ncu .*$", text, flags=re.M):
        assert "--clock-control none" in cmd, (name, cmd[:80])


@pytest.mark.parametrize("name", [n for n in FILES if kernel_of(n)])
def test_kernel_summary_has_stamp_and_bytes(name):
    text = open(os.path.join(PROFILES, name)).read()
    stamp = re.search(r"source_stamp:\s*`([0-9a-f]+)`", text)
    dram = re.search(r"dram_bytes_per_launch:\s*`([0-9]+)`", text)
    assert stamp and len(stamp.group(1)) == 64, name
    assert dram and int(dram.group(1)) > 0, name
    # bench.py uses the bytes exactly when the stamp is that of the sources on disk
    kernel = kernel_of(name)
    workload = "gemm_" + name[len(kernel) + 1:-len(".md")]
    got = bench.profile_traffic(kernel, workload)
    if stamp.group(1) == _build.kernel_stamp(kernel):
        assert got == float(dram.group(1)), name
    else:
        assert got is None, name

