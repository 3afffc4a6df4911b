"""Host-side consistency of the benchmark with the library (CPU only).

bench.py names the dominant kernel from the per-kernel timings the library records, looks up
that kernel's algorithmic bytes and, through the source digest, the DRAM traffic of a committed
ncu summary.  These tests read the library's sources and the summaries as text and check that
every recorded kernel name has a byte count and a source list, and that every summary carries
the keys the benchmark parses.
"""
import os
import re

import pytest

import bench
from ssm_sequence_layer_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "ssm_sequence_layer_gb300", "csrc")


def recorded_names():
    names = set()
    for fn in os.listdir(CSRC):
        if fn.endswith(".cu"):
            names |= set(re.findall(r'tm\.begin\("([a-z_0-9]+)"\)', open(os.path.join(CSRC, fn)).read()))
    return names


def test_every_backward_kernel_has_algorithmic_bytes():
    w = WORKLOADS["seqrec_16k"]
    bwd = {n for n in recorded_names() if n.startswith("bwd_")}
    assert bwd, "no backward kernel names found"
    for n in bwd:
        assert bench.backward_kernel_bytes(n, w) > 0, n


def test_every_forward_kernel_has_algorithmic_bytes():
    w = WORKLOADS["seqrec_16k"]
    for n in recorded_names():
        if n.startswith(("simt_", "tc_", "map_")):
            assert bench.kernel_alg_bytes(n, w) > 0, n


@pytest.mark.parametrize("prefix", sorted(bench.KERNEL_SOURCES))
def test_kernel_source_lists_name_existing_files(prefix):
    for fn in bench.KERNEL_SOURCES[prefix]:
        assert os.path.exists(os.path.join(CSRC, fn)), fn
    assert re.fullmatch(r"[0-9a-f]{16}", bench.source_digest(prefix + "x"))


def test_profile_summaries_carry_the_parsed_keys():
    prof = os.path.join(ROOT, "profiles")
    for fn in sorted(os.listdir(prof)):
        text = open(os.path.join(prof, fn)).read()
        assert fn.endswith((".md", ".txt")), fn
        assert "ncu" in text, f"{fn} does not give the command that made it"
        if "dram_bytes_per_launch:" in text:
            assert re.search(r"dram_bytes_per_launch:\s*[0-9.eE+]+", text), fn
            assert re.search(r"source_digest:\s*[0-9a-f]{16}\b", text), fn
