"""bench.py host logic on CPU: the `traffic` lookup in the committed ncu summaries.

A summary covers one kernel on one workload and records the hash of the kernel's
sources when it was captured; the benchmark reports its DRAM bytes only while the
sources still hash to that, and only for the workload the summary names.
"""
import hashlib
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _profile(kernel, digest, traffic):
    return (f"ncu --set full summary: {kernel}, test workload\nkernel: {kernel}\n"
            f"source_sha256_16: {digest}\ntraffic_bytes_per_launch: {traffic}\n\nbody\n")


def test_read_traffic_keyed_to_kernel_workload_and_sources(tmp_path):
    import bench
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    pdir = tmp_path / "profiles"
    pdir.mkdir()
    (pdir / "k_kernel_wl.txt").write_text(_profile("k_kernel", digest, 123456))
    assert bench.read_traffic("k_kernel_wl", "k_kernel", [str(src)], str(pdir)) == (123456.0, digest)
    # another kernel's name, another workload's file, no file at all
    assert bench.read_traffic("k_kernel_wl", "other_kernel", [str(src)], str(pdir))[0] is None
    assert bench.read_traffic("k_kernel_other_wl", "k_kernel", [str(src)], str(pdir))[0] is None
    # a source edited after the capture: the summary no longer describes the kernel
    src.write_bytes(b"__global__ void k() { /* changed */ }\n")
    got, new_digest = bench.read_traffic("k_kernel_wl", "k_kernel", [str(src)], str(pdir))
    assert got is None and new_digest != digest


def test_committed_summaries_are_well_formed():
    """Every committed summary that carries a traffic figure names its kernel, its
    source hash and the source files that hash covers, and those files exist."""
    pdir = os.path.join(ROOT, "profiles")
    found = 0
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".txt"):
            continue
        txt = open(os.path.join(pdir, f)).read()
        if not re.search(r"^traffic_bytes_per_launch:", txt, re.M):
            continue
        found += 1
        kernel = re.search(r"^kernel:\s*(\S+)", txt, re.M)
        digest = re.search(r"^source_sha256_16:\s*([0-9a-f]{16})$", txt, re.M)
        traffic = re.search(r"^traffic_bytes_per_launch:\s*([0-9]+)$", txt, re.M)
        srcs = re.search(r"^source hash: sha256 of (.+?), first 16 hex", txt, re.M | re.S)
        assert kernel and digest and traffic and srcs, f
        assert f.startswith(kernel.group(1)), f
        assert int(traffic.group(1)) > 0, f
        for name in re.split(r"\s*\+\s*", " ".join(srcs.group(1).split())):
            assert os.path.isfile(os.path.join(ROOT, "sparse_selected_cell_gb300", "csrc", name)), (f, name)
    assert found >= 4
