"""The C-ABI example (paged_kv_cache_317_gb300/examples/c_abi_step.cu) builds
against include/pagedkv.h and libpagedkv.so alone, and on a GPU runs a decode step
whose exact self-checks pass (decode, shared-partition decode and chunked prefill)."""

import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_317_gb300")
SRC = os.path.join(PKG, "examples", "c_abi_step.cu")


def _build(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "c_abi_step")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-I", os.path.join(ROOT, "include"), SRC, "-L", PKG, "-lpagedkv",
           "-Xlinker", "-rpath," + PKG, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return exe


def test_c_example_builds_against_the_header_and_library(lib, tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_example_runs(lib, tmp_path):
    r = subprocess.run([_build(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok:" in r.stdout
    m = re.search(r"(\d+)-token partitions, (\d+) work items", r.stdout)
    assert m and int(m.group(1)) <= 64 and int(m.group(2)) > 3   # the split path, work list
    assert "2 records" in r.stdout                  # the shared-partition pass ran
    assert "prefix records: 1 record" in r.stdout   # prefix record, tail item, device counts
    assert "prefill: fork exact" in r.stdout        # the tensor-core prefill ran
