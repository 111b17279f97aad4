"""The decode work partition, checked on the host against the real map
functions of kivi_common.cuh (compiled with nvcc as host code; no GPU):
every unit owned once, contiguous partial indices, at most the workspace's
partials per slot, for dense, ragged, lead-in and capped grids."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_partition_covers_every_unit_once(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "partition_check"
    src = os.path.join(ROOT, "tests", "partition_check.cu")
    cmd = [nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "bit_kivi_kv_gb300", "csrc"), src, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:]
