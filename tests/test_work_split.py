"""The tensor-core kernels' work split, checked on the CPU: `tests/host/work_split_check.cu` includes the
kernels' own `la_tc_common.cuh` (slices, chunk owner, pieces, slot numbering and slot layout, the grid
size choice), is compiled by nvcc as a host program and brute-forces their invariants over every small
shape and 3000 random large ones.  No GPU is used."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_split_invariants(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = tmp_path / "work_split_check"
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "bwd_la_fwd_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "host", "work_split_check.cu"), "-o", str(exe)],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
