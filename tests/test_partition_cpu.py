"""The static work partition (csrc/common.cuh) checked on the host: tests/host/partition_check.cpp
is compiled against the library's own header and run."""
import os
import shutil
import subprocess

import pytest

from sparse_mla_paged_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))


def test_partition_invariants(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(B.nvcc())), "include")
    exe = str(tmp_path / "partition_check")
    subprocess.check_call([cxx, "-std=c++17", "-O2", "-I", B.INCLUDE, "-I", B.CSRC, "-I", cuda_inc,
                           os.path.join(HERE, "host", "partition_check.cpp"), "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "partition ok" in r.stdout
