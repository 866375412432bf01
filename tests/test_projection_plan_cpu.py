"""The tensor-core projection's host-side launch plan, checked over a sweep of shapes
by a small host program compiled here (no GPU): chunk coverage, shared-memory and TMEM
limits, pairing rules and the split-partial budget (tests/host/projection_plan_check.cc)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CUDA_INC = "/usr/local/cuda/include"


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                    reason="needs g++ and the CUDA headers")
def test_projection_plans_respect_the_kernel_limits(tmp_path):
    exe = tmp_path / "projection_plan_check"
    src = os.path.join(HERE, "host", "projection_plan_check.cc")
    inc = os.path.join(os.path.dirname(HERE), "include")
    subprocess.run(["g++", "-std=c++17", "-O1", "-x", "c++", "-I", CUDA_INC, "-I", inc, src,
                    "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok ")
