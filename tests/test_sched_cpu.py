"""The GEMM's tile schedule (whole-tile waves, then stream-K pieces), checked
on the CPU: tests/sched_check.cu includes the kernel header, walks every
CTA's segments for a sweep of shapes and checks coverage, K order, the
partial-tile slots and the workspace capacity that the kernels and the
stream-K reduction rely on.  Compiled with nvcc (host code; no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


@pytest.mark.skipif(not os.path.exists(NVCC) and shutil.which("nvcc") is None, reason="no nvcc")
def test_schedule_invariants(tmp_path):
    nvcc = NVCC if os.path.exists(NVCC) else shutil.which("nvcc")
    exe = str(tmp_path / "sched_check")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "fp8_fine_grained_21_b300", "csrc"),
                    os.path.join(ROOT, "tests", "sched_check.cu"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok "), out.stdout
