"""The CUDA library's work partition (xsymv_plan.h, host-side integer logic)
checked by brute force on the CPU: a C++ harness simulates every warp of the
main kernel for many sizes, tile edges, warp counts and column costs."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_partition_brute_force(tmp_path):
    exe = tmp_path / "plan_check"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I",
                    os.path.join(ROOT, "symmetric_matrix_vector_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "plan_check.cpp"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-2000:]
    assert "0 failures" in out.stdout
