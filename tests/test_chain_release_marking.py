"""The decode chain publishes a dependency group's completion with a GPU-scope
release only where a later matmul reads or rewrites memory written up to that
group, or rewrites memory read up to it.  The host-side marking is checked here
against brute force on random chains whose buffers overlap (no GPU: the check
program makes no CUDA call)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_release_marking_matches_brute_force(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "chain_release_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-gencode",
                    "arch=compute_103a,code=sm_103a", "-o", exe, os.path.join(HERE, "chain_release_check.cu")],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches 0" in out.stdout
