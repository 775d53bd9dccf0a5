"""The band's tile ranges (shared by the forward and backward kernels) against
brute force over thousands of shapes and windows, on the host: compiles
tests/tile_ranges_check.cu with nvcc and runs it (no GPU needed)."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tile_ranges_match_brute_force():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "tile_ranges_check")
        subprocess.run([nvcc, "-O2", "-std=c++17", "-o", exe,
                        os.path.join(HERE, "tile_ranges_check.cu")], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "bad 0" in r.stdout
