"""The debug build's index check (GCL_DEBUG_BOUNDS) on the CPU: the same header the kernels
include, compiled with g++ with and without the macro."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("debug", [True, False], ids=["debug", "release"])
def test_bounds_check_flags_out_of_range_indices(debug, tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "bounds_check")
    cmd = [gxx, "-std=c++17", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "chunked_gated_linear_gb300", "csrc"),
           os.path.join(ROOT, "tests", "c", "bounds_check.cpp"), "-o", exe]
    if debug:
        cmd.insert(1, "-DGCL_DEBUG_BOUNDS")
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert ("debug build" if debug else "release build") in r.stdout
