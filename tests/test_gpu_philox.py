"""The device Philox4x32-10 that draws every sample, pinned to the generator's published
known-answer vectors (tests/golden/philox4x32_10_kat.txt): tests/philox_harness.cu runs the
library's own device function on them on the GPU."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_device_philox_matches_known_answers(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    assert os.path.exists(nvcc), "nvcc is needed to build the harness"
    exe = str(tmp_path / "philox_harness")
    subprocess.check_call([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe,
                           os.path.join(HERE, "philox_harness.cu")])
    r = subprocess.run([exe, os.path.join(HERE, "golden", "philox4x32_10_kat.txt")], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok 3"
