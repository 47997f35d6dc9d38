"""The operand split of the tensor-core span products, checked on the host (no GPU):
tests/split_harness.cu calls the library's own fa_split_bf16x3 (the function the operand
image kernel applies to every span entry) on floats over the whole fp32 range and checks
that the three bf16 parts sum to the value exactly, and that the six part products the MMAs
form stay within 2^-21 of the exact product."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bf16_three_part_split_is_exact(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "split_harness")
    subprocess.check_call([nvcc, "-std=c++17", "-O2", "-o", exe, os.path.join(HERE, "split_harness.cu")])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok ") and int(r.stdout.split()[1]) > 300000, r.stdout
