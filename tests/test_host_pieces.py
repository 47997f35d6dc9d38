"""The piece schedule of the host-input step, checked on the host (no GPU):
tests/pieces_harness.cu calls the library's own fa_host_pieces (the bounds
fa_constrained_step_host copies and reweights by) for every batch size up to 20000 positions
and a few large ones, and checks that the pieces tile the batch in order, number at most
eight, start with a thirty-second of the batch and grow by at most 1.4 times."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_host_input_pieces_tile_the_batch(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "pieces_harness")
    subprocess.check_call([nvcc, "-std=c++17", "-O2", "-o", exe, os.path.join(HERE, "pieces_harness.cu")])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok 20006", r.stdout
