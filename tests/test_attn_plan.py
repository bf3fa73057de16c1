"""Host check of the attention kernel's work division: the plan and item
iterator the kernel's roles share (attn_plan.cuh) compiled for the host with
g++ and walked for every CTA over random batches and grid sizes (no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "eagle_speculative_decoding_attn_gb300", "csrc")


def test_every_tile_once_and_splits_consistent(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "plan_check")
    subprocess.run([gxx, "-O2", "-std=c++17", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "plan_check.cpp"), "-o", exe], check=True)
    res = subprocess.run([exe, "600"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.startswith("OK"), res.stdout + res.stderr
