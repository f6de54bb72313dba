"""Host-side checks of the forward scan's plans (no GPU): tests/plan/plan_check.cpp includes the
library's plan header (csrc/scan_plan.h), builds with the host compiler, and walks the plans the
library would launch, as the kernel decodes them, for the balanced form and for both passes of the
split form (full and tail splits) on several SM counts: every channel, chunk and carry slot is
scanned exactly once."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = "/usr/local/cuda/include"


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_plans_cover_every_channel_and_chunk_once(tmp_path):
    exe = tmp_path / "plan_check"
    cmd = ["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "selective_state_space_155_b300", "csrc"), "-I", CUDA_INCLUDE,
           "-o", str(exe), os.path.join(ROOT, "tests", "plan", "plan_check.cpp")]
    build = subprocess.run(cmd, capture_output=True, text=True)
    assert build.returncode == 0, build.stdout + build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("all ok"), run.stdout + run.stderr
    # the long workload takes the tail split, the mid workload stays whole
    assert "split b1 d5120 L65536 on 148 SMs: 32 segments" in run.stdout
    assert "split b8 d1536 L2048 on 148 SMs: unsplit" in run.stdout
