"""The two standalone probes behind the forward kernel's design choices (tests/probes/), built with
nvcc for sm_103a and run on the GPU: tensor-copy issue cost, and shared-memory load patterns.  The
checks are loose plausibility bounds (the probes exist to measure, not to enforce a number): every
copy lands, issuing a copy costs tens of cycles or more, and a quarter-wise distinct 16-byte load
costs more SM cycles than a quarter-uniform one."""
import os
import re
import subprocess

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "probes")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build_and_run(name, tmp_path):
    exe = str(tmp_path / name)
    subprocess.run(["nvcc", *ARCH, "-O3", "-std=c++17", "-o", exe, os.path.join(HERE, name + ".cu")], check=True,
                   capture_output=True, timeout=300)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip().endswith("done"), res.stdout
    return res.stdout


def test_tma_issue_probe(tmp_path):
    out = build_and_run("tma_issue_probe", tmp_path)
    rows = re.findall(r"issue\s+(\d+) cyc \(\s*(\d+) per copy per issuer\)\s+all landed\s+(-?\d+) cyc\s+timeouts (\d+)",
                      out)
    assert len(rows) == 8, out
    for issue, per_copy, landed, timeouts in rows:
        assert int(timeouts) == 0 and int(landed) > 0, out
        assert 10 <= int(per_copy) <= 100000, out


def test_lds_pattern_probe(tmp_path):
    out = build_and_run("lds_pattern_probe", tmp_path)
    cyc = {m.group(1).strip(): float(m.group(2)) for m in re.finditer(r"^(.*?)\s+([\d.]+) cycles per", out, re.M)}
    assert len(cyc) == 5, out
    assert cyc["LDS.128 row per quarter (g = lane%4)"] > cyc["LDS.128 quarter-uniform (g = lane/8)"], out
