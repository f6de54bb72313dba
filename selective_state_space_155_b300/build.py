"""Build the in-tree CUDA library libssm_scan.so for sm_103a (B300).

    python -m selective_state_space_155_b300.build [--force] [--verbose]

nvcc cross-compiles without a GPU.  The CUDA runtime is linked statically, so the
library loads on machines without a driver (calls then fail with SSM_ERR_LAUNCH).
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libssm_scan.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--use_fast_math", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-shared", "-cudart", "static"]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + [
        os.path.join(INCLUDE, "ssm_scan.h"), os.path.abspath(__file__)]


def _digest() -> str:
    """Hash of every build input's bytes and of the compiler command: what the library was built from."""
    import hashlib
    h = hashlib.sha256(" ".join(ARCH + NVCC_FLAGS).encode())
    for p in _inputs():
        h.update(os.path.relpath(p, ROOT).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


STAMP = LIB + ".sha256"


def up_to_date() -> bool:
    """The in-tree library exists and was built from the current sources (by content, not mtime:
    a copied tree can carry a stale library with a newer timestamp)."""
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == _digest()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-o", LIB, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed ({res.returncode}): {' '.join(cmd)}")
    if verbose:
        sys.stdout.write(res.stdout + res.stderr)
    with open(STAMP, "w") as f:
        f.write(_digest() + "\n")
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
