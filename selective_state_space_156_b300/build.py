"""Builds libssm_b300.so in-tree from csrc/*.cu with nvcc for sm_103a.

Usage: python -m selective_state_space_156_b300.build [--force] [-j N]
Each translation unit is compiled in parallel; the shared library is relinked only when a
source, header or this file is newer than it.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libssm_b300.so")
BUILD_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(ROOT, "include", "ssm_scan.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str) -> tuple:
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(force: bool = False, jobs: int = 0, verbose: bool = False) -> str:
    """Compile every csrc/*.cu and link libssm_b300.so.  Returns the library path."""
    if not force and up_to_date():
        return OUT
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = jobs or min(8, os.cpu_count() or 4)
    objs, logs = [], []
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        for src, obj, rc, log in ex.map(_compile, _sources()):
            logs.append((src, log))
            if rc != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{log}")
            objs.append(obj)
    tmp = OUT + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, OUT)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        for src, log in logs:
            f.write(f"==== {os.path.basename(src)}\n{log}\n")
    if verbose:
        for src, log in logs:
            print(f"==== {os.path.basename(src)}\n{log}")
    return OUT


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-j", type=int, default=0)
    ap.add_argument("-v", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, jobs=args.j, verbose=args.v))
    sys.exit(0)
