"""Compile liblora.so in-tree for sm_103a (nvcc, no cmake): one object per translation
unit, compiled in parallel, then one link."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SO = os.path.join(PKG, "liblora.so")
OBJ_DIR = os.path.join(PKG, "_build")
# the C ABI, the launch code of each kernel family, and the host runtime (adapter cache,
# scheduler; host-only C++)
SOURCES = [os.path.join(PKG, "csrc", f) for f in
           ("lora_api.cu", "launch_ring.cu", "launch_tile.cu", "launch_cluster.cu", "runtime.cpp")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _obj(src: str) -> str:
    return os.path.join(OBJ_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")


def compile_cmds(extra=()) -> list[list[str]]:
    """One nvcc -c per translation unit (independent: run them in parallel)."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    return [[nvcc(), "-O3", "-Xcompiler", "-fPIC", "-std=c++17",
             "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
             "-I", os.path.join(ROOT, "include"), *extra, "-c", "-o", _obj(s), s] for s in SOURCES]


def link_cmd() -> list[str]:
    return [nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", SO,
            *[_obj(s) for s in SOURCES]]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(PKG, "csrc", "*")) +
                  glob.glob(os.path.join(ROOT, "include", "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(SO):
        return False
    t = os.path.getmtime(SO)
    return all(os.path.getmtime(s) <= t for s in sources())


def run_parallel(cmds: list[list[str]]) -> None:
    procs = [subprocess.Popen(c) for c in cmds]
    bad = [c for c, p in zip(cmds, procs) if p.wait() != 0]
    if bad:
        raise RuntimeError(f"build failed: {bad}")


def build(force: bool = False) -> str:
    if force or not up_to_date():
        run_parallel(compile_cmds())
        subprocess.check_call(link_cmd())
    return SO
