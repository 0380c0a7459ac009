"""Compile liblora.so in-tree for sm_103a (nvcc, no cmake)."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SO = os.path.join(PKG, "liblora.so")
MAIN = os.path.join(PKG, "csrc", "lora_api.cu")
RUNTIME = os.path.join(PKG, "csrc", "runtime.cpp")   # host-only: adapter cache, scheduler


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build_cmd(extra=()) -> list[str]:
    return [nvcc(), "-O3", "-shared", "-Xcompiler", "-fPIC", "-std=c++17",
            "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-I", os.path.join(ROOT, "include"), *extra, "-o", SO, MAIN, RUNTIME]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(PKG, "csrc", "*")) +
                  glob.glob(os.path.join(ROOT, "include", "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(SO):
        return False
    t = os.path.getmtime(SO)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False) -> str:
    if force or not up_to_date():
        subprocess.check_call(build_cmd())
    return SO
