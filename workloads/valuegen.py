"""ctypes loaders for the seeded value generator (definition in valuegen.h).

The host routine fills numpy uint16 arrays (raw bf16 bits); the device routine
fills device buffers given as integer pointers.  Both give identical bits for
the same (seed, row key, element index).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(_HERE, "libvaluegen_host.so")
DEV_SO = os.path.join(_HERE, "libvaluegen_dev.so")

DIST_UNIFORM = 0
DIST_NORMAL = 1


def uniform_param(bound: float) -> float:
    """Multiplier turning the odd integer m in (-2^24, 2^24) into U(-bound, bound)."""
    return bound * 2.0 ** -24


def normal_param(sigma: float) -> float:
    """Multiplier turning the centred Irwin-Hall(4) sum of 16-bit fields into sd `sigma`."""
    return sigma / math.sqrt((2.0 ** 32 - 1.0) / 3.0)


def host_build_cmd() -> list[str]:
    return ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
            "-o", HOST_SO, os.path.join(_HERE, "valuegen_host.c")]


def dev_build_cmd(nvcc: str = "nvcc") -> list[str]:
    return [nvcc, "-O3", "-shared", "-Xcompiler", "-fPIC", "-fmad=false",
            "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-o", DEV_SO, os.path.join(_HERE, "valuegen_dev.cu")]


def build(dev: bool = True) -> None:
    """Compile the host (gcc) and, if requested, the device (nvcc) generator."""
    procs = [subprocess.Popen(host_build_cmd())]
    if dev:
        procs.append(subprocess.Popen(dev_build_cmd()))
    for p in procs:
        if p.wait() != 0:
            raise RuntimeError(f"value generator build failed: {p.args}")


_host = None
_dev = None


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(HOST_SO):
            subprocess.check_call(host_build_cmd())
        lib = ctypes.CDLL(HOST_SO)
        lib.wl_fill_rows_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                          ctypes.c_int, ctypes.c_double]
        lib.wl_fill_rows_host.restype = None
        _host = lib
    return _host


def _load_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_SO):
            raise RuntimeError(f"{DEV_SO} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(DEV_SO)
        lib.wl_fill_rows_dev.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                         ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
        lib.wl_fill_rows_dev.restype = ctypes.c_int
        _dev = lib
    return _dev


def fill_rows_host(dst: np.ndarray, row_ids: np.ndarray, keys: np.ndarray, seed: int,
                   dist: int, param: float) -> None:
    """Fill rows of the C-contiguous uint16 matrix `dst` [rows, h] in place."""
    assert dst.dtype == np.uint16 and dst.ndim == 2 and dst.flags.c_contiguous
    row_ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    keys = np.ascontiguousarray(keys, dtype=np.uint64)
    assert row_ids.shape == keys.shape
    if row_ids.size == 0:
        return
    assert row_ids.min() >= 0 and row_ids.max() < dst.shape[0]
    _load_host().wl_fill_rows_host(dst.ctypes.data, dst.shape[1], row_ids.ctypes.data,
                                   keys.ctypes.data, row_ids.size, seed & (2 ** 64 - 1),
                                   dist, param)


def fill_rows_dev(dst_ptr: int, h: int, row_ids_ptr: int, keys_ptr: int, n: int, seed: int,
                  dist: int, param: float, stream: int) -> None:
    """Device fill: all pointers are device addresses (row_ids int64, keys uint64)."""
    err = _load_dev().wl_fill_rows_dev(dst_ptr, h, row_ids_ptr, keys_ptr, n,
                                       seed & (2 ** 64 - 1), dist, param, stream)
    if err != 0:
        raise RuntimeError(f"wl_fill_rows_dev failed with CUDA error {err}")


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to float64 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
