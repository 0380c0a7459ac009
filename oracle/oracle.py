"""ORACLE — test infrastructure only (tests, the package smoke check and the
bench's CPU-baseline leg).  Python face of the fp64 C oracle plus the integer
parts of the method (grouping tokens by adapter, walking the page table).

The GPU product path never imports this module.

Sources, by page and section:
  * "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels
    work": SGMV sorts or groups tokens so each contiguous segment shares an
    adapter; engines precompute per step an index mapping tokens to adapters.
  * "S-LoRA: Serving Thousands of Concurrent Adapters in 2026", "The Three Core
    Pillars": the fused kernel groups token slices by target adapter id.
  * "S-LoRA: Serving Thousands of Concurrent LoRA Adapters": adapters are gathered
    from non-contiguous pages of the unified pool.
Readings (the pages fix no order): groups are listed by ascending adapter id;
inside a group tokens keep their batch order; base-only tokens (-1) are in no group.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(_HERE, "liboracle.so")
SRC = os.path.join(_HERE, "lora_oracle.c")

ERRORS = {1: "adapter id out of range", 2: "rank out of range",
          3: "page-table block out of range", 4: "page id out of range"}


def build_cmd() -> list[str]:
    return ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
            "-o", SO, SRC]


def build() -> None:
    subprocess.check_call(build_cmd())


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(SO) or os.path.getmtime(SO) < os.path.getmtime(SRC):
            build()
        lib = ctypes.CDLL(SO)
        p = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_lora_delta.argtypes = [p, i64, i32, p, i64, p, p, p, i32, i32, i32, i32, p,
                                          i32, i32, p, i64, p, i64, p, i32, p, i64, p, p]
        lib.oracle_lora_delta.restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def lora_delta(pool: np.ndarray, pt: np.ndarray, pt_off: np.ndarray, ranks: np.ndarray,
               scales: np.ndarray, num_layers: int, num_proj: int, layer: int, proj: int,
               x: np.ndarray, y0: np.ndarray, token_adapter: np.ndarray,
               want_t: bool = False, proj_dims=None):
    """y_ref = y0 + delta for one (layer, proj) problem, in float64.

    pool: uint16 [num_pages, h] raw bf16 bits;  x: uint16 [T, d_in] raw bf16 bits;
    y0: float64 [T, d_out] (bf16 inputs widened by the caller); token_adapter int32 [T].
    proj_dims: (d_in, d_out) of every projection, or None for h x h everywhere.
    Returns (y_ref [T, d_out] float64, t [T, r_max] float64 or None, multiply-adds).
    """
    pool = np.ascontiguousarray(pool, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    y0 = np.ascontiguousarray(y0, dtype=np.float64)
    pt = np.ascontiguousarray(pt, dtype=np.int32)
    pt_off = np.ascontiguousarray(pt_off, dtype=np.int64)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    ids = np.ascontiguousarray(token_adapter, dtype=np.int32)
    T = ids.size
    h = pool.shape[1]
    dims = None if proj_dims is None else np.ascontiguousarray(proj_dims, dtype=np.int32).reshape(-1)
    d_in, d_out = (h, h) if dims is None else (int(dims[2 * proj]), int(dims[2 * proj + 1]))
    assert x.shape == (T, d_in) and y0.shape == (T, d_out)
    r_max = int(ranks.max()) if ranks.size else 1
    y = np.empty((T, d_out), dtype=np.float64)
    t = np.empty((T, r_max), dtype=np.float64) if want_t else None
    madds = ctypes.c_int64(0)
    err = _load().oracle_lora_delta(
        pool.ctypes.data, pool.shape[0], h, pt.ctypes.data, pt.size, pt_off.ctypes.data,
        ranks.ctypes.data, scales.ctypes.data, ranks.size, num_layers, num_proj, r_max,
        dims.ctypes.data if dims is not None else None,
        layer, proj, x.ctypes.data, d_in, y0.ctypes.data, d_out, ids.ctypes.data, T,
        y.ctypes.data, d_out, t.ctypes.data if t is not None else None, ctypes.byref(madds))
    if err:
        raise OracleError(ERRORS.get(err, str(err)))
    return y, t, int(madds.value)


def lora_expand(pool: np.ndarray, pt: np.ndarray, pt_off: np.ndarray, ranks: np.ndarray,
                scales: np.ndarray, num_layers: int, num_proj: int, layer: int, proj: int,
                t: np.ndarray, y0: np.ndarray, token_adapter: np.ndarray, proj_dims=None) -> np.ndarray:
    """The expand step alone, in float64: y[i, n] = y0[i, n] + s_a * sum_j t[i, j] B_a[n, j]
    for every token i with adapter a >= 0 (base-only rows are y0 unchanged).

    "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work":
    expand y_i += gamma B_{a(i)} v_i after the shrink v_i = A_{a(i)} x_i; "What the engine
    does each step": the two are separate steps with v between them.  t is the unscaled
    shrink (lora_delta's t, or a sum of partial t); B column j of (layer, proj) is read from
    its pages by walking the page table (page q of column j at the B block's entry q r + j).
    pool: uint16 [num_pages, h] bf16 bits; t: float64 [T, >= r_max]; y0: float64 [T, d_out]."""
    pool = np.asarray(pool, dtype=np.uint16)
    h = pool.shape[1]
    U, pre, pv_in, pv_out = block_units(num_proj, h, proj_dims)
    d_out = h if proj_dims is None else int(np.asarray(proj_dims).reshape(-1, 2)[proj][1])
    y = np.array(y0, dtype=np.float64, copy=True)
    ids = np.asarray(token_adapter, dtype=np.int64)
    for i in range(ids.size):
        a = int(ids[i])
        if a < 0:
            continue
        r = int(ranks[a])
        b0 = int(pt_off[a]) + r * (layer * U + pre[proj] + pv_in[proj])   # first B-block entry
        acc = np.zeros(d_out, dtype=np.float64)
        for j in range(r):
            col = np.concatenate([_bf16_to_f64(pool[int(pt[b0 + q * r + j])]) for q in range(pv_out[proj])])
            acc += float(t[i, j]) * col[:d_out]
        y[i] += float(scales[a]) * acc
    return y


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) widened exactly to float64."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def group_tokens(token_adapter: np.ndarray):
    """Stable grouping of the adapted tokens by adapter id.

    Returns perm (token indices, ascending adapter id, batch order inside a group),
    grp_start [G+1] (offsets into perm) and grp_adapter [G]."""
    ids = np.asarray(token_adapter, dtype=np.int64)
    adapted = np.nonzero(ids >= 0)[0]
    perm = adapted[np.argsort(ids[adapted], kind="stable")]
    sid = ids[perm]
    if perm.size == 0:
        return perm.astype(np.int32), np.zeros(1, np.int32), np.zeros(0, np.int32)
    starts = np.concatenate([[0], np.nonzero(np.diff(sid))[0] + 1])
    grp_start = np.concatenate([starts, [perm.size]]).astype(np.int32)
    return perm.astype(np.int32), grp_start, sid[starts].astype(np.int32)


def block_units(num_proj: int, h: int, proj_dims=None):
    """Page-table layout in units of an adapter's rank: (units of one layer, units before
    projection p, pages per A row of p, pages per B column of p) for every p; a vector of
    length d takes ceil(d / h) pages."""
    def pv(d):
        return -(-int(d) // h)
    dims = [(h, h)] * num_proj if proj_dims is None else [tuple(map(int, d)) for d in
                                                         np.asarray(proj_dims).reshape(-1, 2)]
    pre, acc = [], 0
    for d_in, d_out in dims:
        pre.append(acc)
        acc += pv(d_in) + pv(d_out)
    return acc, pre, [pv(d[0]) for d in dims], [pv(d[1]) for d in dims]


def page_list(pt: np.ndarray, pt_off: np.ndarray, ranks: np.ndarray, num_proj: int,
              layer: int, proj: int, grp_adapter: np.ndarray, h: int = 0, proj_dims=None) -> np.ndarray:
    """Gathered page ids of one problem, group by group: the A-row pages then the
    B-column pages of each group's adapter (page-table walk), each block page block by
    page block (page kb of every row, then page kb + 1)."""
    U, pre, pv_in, pv_out = block_units(num_proj, max(h, 1), proj_dims)
    out = []
    for a in np.asarray(grp_adapter, dtype=np.int64):
        r = int(ranks[a])
        base = int(pt_off[a]) + r * (layer * U + pre[proj])
        out.append(np.asarray(pt[base:base + r * (pv_in[proj] + pv_out[proj])], dtype=np.int32))
    return np.concatenate(out) if out else np.zeros(0, np.int32)

