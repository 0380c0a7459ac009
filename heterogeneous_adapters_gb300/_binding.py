"""ctypes binding of liblora.so: the same names as include/lora.h, argument
marshalling only.  Every step of the path runs in the library's CUDA kernels;
there is no Python or CPU fallback: if the library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(_PKG, "liblora.so")

(LORA_OK, LORA_EINVAL, LORA_EALIGN, LORA_EWORKSPACE, LORA_ETOOBIG, LORA_ECUDA, LORA_EDEVICE,
 LORA_ENOSPACE) = range(8)
LORA_UNIT_ABSENT, LORA_UNIT_LOADING, LORA_UNIT_READY = range(3)
DERR = {0x1: "adapter", 0x2: "rank", 0x4: "page-table block", 0x8: "page", 0x10: "segment",
        0x20: "timeout"}
LORA_MAX_PROBLEMS_PER_LAUNCH = 256
LORA_MAX_SEGMENTS = 16384
LORA_MAX_RANK = 256
LORA_NOALLOC_MAX_TOKENS = 4096
LORA_STAGE_MAX_RUNS = 64

EXPORTED = ["lora_pool_create", "lora_pool_destroy", "lora_pool_set_tuning", "lora_pool_get_tuning",
            "lora_workspace_size", "lora_workspace_init",
            "lora_segment", "lora_workspace_view", "lora_bgmv", "lora_sgmv", "lora_apply_mixed",
            "lora_delta_grouped", "lora_debug_page_list", "lora_debug_delta_with_t", "lora_debug_wait_limit",
            "lora_stage_pages", "lora_bgmv_noalloc", "lora_get_device_error", "lora_shrink",
            "lora_expand", "lora_stage_pages_ce",
            "lora_last_cuda_error", "lora_status_string",
            # host runtime (include/lora_runtime.h)
            "lora_cache_create", "lora_cache_destroy", "lora_cache_acquire", "lora_cache_loaded",
            "lora_cache_release", "lora_cache_query", "lora_cache_stats", "lora_sched_create",
            "lora_sched_destroy", "lora_sched_enqueue", "lora_sched_pick", "lora_sched_pending"]


class lora_pool_desc(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("num_pages", ctypes.c_int64), ("h", ctypes.c_int32),
                ("num_adapters", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_proj", ctypes.c_int32), ("r_max", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("page_table_len", ctypes.c_int64), ("adapter_pt_off", ctypes.c_void_p),
                ("ranks", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("proj_dims", ctypes.c_void_p)]


class lora_tuning(ctypes.Structure):
    _fields_ = [("ring_rows_per_stage", ctypes.c_int32), ("split_max_problems", ctypes.c_int32),
                ("mma_min_rows", ctypes.c_int32), ("mma_y_stages", ctypes.c_int32),
                ("fused_ring_speed", ctypes.c_float), ("reserved", ctypes.c_int32 * 3)]


# lora_tuning fields and the value that keeps a field's default
TUNING_KEEP = {"ring_rows_per_stage": 0, "split_max_problems": -1, "mma_min_rows": -1,
               "mma_y_stages": 0, "fused_ring_speed": 0.0}


class lora_problem(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("ldx", ctypes.c_int64),
                ("ldy", ctypes.c_int64), ("layer", ctypes.c_int32), ("proj", ctypes.c_int32)]


class lora_ws_view(ctypes.Structure):
    _fields_ = [("error_word", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("grp_start", ctypes.c_void_p),
                ("grp_adapter", ctypes.c_void_p)]


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {status_string(status)}"
        if status == LORA_ECUDA:
            msg += f" (cudaError {lib().lora_last_cuda_error()})"
        super().__init__(msg + (f" {detail}" if detail else ""))


_lib = None


def lib():
    """Load liblora.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            raise RuntimeError(f"{SO} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(SO)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "lora_pool_create": [ctypes.POINTER(p), ctypes.POINTER(lora_pool_desc)],
            "lora_pool_destroy": [p],
            "lora_pool_set_tuning": [p, ctypes.POINTER(lora_tuning)],
            "lora_pool_get_tuning": [p, ctypes.POINTER(lora_tuning)],
            "lora_workspace_size": [p, i32, i32, ctypes.POINTER(sz)],
            "lora_workspace_init": [p, sz, p],
            "lora_segment": [p, p, p, i32, p, i32, i32, p, sz, p],
            "lora_workspace_view": [p, p, sz, i32, i32, ctypes.POINTER(lora_ws_view)],
            "lora_bgmv": [p, p, i32, p, i32, p, sz, p],
            "lora_sgmv": [p, p, i32, p, p, i32, i32, p, sz, p],
            "lora_apply_mixed": [p, p, i32, p, p, i32, p, i32, i32, p, sz, p],
            "lora_delta_grouped": [p, p, i32, i32, i32, p, sz, p],
            "lora_debug_page_list": [p, p, sz, i32, i32, p, i64, p, p],
            "lora_debug_delta_with_t": [p, ctypes.POINTER(lora_problem), p, sz, p, p],
            "lora_debug_wait_limit": [p, sz, ctypes.c_uint64, p, p],
            "lora_stage_pages": [p, p, p, i32, p, p, p, i64, p],
            "lora_stage_pages_ce": [p, p, p, sz, p, i32, p, p, p, i64, p, p],
            "lora_bgmv_noalloc": [p, p, i32, p, i32, p, p],
            "lora_shrink": [p, p, i32, p, i32, p, sz, p, p],
            "lora_expand": [p, p, i32, i32, p, sz, p, p],
            "lora_get_device_error": [p, p, ctypes.POINTER(ctypes.c_uint32)],
            "lora_last_cuda_error": [],
            "lora_status_string": [ctypes.c_int],
            "lora_cache_create": [ctypes.POINTER(p), p, i64, p, i32],
            "lora_cache_destroy": [p],
            "lora_cache_acquire": [p, i32, ctypes.POINTER(i32), p, i64, p, i32, ctypes.POINTER(i32)],
            "lora_cache_loaded": [p, i32],
            "lora_cache_release": [p, i32],
            "lora_cache_query": [p, i32, ctypes.POINTER(i32), ctypes.POINTER(i32), p, i64],
            "lora_cache_stats": [p] + [ctypes.POINTER(i64)] * 4,
            "lora_sched_create": [ctypes.POINTER(p), p],
            "lora_sched_destroy": [p],
            "lora_sched_enqueue": [p, i64, i32, i32],
            "lora_sched_pick": [p, i32, i32, p, p, p, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                ctypes.POINTER(i32)],
            "lora_sched_pending": [p, ctypes.POINTER(i64)],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.lora_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().lora_status_string(st).decode()


def _check(st: int, where: str):
    if st != LORA_OK:
        raise LoraError(st, where)


def _ptr(t) -> int | None:
    """Device or host address of a tensor / integer (None stays NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def problems_array(problems):
    """problems: iterable of (x, y, ldx, ldy, layer, proj) with x/y tensors or addresses."""
    problems = list(problems)
    arr = (lora_problem * max(1, len(problems)))()
    for i, (x, y, ldx, ldy, layer, proj) in enumerate(problems):
        arr[i] = lora_problem(_ptr(x), _ptr(y), ldx, ldy, layer, proj)
    return arr, len(problems)


class Pool:
    """Handle of a lora_pool (host metadata only; device arrays stay the caller's)."""

    def __init__(self, pages, num_pages, h, page_table, page_table_len, pt_off, ranks, scales,
                 num_adapters, num_layers, num_proj, r_max, proj_dims=None):
        """proj_dims: (d_in, d_out) of every projection (copied by the library), or None
        for h x h projections."""
        import numpy as np
        dims = None if proj_dims is None else np.ascontiguousarray(proj_dims, np.int32).reshape(-1)
        d = lora_pool_desc(_ptr(pages), num_pages, h, num_adapters, num_layers, num_proj, r_max, 0,
                           _ptr(page_table), page_table_len, _ptr(pt_off), _ptr(ranks), _ptr(scales),
                           dims.ctypes.data if dims is not None else None)
        self._h = ctypes.c_void_p()
        _check(lib().lora_pool_create(ctypes.byref(self._h), ctypes.byref(d)), "lora_pool_create")
        self.h = h
        self.r_max = r_max

    @property
    def handle(self):
        return self._h

    def set_tuning(self, **fields):
        """Launch tuning (lora_pool_set_tuning): the named fields, every other one at its
        default; no fields restores all the defaults."""
        unknown = set(fields) - set(TUNING_KEEP)
        if unknown:
            raise ValueError(f"unknown tuning fields {sorted(unknown)}")
        t = lora_tuning(**{k: fields.get(k, v) for k, v in TUNING_KEEP.items()})
        _check(lib().lora_pool_set_tuning(self._h, ctypes.byref(t)), "lora_pool_set_tuning")

    def get_tuning(self) -> dict:
        t = lora_tuning()
        _check(lib().lora_pool_get_tuning(self._h, ctypes.byref(t)), "lora_pool_get_tuning")
        return {k: getattr(t, k) for k in TUNING_KEEP}

    def close(self):
        if self._h:
            lib().lora_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def workspace_size(pool: Pool, max_tokens: int, max_segments: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().lora_workspace_size(pool.handle, max_tokens, max_segments, ctypes.byref(n)),
           "lora_workspace_size")
    return n.value


def workspace_init(ws, ws_bytes: int, stream: int):
    _check(lib().lora_workspace_init(_ptr(ws), ws_bytes, stream), "lora_workspace_init")


def segment(pool, seg_start, seg_adapter, S, dec_adapter, Td, T, ws, ws_bytes, stream):
    _check(lib().lora_segment(pool.handle, _ptr(seg_start), _ptr(seg_adapter), S,
                              _ptr(dec_adapter), Td, T, _ptr(ws), ws_bytes, stream), "lora_segment")


def workspace_view(pool, ws, ws_bytes, max_tokens, max_segments) -> lora_ws_view:
    v = lora_ws_view()
    _check(lib().lora_workspace_view(pool.handle, _ptr(ws), ws_bytes, max_tokens, max_segments,
                                     ctypes.byref(v)), "lora_workspace_view")
    return v


def bgmv(pool, problems, token_adapter, T, ws, ws_bytes, stream):
    arr, n = problems_array(problems)
    _check(lib().lora_bgmv(pool.handle, arr, n, _ptr(token_adapter), T, _ptr(ws), ws_bytes, stream),
           "lora_bgmv")


def sgmv(pool, problems, seg_start, seg_adapter, S, T, ws, ws_bytes, stream):
    arr, n = problems_array(problems)
    _check(lib().lora_sgmv(pool.handle, arr, n, _ptr(seg_start), _ptr(seg_adapter), S, T, _ptr(ws),
                           ws_bytes, stream), "lora_sgmv")


def apply_mixed(pool, problems, seg_start, seg_adapter, S, dec_adapter, Td, T, ws, ws_bytes, stream):
    arr, n = problems_array(problems)
    _check(lib().lora_apply_mixed(pool.handle, arr, n, _ptr(seg_start), _ptr(seg_adapter), S,
                                  _ptr(dec_adapter), Td, T, _ptr(ws), ws_bytes, stream),
           "lora_apply_mixed")


def delta_grouped(pool, problems, T, S, ws, ws_bytes, stream):
    arr, n = problems_array(problems)
    _check(lib().lora_delta_grouped(pool.handle, arr, n, T, S, _ptr(ws), ws_bytes, stream),
           "lora_delta_grouped")


def debug_page_list(pool, ws, ws_bytes, layer, proj, out_pages, cap, count_dev, stream):
    _check(lib().lora_debug_page_list(pool.handle, _ptr(ws), ws_bytes, layer, proj, _ptr(out_pages),
                                      cap, _ptr(count_dev), stream), "lora_debug_page_list")


def debug_delta_with_t(pool, problem, ws, ws_bytes, t_out, stream):
    arr, _ = problems_array([problem])
    _check(lib().lora_debug_delta_with_t(pool.handle, arr, _ptr(ws), ws_bytes, _ptr(t_out), stream),
           "lora_debug_delta_with_t")


def debug_wait_limit(ws, ws_bytes, limit_ns, elapsed_ns, stream):
    """elapsed_ns: device uint64 (int64 tensor of one element) or None."""
    _check(lib().lora_debug_wait_limit(_ptr(ws), ws_bytes, limit_ns, _ptr(elapsed_ns), stream),
           "lora_debug_wait_limit")


def stage_pages(pool, host_rows, dst_pages, npages, page_table, upd_index, upd_page, nupd, stream):
    """host_rows, dst_pages, upd_index, upd_page: pinned host tensors (or addresses)."""
    _check(lib().lora_stage_pages(pool.handle, _ptr(host_rows), _ptr(dst_pages), npages,
                                  _ptr(page_table), _ptr(upd_index), _ptr(upd_page), nupd, stream),
           "lora_stage_pages")


def stage_pages_ce(pool, host_rows, staging, staging_bytes, dst_pages, npages, page_table, upd_index, upd_page,
                   nupd, stream, copied_event=None):
    """Staging through the copy engines: each run of consecutive destination pages copied
    straight into the pool (at most LORA_STAGE_MAX_RUNS runs), else host rows -> device
    staging buffer (one copy) -> pool pages (one kernel); then the page-table rewrite.
    host_rows, dst_pages, upd_index, upd_page: pinned host tensors; staging: a device buffer of
    npages * 2h bytes, or None when the pages form at most LORA_STAGE_MAX_RUNS runs;
    copied_event: a torch.cuda.Event (or raw handle) recorded right after the copies."""
    ev = None
    if copied_event is not None:
        ev = copied_event.cuda_event if hasattr(copied_event, "cuda_event") else copied_event
    _check(lib().lora_stage_pages_ce(pool.handle, _ptr(host_rows), _ptr(staging), staging_bytes,
                                     _ptr(dst_pages), npages, _ptr(page_table), _ptr(upd_index),
                                     _ptr(upd_page), nupd, ev, stream), "lora_stage_pages_ce")


def bgmv_noalloc(pool, problems, token_adapter, T, error_bits, stream):
    """BGMV with the library's own fixed scratch (no caller workspace, no allocation)."""
    arr, n = problems_array(problems)
    _check(lib().lora_bgmv_noalloc(pool.handle, arr, n, _ptr(token_adapter), T, _ptr(error_bits),
                                   stream), "lora_bgmv_noalloc")


def shrink(pool, problems, token_adapter, T, ws, ws_bytes, t, stream):
    """t[p][row][j] = s * x_p[row] . A_j (fp32 [nprob][T][r_max]); groups the batch into ws."""
    arr, n = problems_array(problems)
    _check(lib().lora_shrink(pool.handle, arr, n, _ptr(token_adapter), T, _ptr(ws), ws_bytes, _ptr(t),
                             stream), "lora_shrink")


def expand(pool, problems, T, ws, ws_bytes, t, stream):
    """y_p[row] += t[p][row] . B^T with the grouping lora_shrink left in ws."""
    arr, n = problems_array(problems)
    _check(lib().lora_expand(pool.handle, arr, n, T, _ptr(ws), ws_bytes, _ptr(t), stream), "lora_expand")


def get_device_error(ws, stream) -> int:
    """Synchronises the stream; returns and clears the device error bits (no raise)."""
    bits = ctypes.c_uint32()
    st = lib().lora_get_device_error(_ptr(ws), stream, ctypes.byref(bits))
    if st not in (LORA_OK, LORA_EDEVICE):
        raise LoraError(st, "lora_get_device_error")
    return bits.value


# ----------------------------------------------------------------------------- host runtime

def _np_ptr(a):
    return a.ctypes.data if a is not None and a.size else None


class AdapterCache:
    """lora_cache_*: LRU residency of units (adapters or adapter slices) in pool pages."""

    def __init__(self, managed_pages, unit_pages):
        import numpy as np
        self._np = np
        self.managed = np.ascontiguousarray(managed_pages, np.int32)
        self.unit_pages = np.ascontiguousarray(unit_pages, np.int32)
        h = ctypes.c_void_p()
        _check(lib().lora_cache_create(ctypes.byref(h), _np_ptr(self.managed), self.managed.size,
                                       _np_ptr(self.unit_pages), self.unit_pages.size), "lora_cache_create")
        self.handle = h

    def _unit_pages(self, u: int) -> int:
        # out-of-range units go to the library, which rejects them
        return int(self.unit_pages[u]) if 0 <= u < self.unit_pages.size else 1

    def acquire(self, u: int, evicted_cap: int = 64):
        """(loaded, pages or None, evicted units); raises LoraError (LORA_ENOSPACE) when full."""
        np = self._np
        pages = np.empty(self._unit_pages(u), np.int32)
        ev = np.empty(evicted_cap, np.int32)
        loaded, n_ev = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().lora_cache_acquire(self.handle, u, ctypes.byref(loaded), pages.ctypes.data, pages.size,
                                        ev.ctypes.data, evicted_cap, ctypes.byref(n_ev)), "lora_cache_acquire")
        return bool(loaded.value), (pages if loaded.value else None), ev[:min(n_ev.value, evicted_cap)].copy()

    def try_acquire(self, u: int):
        """acquire, or None when no pages can be freed."""
        try:
            return self.acquire(u)
        except LoraError as e:
            if e.status == LORA_ENOSPACE:
                return None
            raise

    def loaded(self, u: int):
        _check(lib().lora_cache_loaded(self.handle, u), "lora_cache_loaded")

    def release(self, u: int):
        _check(lib().lora_cache_release(self.handle, u), "lora_cache_release")

    def query(self, u: int):
        """(state, users, pages of a resident unit)."""
        np = self._np
        st, us = ctypes.c_int32(), ctypes.c_int32()
        pages = np.empty(self._unit_pages(u), np.int32)
        _check(lib().lora_cache_query(self.handle, u, ctypes.byref(st), ctypes.byref(us), pages.ctypes.data,
                                      pages.size), "lora_cache_query")
        return st.value, us.value, (pages if st.value != LORA_UNIT_ABSENT else None)

    def stats(self):
        """dict of hits, misses, evictions, free_pages."""
        v = [ctypes.c_int64() for _ in range(4)]
        _check(lib().lora_cache_stats(self.handle, *[ctypes.byref(x) for x in v]), "lora_cache_stats")
        return dict(zip(("hits", "misses", "evictions", "free_pages"), (x.value for x in v)))

    def close(self):
        if self.handle:
            lib().lora_cache_destroy(self.handle)
            self.handle = None


class Scheduler:
    """lora_sched_*: arrival-ordered request queue and the per-step batch pick."""

    def __init__(self, cache: AdapterCache | None = None):
        h = ctypes.c_void_p()
        _check(lib().lora_sched_create(ctypes.byref(h), cache.handle if cache is not None else None),
               "lora_sched_create")
        self.handle = h
        self.cache = cache

    def enqueue(self, req_id: int, adapter: int, tokens: int = 1):
        _check(lib().lora_sched_enqueue(self.handle, req_id, adapter, tokens), "lora_sched_enqueue")

    def pick(self, max_tokens: int, max_distinct: int, cap: int = 4096):
        """(ids, adapters, tokens) of the batch, numpy arrays in queue order."""
        import numpy as np
        ids = np.empty(cap, np.int64)
        ad = np.empty(cap, np.int32)
        tk = np.empty(cap, np.int32)
        n, nt, nd = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().lora_sched_pick(self.handle, max_tokens, max_distinct, ids.ctypes.data, ad.ctypes.data,
                                     tk.ctypes.data, cap, ctypes.byref(n), ctypes.byref(nt), ctypes.byref(nd)),
               "lora_sched_pick")
        k = n.value
        return ids[:k].copy(), ad[:k].copy(), tk[:k].copy()

    def pending(self) -> int:
        v = ctypes.c_int64()
        _check(lib().lora_sched_pending(self.handle, ctypes.byref(v)), "lora_sched_pending")
        return v.value

    def close(self):
        if self.handle:
            lib().lora_sched_destroy(self.handle)
            self.handle = None
