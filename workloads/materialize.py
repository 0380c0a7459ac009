"""Turn a Workload into concrete buffers.

host_inputs()   -> numpy buffers for the CPU oracle: a compact pool holding only the
                   pages the chosen problems read, a page table relabelled onto it
                   (a pure renaming of page ids), and the x / y0 rows.
device_inputs() -> torch CUDA buffers for the GPU path, filled on the device by the
                   same generator (bit-identical values).

No arithmetic of the method lives here: only placement, keys and generator calls.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import valuegen as vg
from .spec import KIND_X, KIND_Y, SIGMA_B, SIGMA_X, SIGMA_Y, Workload, row_key


def a_param(h: int) -> float:
    """A ~ U(-1/sqrt(h), 1/sqrt(h))."""
    return vg.uniform_param(1.0 / np.sqrt(h))


def _page_lookup(pool, pages: np.ndarray):
    """Generator keys and A/B flags of physical pages (all must hold adapter values)."""
    order = np.argsort(pool.page_ids, kind="stable")
    sorted_ids = pool.page_ids[order]
    pos = np.searchsorted(sorted_ids, pages)
    assert np.all(pos < sorted_ids.size) and np.all(sorted_ids[pos] == pages), "page not filled"
    return pool.page_keys[order[pos]], pool.page_ab[order[pos]]


@dataclass
class HostInputs:
    pool: np.ndarray          # uint16 [n_compact, h] (raw bf16 bits)
    pt: np.ndarray            # int32, same length as Workload.pool.pt; unread entries -1
    x: dict                   # (layer, proj) -> uint16 [T, h]
    y0: dict                  # (layer, proj) -> uint16 [T, h]


def needed_entries(wl: Workload, problems, adapters=None) -> np.ndarray:
    pool = wl.pool
    if adapters is None:
        ids = wl.batch.token_adapter()
        adapters = np.unique(ids[(ids >= 0) & (ids < pool.num_adapters)])
    out = []
    for a in adapters:
        for (l, p) in problems:
            for ab in (0, 1):
                out.append(pool.block_entries(int(a), l, p, ab))
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def host_inputs(wl: Workload, problems=None, adapters=None, with_xy: bool = True) -> HostInputs:
    problems = wl.problems if problems is None else problems
    pool = wl.pool
    h = pool.h
    ent = needed_entries(wl, problems, adapters)
    pages = pool.pt[ent].astype(np.int64)
    assert np.all(pages >= 0), "a needed page is not resident"
    uniq, inv = np.unique(pages, return_inverse=True)
    compact = np.zeros((max(uniq.size, 1), h), dtype=np.uint16)
    keys, ab = _page_lookup(pool, uniq)
    rows = np.arange(uniq.size, dtype=np.int64)
    vg.fill_rows_host(compact, rows[ab == 0], keys[ab == 0], wl.seed, vg.DIST_UNIFORM, a_param(h))
    vg.fill_rows_host(compact, rows[ab == 1], keys[ab == 1], wl.seed, vg.DIST_NORMAL,
                      vg.normal_param(SIGMA_B))
    pt = np.full(pool.pt.size, -1, dtype=np.int32)
    pt[ent] = inv.astype(np.int32)
    x, y0 = {}, {}
    if with_xy:
        T = wl.batch.num_tokens
        for (l, p) in problems:
            d_in, d_out = pool.dims(p)
            x[(l, p)] = host_rows(wl, KIND_X, *wl.x_source(l, p), T, width=d_in)
            y0[(l, p)] = host_rows(wl, KIND_Y, l, p, T, width=d_out)
    return HostInputs(compact, pt, x, y0)


def host_rows(wl: Workload, kind: int, l: int, p: int, T: int, rows=None, width=None) -> np.ndarray:
    """x (KIND_X) or y0 (KIND_Y) rows of problem (l, p) as uint16 [len(rows), width]
    (width h by default); element e of a row does not depend on the width."""
    rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, wl.h if width is None else width), dtype=np.uint16)
    sigma = SIGMA_X if kind == KIND_X else SIGMA_Y
    vg.fill_rows_host(out, np.arange(rows.size), row_key(kind, l, p, rows), wl.seed,
                      vg.DIST_NORMAL, vg.normal_param(sigma))
    return out


@dataclass
class DeviceInputs:
    pool: object              # torch bf16 [num_pages, h]
    pt: object                # torch int32
    pt_off: object            # torch int64
    ranks: object             # torch int32
    scales: object            # torch float32
    x: object                 # torch bf16 [nprob, T, max d_in]  (h x h pools: h)
    y: object                 # torch bf16 [nprob, T, max d_out]
    seg_start: object         # torch int32 [S+1]
    seg_adapter: object       # torch int32 [S]
    dec_adapter: object       # torch int32 [Td]
    token_adapter: object     # torch int32 [T]
    problems: list
    x_src: list = None        # problem i reads x[x_src[i]] (its own x unless inputs are shared)


def device_fill_pool(wl: Workload, pool_t, stream: int, nan_dummies: bool = True) -> None:
    import torch
    pool = wl.pool
    if nan_dummies and pool.page_ids.size < pool.num_pages:
        pool_t.fill_(float("nan"))
    dev = pool_t.device
    for ab, dist, param in ((0, vg.DIST_UNIFORM, a_param(pool.h)),
                            (1, vg.DIST_NORMAL, vg.normal_param(SIGMA_B))):
        sel = pool.page_ab == ab
        rows = torch.from_numpy(pool.page_ids[sel].astype(np.int64)).to(dev)
        keys = torch.from_numpy(pool.page_keys[sel].view(np.int64)).to(dev)
        vg.fill_rows_dev(pool_t.data_ptr(), pool.h, rows.data_ptr(), keys.data_ptr(),
                         rows.numel(), wl.seed, dist, param, stream)
        torch.cuda.current_stream(dev).synchronize()
        del rows, keys


def device_fill_rows(wl: Workload, buf, kind: int, problems, stream: int) -> None:
    """Fill buf [nprob, T, h] with the x or y0 rows of the given problems."""
    import torch
    T = buf.shape[1]
    src = [wl.x_source(l, p) if kind == KIND_X else (l, p) for (l, p) in problems]
    keys = np.concatenate([row_key(kind, l, p, np.arange(T)) for (l, p) in src])
    rows = torch.arange(len(problems) * T, dtype=torch.int64, device=buf.device)
    keys_t = torch.from_numpy(keys.view(np.int64)).to(buf.device)
    sigma = SIGMA_X if kind == KIND_X else SIGMA_Y
    vg.fill_rows_dev(buf.data_ptr(), buf.shape[2], rows.data_ptr(), keys_t.data_ptr(), rows.numel(),
                     wl.seed, vg.DIST_NORMAL, vg.normal_param(sigma), stream)
    torch.cuda.current_stream(buf.device).synchronize()


def device_inputs(wl: Workload, problems=None, device="cuda", nan_dummies: bool = True,
                  pool_t=None) -> DeviceInputs:
    """Allocate and fill every device buffer of one step (pool_t may be reused)."""
    import torch
    problems = wl.problems if problems is None else problems
    pool = wl.pool
    stream = torch.cuda.current_stream(device).cuda_stream
    if pool_t is None:
        pool_t = torch.empty((pool.num_pages, pool.h), dtype=torch.bfloat16, device=device)
        device_fill_pool(wl, pool_t, stream, nan_dummies)
    T = wl.batch.num_tokens
    w_in = max(pool.dims(p)[0] for (_, p) in problems) if problems else pool.h
    w_out = max(pool.dims(p)[1] for (_, p) in problems) if problems else pool.h
    x = torch.empty((len(problems), T, w_in), dtype=torch.bfloat16, device=device)
    y = torch.empty((len(problems), T, w_out), dtype=torch.bfloat16, device=device)
    if T > 0 and problems:
        device_fill_rows(wl, x, KIND_X, problems, stream)
        device_fill_rows(wl, y, KIND_Y, problems, stream)
    b = wl.batch

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    return DeviceInputs(
        pool=pool_t, pt=i32(pool.pt),
        pt_off=torch.from_numpy(pool.pt_off.astype(np.int64)).to(device),
        ranks=i32(pool.ranks), scales=torch.from_numpy(pool.scales).to(device),
        x=x, y=y, seg_start=i32(b.seg_start), seg_adapter=i32(b.seg_adapter),
        dec_adapter=i32(b.dec_adapter), token_adapter=i32(b.token_adapter()),
        problems=list(problems),
        x_src=[problems.index(wl.x_source(l, p)) if wl.x_source(l, p) in problems else i
               for i, (l, p) in enumerate(problems)])
