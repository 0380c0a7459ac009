"""Byte and flop model of the multi-LoRA delta (host logic for measurement).

From "Multi-LoRA serving: S-LoRA, Punica and adapter batching":
  * "The bottleneck: merged models do not batch together": per layer, n distinct
    adapters of rank r add n*r*(d_in + d_out) weights next to the base d_in*d_out,
    and every token pays 2*r*(d_in + d_out) extra flops;
  * "Worked example: a thousand adapters on one 8B base": adapter size, H2D copy
    time at a given link bandwidth, and decode time per distinct adapter at a
    given HBM bandwidth.

Algorithmic bytes of one launch (the roofline numerator) count each distinct
adapter's A and B pages once per projection, each adapted token's x row once and
its y row twice (read + write), and the page-table and index words read.
"""
from __future__ import annotations

import numpy as np

BF16 = 2


def extra_weight_ratio(n_adapters: int, rank: int, d_in: int, d_out: int) -> float:
    """Adapter weights of n distinct adapters relative to the base weight of one projection."""
    return n_adapters * rank * (d_in + d_out) / (d_in * d_out)


def extra_flops_per_token(rank: int, d_in: int, d_out: int) -> int:
    """Extra flops of one adapted token in one projection (multiply + add counted)."""
    return 2 * rank * (d_in + d_out)


def adapter_params(num_layers: int, proj_dims, rank: int) -> int:
    """LoRA parameters of one adapter: layers * sum(d_in + d_out) * r."""
    return num_layers * sum(di + do for di, do in proj_dims) * rank


def transfer_seconds(nbytes: float, bytes_per_s: float) -> float:
    return nbytes / bytes_per_s


def physical_page_bytes(pt: np.ndarray, pt_off: np.ndarray, ranks_by_adapter: np.ndarray,
                        token_adapter: np.ndarray, h: int, blocks) -> tuple[int, int]:
    """Bytes of the distinct physical pool pages one launch reads, and of the logical
    (adapter, projection) blocks it reads.  The two differ only where page tables of
    different blocks point at the same pages (a pool that holds one layer's slice of each
    adapter and maps every layer onto it): a page read twice by one launch is a DRAM read
    once and an L2 hit after, so the roofline numerator counts it once.
    blocks: per projection of the launch, (blk, d_in, d_out) with blk the A block's offset
    in units of r_a page-table entries (l * U + pre(p)); only the used part of a partly
    used last page counts."""
    ids = np.asarray(token_adapter, dtype=np.int64)
    distinct = np.unique(ids[ids >= 0])
    pages, used = [], []
    logical = 0
    for a in distinct:
        r = int(ranks_by_adapter[a])
        off = int(pt_off[a])
        for blk, d_in, d_out in blocks:
            pv_in, pv_out = -(-d_in // h), -(-d_out // h)
            start = off + r * blk
            ent = np.arange(start, start + r * (pv_in + pv_out), dtype=np.int64)
            kb = (ent - start) // r                     # page block of each entry
            width = np.where(kb < pv_in, np.minimum(h, d_in - kb * h),
                             np.minimum(h, d_out - (kb - pv_in) * h))
            pages.append(pt[ent].astype(np.int64))
            used.append(width.astype(np.int64) * BF16)
            logical += int(width.sum()) * BF16
    if not pages:
        return 0, 0
    pages, used = np.concatenate(pages), np.concatenate(used)
    order = np.lexsort((-used, pages))                  # per page, its widest use first
    first = np.ones(order.size, bool)
    first[1:] = pages[order][1:] != pages[order][:-1]
    return int(used[order][first].sum()), logical


def decode_step_bytes(ranks_by_adapter: np.ndarray, token_adapter: np.ndarray, h: int,
                      nprob: int, x_buffers: int | None = None, dims=None, x_widths=None,
                      page_bytes_physical: int | None = None) -> dict:
    """Algorithmic bytes and flops of one multi-problem launch over nprob projections,
    for a batch whose per-token adapter ids are token_adapter.
    dims: the projections' (d_in, d_out) widths; h x h each if None.  Only the d_in + d_out
    used elements of an adapter's vectors count, not the unused tail of their last page.
    x_widths: the widths of the distinct x buffers the launch reads (projections that
    share their input, as q, k and v of a layer do, read it once); one buffer per
    projection of its d_in if None, or x_buffers buffers of width h when that is given.
    page_bytes_physical: the distinct physical page bytes of the launch
    (physical_page_bytes); when given, it replaces the per-block page count in "bytes"
    (the per-block count stays in "page_bytes_logical")."""
    ids = np.asarray(token_adapter, dtype=np.int64)
    adapted = ids[ids >= 0]
    distinct = np.unique(adapted)
    r_d = np.asarray(ranks_by_adapter, dtype=np.int64)[distinct]
    r_t = np.asarray(ranks_by_adapter, dtype=np.int64)[adapted]
    dims = [(h, h)] * nprob if dims is None else [(int(a), int(b)) for a, b in dims]
    assert len(dims) == nprob
    if x_widths is None:
        x_widths = [di for di, _ in dims] if x_buffers is None else [h] * x_buffers
    rs, rt = int(r_d.sum()), int(r_t.sum())
    page_bytes = sum(rs * (di + do) * BF16 for di, do in dims)
    meta_bytes = sum(rs * (-(-di // h) + -(-do // h)) * 4 + ids.size * 4 for di, do in dims)
    x_bytes = adapted.size * sum(x_widths) * BF16                      # x read
    y_bytes = adapted.size * 2 * sum(do for _, do in dims) * BF16      # y read and written
    flops = sum(2 * rt * (di + do) for di, do in dims)
    logical = page_bytes
    if page_bytes_physical is not None:
        page_bytes = int(page_bytes_physical)
    return {"bytes": page_bytes + meta_bytes + x_bytes + y_bytes, "page_bytes": page_bytes,
            "page_bytes_logical": logical,
            "xy_bytes": x_bytes + y_bytes, "meta_bytes": meta_bytes,
            "flops": flops, "adapted_tokens": int(adapted.size),
            "tokens": int(ids.size), "distinct_adapters": int(distinct.size)}
