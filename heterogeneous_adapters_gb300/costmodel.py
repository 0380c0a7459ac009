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


def decode_step_bytes(ranks_by_adapter: np.ndarray, token_adapter: np.ndarray, h: int,
                      nprob: int, x_buffers: int | None = None, dims=None, x_widths=None) -> dict:
    """Algorithmic bytes and flops of one multi-problem launch over nprob projections,
    for a batch whose per-token adapter ids are token_adapter.
    dims: the projections' (d_in, d_out) widths; h x h each if None.  Only the d_in + d_out
    used elements of an adapter's vectors count, not the unused tail of their last page.
    x_widths: the widths of the distinct x buffers the launch reads (projections that
    share their input, as q, k and v of a layer do, read it once); one buffer per
    projection of its d_in if None, or x_buffers buffers of width h when that is given."""
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
    return {"bytes": page_bytes + meta_bytes + x_bytes + y_bytes, "page_bytes": page_bytes,
            "xy_bytes": x_bytes + y_bytes, "meta_bytes": meta_bytes,
            "flops": flops, "adapted_tokens": int(adapted.size),
            "tokens": int(ids.size), "distinct_adapters": int(distinct.size)}
