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
                      nprob: int, x_buffers: int | None = None) -> dict:
    """Algorithmic bytes and flops of one multi-problem launch over nprob projections
    of size h x h, for a batch whose per-token adapter ids are token_adapter.
    x_buffers: the distinct x buffers the projections read (projections that share their
    input, as q, k and v of a layer do, read it once); nprob if None."""
    ids = np.asarray(token_adapter, dtype=np.int64)
    adapted = ids[ids >= 0]
    distinct = np.unique(adapted)
    r_d = np.asarray(ranks_by_adapter, dtype=np.int64)[distinct]
    r_t = np.asarray(ranks_by_adapter, dtype=np.int64)[adapted]
    page_bytes = int(2 * r_d.sum()) * h * BF16
    x_bytes = adapted.size * h * BF16            # x read
    y_bytes = adapted.size * 2 * h * BF16        # y read and written
    meta_bytes = int(2 * r_d.sum()) * 4 + ids.size * 4
    xb = nprob if x_buffers is None else x_buffers
    xy_total = x_bytes * xb + y_bytes * nprob
    flops = int(adapted.size and (2 * r_t * (2 * h)).sum())
    return {"bytes": (page_bytes + meta_bytes) * nprob + xy_total, "page_bytes": page_bytes * nprob,
            "xy_bytes": xy_total, "meta_bytes": meta_bytes * nprob,
            "flops": flops * nprob, "adapted_tokens": int(adapted.size),
            "tokens": int(ids.size), "distinct_adapters": int(distinct.size)}
