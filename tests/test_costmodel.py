"""Byte model of the roofline numerator, counted against the arrays one step touches."""
import numpy as np

from heterogeneous_adapters_gb300 import costmodel
from workloads import spec
from workloads.materialize import host_inputs
from workloads.spec import Batch, Workload, all_problems, make_pool_all_resident

from .harness import block_values


def test_width_bytes_equal_the_arrays_a_step_reads_and_writes():
    """Adapter values of every distinct adapter of the batch, x rows read and y rows read
    and written by adapted tokens, at each projection's own widths (base-only rows are
    not touched)."""
    rng = np.random.default_rng(5)
    h, dims = 256, [(256, 64), (256, 640), (640, 256)]
    ranks = rng.choice(np.asarray([2, 5, 8], np.int32), size=6)
    pool = make_pool_all_resident(rng, h, 2, 3, ranks, proj_dims=dims)
    ids = np.asarray([0, 3, -1, 3, 5, -1, 0, 0], np.int32)
    wl = Workload("w", 5, pool, Batch(np.zeros(1, np.int32), np.zeros(0, np.int32), ids),
                  all_problems(2, 3))
    hi = host_inputs(wl)
    want = 0
    adapted = ids[ids >= 0]
    for (l, p) in wl.problems:
        for a in np.unique(adapted):
            want += 2 * (block_values(wl, hi, a, l, p, 0).size + block_values(wl, hi, a, l, p, 1).size)
        want += 2 * hi.x[(l, p)][ids >= 0].size + 2 * 2 * hi.y0[(l, p)][ids >= 0].size
    m = costmodel.decode_step_bytes(pool.ranks, ids, h, len(wl.problems),
                                    dims=[pool.dims(p) for (_, p) in wl.problems])
    assert m["page_bytes"] + m["xy_bytes"] == want
    assert m["meta_bytes"] > 0 and m["bytes"] == want + m["meta_bytes"]


def test_square_dims_match_the_h_by_h_model_and_adapter_size():
    wl = spec.tiny_decode()
    p = wl.pool
    ids = wl.batch.token_adapter()
    a = costmodel.decode_step_bytes(p.ranks, ids, p.h, 3)
    b = costmodel.decode_step_bytes(p.ranks, ids, p.h, 3, dims=[(p.h, p.h)] * 3)
    assert a == b
    # one token of one adapter: its page bytes are the adapter's parameters of that layer
    one = costmodel.decode_step_bytes(np.asarray([16]), np.asarray([0]), 4096, 7,
                                      dims=spec.LLAMA3_8B_DIMS)
    assert one["page_bytes"] == 2 * costmodel.adapter_params(1, spec.LLAMA3_8B_DIMS, 16)


def test_llama3_8b_worked_example():
    """"Multi-LoRA serving: S-LoRA, Punica and adapter batching", "Worked example: a thousand
    adapters on one 8B base": a layer's sum of (d_in + d_out) over the seven projections is
    81,920; at r = 16 an adapter has 41.9M parameters (83.9 MB in bf16) against 6.98B base
    parameters in the linear layers."""
    dims = spec.LLAMA3_8B_DIMS
    assert sum(a + b for a, b in dims) == 81920
    n = costmodel.adapter_params(32, dims, 16)
    assert round(n / 1e6, 1) == 41.9 and round(2 * n / 1e6, 1) == 83.9
    assert round(32 * sum(a * b for a, b in dims) / 1e9, 2) == 6.98


def test_physical_page_bytes_count_shared_pages_once():
    """A pool whose layers map onto one shared slice of pages (the unified-pool stress
    layout): the physical count is the set of page ids the launch's page-table entries
    hold, each counted once at its widest use; the logical count is per block."""
    h = 256
    rng = np.random.default_rng(11)
    ranks = np.asarray([2, 4, 4], np.int64)
    L, P = 3, 2
    U = 2 * P
    pt_off = np.concatenate([[0], np.cumsum(L * U * ranks)[:-1]])
    pt = np.zeros(int((L * U * ranks).sum()), np.int32)
    # every adapter owns U * r physical pages; layer l maps onto them through a permutation
    # of the adapter's slice entries, so the 3 layers read the same pages
    base = 0
    for a, r in enumerate(ranks):
        slice_pages = base + np.arange(U * r)
        base += U * r
        for l in range(L):
            perm = rng.permutation(U * r)
            pt[pt_off[a] + l * U * r: pt_off[a] + (l + 1) * U * r] = slice_pages[perm]
    ids = np.asarray([0, 2, 2, -1, 0], np.int32)
    blocks = [(l * U + 2 * p, h, h) for l in range(L) for p in range(P)]
    phys, logical = costmodel.physical_page_bytes(pt, pt_off, ranks, ids, h, blocks)
    read = set()
    for a in (0, 2):
        r = int(ranks[a])
        for blk, _, _ in blocks:
            read |= set(pt[pt_off[a] + r * blk: pt_off[a] + r * blk + 2 * r].tolist())
    assert phys == len(read) * h * 2
    assert logical == len(blocks) * 2 * (2 + 4) * h * 2
    assert phys == (U * (2 + 4)) * h * 2 < logical
    # a pool where every block owns its pages: the two counts agree, and agree with the
    # per-block model of decode_step_bytes
    wl = spec.tiny_decode()
    p = wl.pool
    Up, pre, _, _ = p.layout_units()
    blocks = [(l * Up + pre[pj],) + p.dims(pj) for (l, pj) in wl.problems]
    phys, logical = costmodel.physical_page_bytes(p.pt, p.pt_off, p.ranks, wl.batch.token_adapter(),
                                                  p.h, blocks)
    m = costmodel.decode_step_bytes(p.ranks, wl.batch.token_adapter(), p.h, len(wl.problems),
                                    page_bytes_physical=phys)
    assert phys == logical == m["page_bytes_logical"] == m["page_bytes"]
