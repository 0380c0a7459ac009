"""Host side of adapter staging (the unified-pool stress workload's slice LRU): after a
plan every needed slice is resident, new pages come from the free list, the page-table
rewrite keeps every entry on the same position of its slice, capacity holds, and no
slice the running or the next step reads is evicted."""
import numpy as np

import bench
from workloads import spec


def test_slice_cache_invariants():
    wl = spec.decode_workload("slices", 5, 64, 3, 2, 40, [1, 2, 4], 8, None, num_pages=4096,
                              distinct=True, layer_slices=True)
    cache = bench.SliceCache(wl, None, capacity=25)
    pt = wl.pool.pt.astype(np.int64).copy()
    steps = bench.step_batches(wl, 12, "distinct")
    prev = np.zeros(0, np.int64)
    for w in steps:
        need = cache.needed(w.batch.token_adapter())
        resident_before = {s: cache.slice_pages[s].copy() for s in cache.lru}
        plan = cache.plan(need, prev)
        assert set(int(v) for v in need) <= set(cache.lru)
        assert len(cache.lru) <= max(cache.capacity, np.union1d(need, prev).size)
        for s in prev:                       # the running step's slices stayed put
            if int(s) in resident_before:
                assert int(s) in cache.lru
                assert np.array_equal(cache.slice_pages[int(s)], resident_before[int(s)])
        if plan is not None:
            rows, dst, ui, up, nmiss = plan
            assert rows.size == dst.size and ui.size == up.size
            assert np.unique(dst).size == dst.size
            pt[ui] = up
        # every entry of every resident slice points at that slice's current page
        for s in cache.lru:
            ent = cache.ent_sorted[cache.ent_off[s]:cache.ent_off[s + 1]]
            assert np.array_equal(pt[ent], cache.slice_pages[s][cache.ent_pos[ent]])
        # resident slices never share pages
        used = np.concatenate([cache.slice_pages[s] for s in cache.lru])
        assert np.unique(used).size == used.size
        assert not (set(used.tolist()) & set(cache.free))
        prev = need
