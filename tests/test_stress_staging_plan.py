"""Host side of the unified-pool stress workload's staging, run through the library's
adapter cache (lora_cache_*) with slices as units: after planning a step every slice it
reads is resident, the page-table rewrite keeps every entry on the same position of its
slice, resident slices never share pages, and no slice with a user is evicted."""
import numpy as np

import bench
import heterogeneous_adapters_gb300 as lora
from workloads import spec


def test_slice_units_with_the_library_cache():
    wl = spec.decode_workload("slices", 5, 64, 3, 2, 40, [1, 2, 4], 6, None, num_pages=4096,
                              distinct=True, layer_slices=True)
    p = wl.pool
    units = bench.SliceUnits(wl, None)
    spare = np.setdiff1d(np.arange(p.num_pages), p.page_ids)[:200]
    cache = lora.AdapterCache(np.concatenate([p.page_ids, spare]).astype(np.int32), units.spp)
    pt = p.pt.astype(np.int64).copy()
    steps = bench.step_batches(wl, 12, "distinct")
    prev = np.zeros(0, np.int64)
    staged = 0
    for w in steps:
        need = units.needed(w.batch.token_adapter())
        before = {int(s): cache.query(int(s)) for s in prev}
        plan = units.plan(cache, need)
        if plan is not None:
            rows, dst, ui, up, loading = plan
            assert rows.size == dst.size and ui.size == up.size
            assert np.unique(dst).size == dst.size
            pt[ui] = up
            for s in loading:
                cache.loaded(s)
            staged += len(loading)
        for s in prev:                     # the running step's slices stayed put
            state, users, pages = cache.query(int(s))
            assert state == lora.LORA_UNIT_READY and users >= 1
            assert np.array_equal(pages, before[int(s)][2])
        resident = []
        for s in need:                     # every entry of a needed slice points at its pages
            state, _, pages = cache.query(int(s))
            assert state == lora.LORA_UNIT_READY
            ent = units.ent_sorted[units.ent_off[s]:units.ent_off[s + 1]]
            assert np.array_equal(pt[ent], pages.astype(np.int64)[units.ent_pos[ent]])
            resident.append(pages)
        used = np.concatenate(resident)
        assert np.unique(used).size == used.size
        for s in prev:
            cache.release(int(s))
        prev = need
    st = cache.stats()
    assert st["misses"] == staged and st["hits"] > 0
    cache.close()
