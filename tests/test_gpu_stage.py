"""Adapter staging from pinned host memory, by the kernel that reads the host rows
through their mapping (lora_stage_pages) and through the copy engines (lora_stage_pages_ce:
runs of consecutive destination pages copied straight into the pool, or, with more runs
than LORA_STAGE_MAX_RUNS, one copy into a device staging buffer and a kernel moving the
rows): pages land bit-exact in their new pool slots, the page table is rewritten, and a
delta launch ordered after it (event on a side stream) reads the moved adapter correctly."""
import numpy as np
import pytest

from workloads import spec

from .harness import GpuCase, full_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ["mapped", "copy_engine", "copy_engine_runs", "copy_engine_staged"])
def test_stage_moves_adapters_to_free_pages(path):
    import torch

    import heterogeneous_adapters_gb300 as lora
    wl = spec.decode_workload("stage-h1024", 81, 1024, 2, 2, 6, [4, 8, 16], 20, 1.0,
                              num_pages=None)
    pool = wl.pool
    extra = 4096
    # room for the moved copies: grow the pool with free pages after the adapters' pages
    wl.pool.num_pages = pool.num_pages + extra
    case = GpuCase(wl, nan_dummies=True)
    try:
        dev = case.dev
        ids = wl.batch.token_adapter()
        movers = np.unique(ids[ids >= 0])[:3]
        entries = np.concatenate([np.arange(pool.pt_off[a], pool.pt_off[a] + pool.num_layers *
                                            pool.num_proj * 2 * pool.ranks[a]) for a in movers])
        old_pages = pool.pt[entries].astype(np.int64)
        new_pages = (pool.num_pages - extra + np.arange(entries.size)).astype(np.int32)
        if path == "copy_engine_runs":   # a few runs of consecutive pages, separated by gaps
            new_pages = (new_pages + 3 * (np.arange(new_pages.size) // 37)).astype(np.int32)
            runs = 1 + int(np.count_nonzero(np.diff(new_pages) != 1))
            assert 1 < runs <= lora.LORA_STAGE_MAX_RUNS
        if path == "copy_engine_staged":   # scattered destinations: more runs than direct copies take
            new_pages = np.random.default_rng(5).permutation(new_pages).astype(np.int32)
            runs = 1 + int(np.count_nonzero(np.diff(new_pages) != 1))
            assert runs > lora.LORA_STAGE_MAX_RUNS
        # host copy of the rows (the staging source), then poison the old pages
        host_rows = dev.pool[torch.from_numpy(old_pages).to(case.device)].cpu().pin_memory()
        dev.pool[torch.from_numpy(old_pages).to(case.device)] = float("nan")
        dst = torch.from_numpy(new_pages).pin_memory()
        upd_index = torch.from_numpy(entries.astype(np.int64)).pin_memory()
        upd_page = torch.from_numpy(new_pages).pin_memory()
        side = torch.cuda.Stream(device=case.device)
        staging = torch.empty(entries.size * wl.pool.h * 2, dtype=torch.uint8, device=case.device)
        with torch.cuda.stream(side):
            if path == "mapped":
                lora.stage_pages(case.pool, host_rows, dst, entries.size, dev.pt, upd_index, upd_page,
                                 entries.size, side.cuda_stream)
            elif path in ("copy_engine", "copy_engine_runs"):   # runs of consecutive pages: no staging buffer
                lora.stage_pages_ce(case.pool, host_rows, None, 0, dst, entries.size, dev.pt,
                                    upd_index, upd_page, entries.size, side.cuda_stream)
            else:
                lora.stage_pages_ce(case.pool, host_rows, staging, staging.numel(), dst, entries.size, dev.pt,
                                    upd_index, upd_page, entries.size, side.cuda_stream)
            done = torch.cuda.Event()
            done.record(side)
        torch.cuda.current_stream(case.device).wait_event(done)
        # pages bit-exact, page table rewritten
        got = dev.pool[torch.from_numpy(new_pages.astype(np.int64)).to(case.device)].cpu()
        assert torch.equal(got.view(torch.int16), host_rows.view(torch.int16))
        assert np.array_equal(dev.pt.cpu().numpy()[entries], new_pages)
        # the delta reads the moved adapters from their new pages (old ones are NaN)
        assert case.run() == 0
        # the oracle sees the same move: new pages carry the old pages' generator keys
        order = np.argsort(pool.page_ids, kind="stable")
        pos = order[np.searchsorted(pool.page_ids[order], old_pages)]
        pool.page_ids = np.concatenate([pool.page_ids, new_pages.astype(np.int64)])
        pool.page_keys = np.concatenate([pool.page_keys, pool.page_keys[pos]])
        pool.page_ab = np.concatenate([pool.page_ab, pool.page_ab[pos]])
        pool.pt = dev.pt.cpu().numpy()
        full_check(wl, case, list(range(len(wl.problems))), strict=False)
    finally:
        case.close()
