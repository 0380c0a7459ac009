"""A miniature serving loop on the GPU: requests arrive for adapters held in host memory,
the adapter cache (include/lora_runtime.h) gives each missing adapter pool pages (evicting
least recently used adapters nobody uses), lora_stage_pages (a kernel reading the host rows
through their mapping) or lora_stage_pages_ce (the copy engines: straight into the pool for
runs of consecutive pages, else into a staging buffer and then a kernel) copies its rows in
and points its page-table entries at them, the scheduler picks each step's batch under a token cap and
a distinct-adapter cap, lora_bgmv applies the deltas, and every step is checked against the
fp64 oracle.  Pages freed by evictions are reused, so a stale page-table entry or a missed
copy shows up as a wrong (or NaN) row.

"Multi-LoRA serving: S-LoRA, Punica and adapter batching", "What the engine does each
step"."""
import numpy as np
import pytest

import oracle
from workloads import spec
from workloads import valuegen as vg
from workloads.materialize import host_inputs

from .harness import check_gate

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ["mapped", "copy_engine"])
def test_serving_loop_with_cache_scheduler_and_staging(path):
    import torch

    import heterogeneous_adapters_gb300 as lora
    dev = "cuda:0"
    N, h, L, P = 12, 512, 2, 2
    wl = spec.decode_workload("serve-h512", 95, h, L, P, N, [4, 8, 16], 1, 1.0)
    src = wl.pool
    hi = host_inputs(wl, adapters=np.arange(N), with_xy=False)
    n_pages = (L * P * 2 * src.ranks).astype(np.int32)            # pages per adapter
    # host tier: every adapter's rows in the order of its page-table entries
    host = []
    for a in range(N):
        rows = hi.pool[hi.pt[src.pt_off[a]:src.pt_off[a] + n_pages[a]]]
        host.append(torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).pin_memory())
    # the serving pool: room for about a third of the adapters, NaN until written
    capacity = int(np.sort(n_pages)[::-1][:4].sum())
    pages = torch.full((capacity, h), float("nan"), dtype=torch.bfloat16, device=dev)
    pt = torch.zeros(src.pt.size, dtype=torch.int32, device=dev)  # no adapter resident yet
    off = torch.from_numpy(src.pt_off).to(dev)
    ranks = torch.from_numpy(src.ranks).to(dev)
    scales = torch.from_numpy(src.scales).to(dev)
    pool = lora.Pool(pages, capacity, h, pt, src.pt.size, off, ranks, scales, N, L, P, src.r_max)
    cache = lora.AdapterCache(np.arange(capacity), n_pages)
    sched = lora.Scheduler(cache)
    stream = torch.cuda.current_stream().cuda_stream
    max_tokens, max_distinct = 16, 3
    nbytes = lora.workspace_size(pool, max_tokens, max_tokens)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    lora.workspace_init(ws, nbytes, stream)
    rng = np.random.default_rng(11)
    probs_lp = spec.all_problems(L, P)

    staging = torch.empty(int(n_pages.max()) * h * 2, dtype=torch.uint8, device=dev)

    def stage(a, dst):
        ent = np.arange(src.pt_off[a], src.pt_off[a] + n_pages[a], dtype=np.int64)
        dst_t = torch.from_numpy(dst.astype(np.int32)).pin_memory()
        ui = torch.from_numpy(ent).pin_memory()
        up = torch.from_numpy(dst.astype(np.int32)).pin_memory()
        if path == "mapped":
            lora.stage_pages(pool, host[a], dst_t, dst.size, pt, ui, up, ent.size, stream)
        else:
            lora.stage_pages_ce(pool, host[a], staging, staging.numel(), dst_t, dst.size, pt, ui, up, ent.size,
                                stream)
        torch.cuda.synchronize()        # the copy is done: the adapter becomes ready
        cache.loaded(a)

    def arrive(req, a):
        if a >= 0:
            got = cache.try_acquire(a)
            if got is None:
                return False            # no pages can be freed now: retry later
            loaded, dst, _ = got
            if loaded:
                stage(a, dst)
        sched.enqueue(req, a, 1)
        return True

    later, req, served, checked = [], 0, 0, 0
    probs = rng.choice(N, size=200, p=spec.zipf_probs(N, 0.6))
    for step in range(10):
        arrivals = [(req + i, int(probs[req + i]) if rng.random() > 0.1 else -1) for i in range(6)]
        req += 6
        later = [r for r in later + arrivals if not arrive(*r)]
        ids, ads, _ = sched.pick(max_tokens, max_distinct)
        assert len(set(ads[ads >= 0].tolist())) <= max_distinct and ids.size <= max_tokens
        if ids.size == 0:
            continue
        T = ids.size
        x = torch.randn((len(probs_lp), T, h), generator=torch.Generator().manual_seed(step)).to(torch.bfloat16)
        y = torch.randn((len(probs_lp), T, h), generator=torch.Generator().manual_seed(100 + step)).to(torch.bfloat16)
        xd, yd = x.to(dev), y.to(dev)
        tok = torch.from_numpy(ads.astype(np.int32)).to(dev)
        problems = [(xd[i], yd[i], h, h, l, p) for i, (l, p) in enumerate(probs_lp)]
        lora.bgmv(pool, problems, tok, T, ws, nbytes, stream)
        assert lora.get_device_error(ws, stream) == 0
        out = yd.float().cpu().numpy()
        for i, (l, p) in enumerate(probs_lp):
            xb = x[i].view(torch.int16).numpy().view(np.uint16)
            y0 = vg.bf16_bits_to_f64(y[i].view(torch.int16).numpy().view(np.uint16))
            y_ref, _, _ = oracle.lora_delta(hi.pool, hi.pt, src.pt_off, src.ranks, src.scales, L, P, l, p, xb,
                                            y0, ads.astype(np.int32))
            check_gate(out[i].astype(np.float64), y_ref, f"step {step} problem {(l, p)}")
            checked += 1
        for a in ads[ads >= 0].tolist():
            cache.release(a)            # the request is done with its adapter
        served += T
    st = cache.stats()
    sched.close()
    cache.close()
    pool.close()
    assert checked > 0 and served >= 30
    assert st["misses"] > 4 and st["evictions"] > 0, st      # pages were freed and reused
