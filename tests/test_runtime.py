"""Host runtime (include/lora_runtime.h): the adapter cache over pool pages and the batch
scheduler, on the CPU.

The cache is replayed against an independent model of its documented rules (written here,
sharing nothing with the C++), operation by operation; its page assignments are checked
against invariants; the scheduler against its caps and its readiness rule; and the Zipf /
LRU simulation of "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How many
adapters are actually in a batch?" is reproduced: 1,000 adapters, batches of 64 requests,
200,000 arrivals through an LRU of GPU slots counted after 20,000 of warm-up — about half
of the arrivals miss at 64 slots and Zipf 1.0, and a batch holds 33 to 62 distinct adapters
on average from strong to mild skew."""
from collections import OrderedDict

import numpy as np
import pytest

from workloads.spec import zipf_probs


@pytest.fixture(scope="module")
def rt():
    from heterogeneous_adapters_gb300 import build
    build.build()
    import heterogeneous_adapters_gb300 as lora
    return lora


class ModelCache:
    """The documented rules, in plain Python: hit if loading or ready; a miss frees pages
    by evicting least recently used ready units with no users, else fails; LRU order by
    last acquire."""

    def __init__(self, n_managed, unit_pages):
        self.free = n_managed
        self.unit_pages = list(unit_pages)
        self.state = {}          # unit -> "loading" | "ready"
        self.users = {}
        self.lru = OrderedDict()
        self.hits = self.misses = self.evictions = 0

    def acquire(self, u):
        if u in self.state:
            self.users[u] += 1
            self.hits += 1
            self.lru.move_to_end(u)
            return "hit", []
        need, avail, victims = self.unit_pages[u], self.free, []
        for v in self.lru:
            if avail >= need:
                break
            if self.users[v] == 0 and self.state[v] == "ready":
                victims.append(v)
                avail += self.unit_pages[v]
        if avail < need:
            return "full", []
        for v in victims:
            del self.state[v], self.users[v], self.lru[v]
            self.free += self.unit_pages[v]
            self.evictions += 1
        self.free -= need
        self.state[u], self.users[u], self.lru[u] = "loading", 1, True
        self.misses += 1
        return "miss", victims


def _check_pages(rt, cache, n_units, managed):
    owned = []
    for u in range(n_units):
        st, _, pages = cache.query(u)
        if st != rt.LORA_UNIT_ABSENT:
            assert pages.size == cache.unit_pages[u]
            owned.extend(pages.tolist())
    assert len(owned) == len(set(owned)), "a page is owned by two resident units"
    assert set(owned) <= set(managed.tolist())
    assert len(owned) + cache.stats()["free_pages"] == managed.size


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cache_matches_model_of_its_rules(rt, seed):
    rng = np.random.default_rng(seed)
    n_units = 12
    unit_pages = rng.integers(1, 6, size=n_units)
    managed = rng.permutation(200)[:30].astype(np.int32)      # the cache's share of the pool
    cache, model = rt.AdapterCache(managed, unit_pages), ModelCache(managed.size, unit_pages)
    try:
        for _ in range(600):
            op = rng.random()
            u = int(rng.integers(n_units))
            if op < 0.5:
                want, victims = model.acquire(u)
                if want == "full":
                    before = cache.stats()
                    assert cache.try_acquire(u) is None
                    assert cache.stats() == before
                else:
                    loaded, pages, ev = cache.acquire(u)
                    assert loaded == (want == "miss")
                    assert ev.tolist() == victims
            elif op < 0.75:
                if model.state.get(u) == "loading":
                    cache.loaded(u)
                    model.state[u] = "ready"
                else:
                    with pytest.raises(rt.LoraError):
                        cache.loaded(u)
            else:
                if model.users.get(u, 0) > 0:
                    cache.release(u)
                    model.users[u] -= 1
                else:
                    with pytest.raises(rt.LoraError):
                        cache.release(u)
            s = cache.stats()
            assert (s["hits"], s["misses"], s["evictions"]) == (model.hits, model.misses, model.evictions)
            assert s["free_pages"] == model.free
        _check_pages(rt, cache, n_units, managed)
    finally:
        cache.close()


def test_cache_never_evicts_units_in_use_or_loading(rt):
    cache = rt.AdapterCache(np.arange(4), [2, 2, 2])
    try:
        assert cache.acquire(0)[0] and cache.acquire(1)[0]        # both loading, both in use
        assert cache.try_acquire(2) is None                       # nothing can be freed
        cache.loaded(0)
        assert cache.try_acquire(2) is None                       # 0 is ready but in use
        cache.release(0)
        loaded, pages, ev = cache.acquire(2)                      # now 0 can go
        assert loaded and ev.tolist() == [0] and sorted(pages.tolist()) in ([0, 1], [2, 3])
        assert cache.query(0)[0] == rt.LORA_UNIT_ABSENT
        cache.release(1)
        assert cache.try_acquire(0) is None                       # 1 is still loading
        cache.loaded(1)
        assert cache.acquire(0)[2].tolist() == [1]
    finally:
        cache.close()


def test_cache_argument_checks(rt):
    with pytest.raises(rt.LoraError):
        rt.AdapterCache([0, 1, 1], [1])                           # duplicate page
    with pytest.raises(rt.LoraError):
        rt.AdapterCache([0, 1], [0])                              # empty unit
    cache = rt.AdapterCache([5, 6], [1])
    try:
        with pytest.raises(rt.LoraError):
            cache.acquire(1)                                      # no such unit
        with pytest.raises(rt.LoraError):
            cache.release(0)                                      # no user
    finally:
        cache.close()


def test_scheduler_caps_order_and_readiness(rt):
    cache = rt.AdapterCache(np.arange(16), [1] * 8)
    sched = rt.Scheduler(cache)
    try:
        for a in (0, 1, 2):
            cache.acquire(a)
        cache.loaded(0)
        cache.loaded(1)                                           # adapter 2 is still loading
        reqs = [(10, 0, 5), (11, 2, 1), (12, 1, 4), (13, -1, 2), (14, 1, 3), (15, 0, 1), (16, 3, 1)]
        for r in reqs:
            sched.enqueue(*r)
        ids, ad, tk = sched.pick(max_tokens=12, max_distinct=1)
        # 10 (adapter 0: 5 rows); 11 waits (loading); 12 would be a second adapter; 13 base
        # (2 rows); 14 second adapter; 15 adapter 0 (1 row); 16 not loaded at all
        assert ids.tolist() == [10, 13, 15] and tk.sum() == 8
        assert sched.pending() == 4
        ids, ad, tk = sched.pick(max_tokens=6, max_distinct=2)
        assert ids.tolist() == [12]                               # 14 would exceed 6 rows
        cache.loaded(2)
        ids, ad, tk = sched.pick(max_tokens=100, max_distinct=8)
        assert ids.tolist() == [11, 14]                           # 16's adapter is absent
        assert sched.pending() == 1
        sched.enqueue(20, -1, 1)
        with pytest.raises(rt.LoraError):
            sched.pick(max_tokens=100, max_distinct=8, cap=0)     # too small an output
        assert sched.pending() == 2                               # and nothing was taken
    finally:
        sched.close()
        cache.close()


def _zipf_arrivals(s, n=200_000, num_adapters=1000, seed=0):
    return np.random.default_rng(seed).choice(num_adapters, size=n, p=zipf_probs(num_adapters, s))


def test_lru_simulation_half_of_arrivals_miss_at_64_slots(rt):
    """Zipf 1.0 over 1,000 adapters, 64 one-page slots, 200,000 arrivals, 20,000 warm-up:
    the native cache gives exactly the hits of an OrderedDict LRU, and about half miss."""
    arr = _zipf_arrivals(1.0)
    cache = rt.AdapterCache(np.arange(64), [1] * 1000)
    hits = 0
    try:
        for i, a in enumerate(arr.tolist()):
            loaded, _, _ = cache.acquire(a)
            if loaded:
                cache.loaded(a)
            cache.release(a)
            if i >= 20_000 and not loaded:
                hits += 1
    finally:
        cache.close()
    lru, want = OrderedDict(), 0
    for i, a in enumerate(arr.tolist()):
        hit = a in lru
        if hit:
            lru.move_to_end(a)
        else:
            if len(lru) >= 64:
                lru.popitem(last=False)
            lru[a] = True
        want += hit and i >= 20_000
    assert hits == want
    miss = 1 - hits / (arr.size - 20_000)
    assert 0.45 <= miss <= 0.55, miss


def test_distinct_adapters_per_batch_of_64():
    """Mean distinct adapters in a batch of 64 requests: about 33 under strong skew
    (Zipf 1.2), about 62 under mild skew (Zipf 0.5)."""
    for s, lo, hi in ((1.2, 31, 36), (0.5, 59, 63)):
        arr = _zipf_arrivals(s, n=64 * 2000)
        d = np.array([np.unique(arr[i:i + 64]).size for i in range(0, arr.size, 64)])
        assert lo <= d.mean() <= hi, (s, d.mean())
