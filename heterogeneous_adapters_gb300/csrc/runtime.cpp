// Host runtime: adapter cache over the unified page pool and the batch scheduler
// (contracts in include/lora_runtime.h).  Plain C++; no CUDA call.
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work" and
// "What the engine does each step": resident adapters occupy pages of the shared pool,
// a miss takes the pages of the least recently used adapter that no request uses and is
// copied in asynchronously, a request waits until its adapter's copy is done, and each
// step's batch is capped in tokens and in distinct adapters.
#include <stdint.h>

#include <algorithm>
#include <deque>
#include <list>
#include <new>
#include <unordered_set>
#include <vector>

#include "lora_runtime.h"

struct lora_cache {
    std::vector<int32_t> unit_pages;            // pages each unit occupies
    std::vector<int8_t> state;                  // LORA_UNIT_*
    std::vector<int32_t> users;
    std::vector<std::vector<int32_t>> pages;    // pool pages of resident units, in unit order
    std::list<int32_t> lru;                     // resident units, least recently used first
    std::vector<std::list<int32_t>::iterator> where;
    std::vector<int32_t> free_pages;            // a stack: the most recently freed page first out
    int64_t hits = 0, misses = 0, evictions = 0;
};

struct lora_sched {
    struct Req {
        int64_t id;
        int32_t adapter;
        int32_t tokens;
    };
    std::deque<Req> queue;
    const lora_cache* cache = nullptr;
};

namespace {

bool valid_unit(const lora_cache* c, int32_t u) {
    return c != nullptr && u >= 0 && u < (int32_t)c->unit_pages.size();
}

void touch(lora_cache* c, int32_t u) {
    c->lru.splice(c->lru.end(), c->lru, c->where[u]);
}

}  // namespace

extern "C" {

lora_status lora_cache_create(lora_cache** out, const int32_t* managed_pages, int64_t n_managed,
                              const int32_t* unit_pages, int32_t num_units) {
    if (out == nullptr || n_managed < 0 || num_units <= 0 || unit_pages == nullptr) return LORA_EINVAL;
    if (n_managed > 0 && managed_pages == nullptr) return LORA_EINVAL;
    for (int32_t u = 0; u < num_units; ++u)
        if (unit_pages[u] < 1) return LORA_EINVAL;
    std::unordered_set<int32_t> seen;
    seen.reserve((size_t)n_managed);
    for (int64_t i = 0; i < n_managed; ++i)
        if (managed_pages[i] < 0 || !seen.insert(managed_pages[i]).second) return LORA_EINVAL;
    lora_cache* c = new (std::nothrow) lora_cache;
    if (c == nullptr) return LORA_EINVAL;
    c->unit_pages.assign(unit_pages, unit_pages + num_units);
    c->state.assign((size_t)num_units, (int8_t)LORA_UNIT_ABSENT);
    c->users.assign((size_t)num_units, 0);
    c->pages.resize((size_t)num_units);
    c->where.resize((size_t)num_units, c->lru.end());
    // the first managed page is handed out first
    c->free_pages.assign(managed_pages, managed_pages + n_managed);
    std::reverse(c->free_pages.begin(), c->free_pages.end());
    *out = c;
    return LORA_OK;
}

lora_status lora_cache_destroy(lora_cache* cache) {
    delete cache;
    return LORA_OK;
}

lora_status lora_cache_acquire(lora_cache* c, int32_t u, int32_t* loaded, int32_t* pages, int64_t pages_cap,
                               int32_t* evicted, int32_t evicted_cap, int32_t* n_evicted) {
    if (!valid_unit(c, u) || loaded == nullptr) return LORA_EINVAL;
    if (n_evicted != nullptr) *n_evicted = 0;
    if (c->state[u] != LORA_UNIT_ABSENT) {   // hit: resident, ready or still loading
        ++c->users[u];
        ++c->hits;
        touch(c, u);
        *loaded = 0;
        return LORA_OK;
    }
    const int64_t need = c->unit_pages[u];
    if (pages == nullptr || pages_cap < need) return LORA_EINVAL;
    // victims: least recently used first, only ready units nobody uses
    std::vector<int32_t> victims;
    int64_t avail = (int64_t)c->free_pages.size();
    for (auto it = c->lru.begin(); it != c->lru.end() && avail < need; ++it) {
        const int32_t v = *it;
        if (c->users[v] == 0 && c->state[v] == LORA_UNIT_READY) {
            victims.push_back(v);
            avail += c->unit_pages[v];
        }
    }
    if (avail < need) return LORA_ENOSPACE;   // nothing has been changed
    for (int32_t v : victims) {
        for (auto it = c->pages[v].rbegin(); it != c->pages[v].rend(); ++it) c->free_pages.push_back(*it);
        c->pages[v].clear();
        c->state[v] = LORA_UNIT_ABSENT;
        c->lru.erase(c->where[v]);
        c->where[v] = c->lru.end();
        ++c->evictions;
    }
    if (n_evicted != nullptr) *n_evicted = (int32_t)victims.size();
    if (evicted != nullptr)
        for (size_t k = 0; k < victims.size() && (int64_t)k < evicted_cap; ++k) evicted[k] = victims[k];
    std::vector<int32_t>& mine = c->pages[u];
    mine.resize((size_t)need);
    for (int64_t k = 0; k < need; ++k) {
        mine[(size_t)k] = c->free_pages.back();
        c->free_pages.pop_back();
        pages[k] = mine[(size_t)k];
    }
    c->state[u] = LORA_UNIT_LOADING;
    c->where[u] = c->lru.insert(c->lru.end(), u);
    ++c->users[u];
    ++c->misses;
    *loaded = 1;
    return LORA_OK;
}

lora_status lora_cache_loaded(lora_cache* c, int32_t u) {
    if (!valid_unit(c, u) || c->state[u] != LORA_UNIT_LOADING) return LORA_EINVAL;
    c->state[u] = LORA_UNIT_READY;
    return LORA_OK;
}

lora_status lora_cache_release(lora_cache* c, int32_t u) {
    if (!valid_unit(c, u) || c->users[u] <= 0) return LORA_EINVAL;
    --c->users[u];
    return LORA_OK;
}

lora_status lora_cache_query(const lora_cache* c, int32_t u, int32_t* state, int32_t* users, int32_t* pages,
                             int64_t pages_cap) {
    if (!valid_unit(c, u)) return LORA_EINVAL;
    if (state != nullptr) *state = c->state[u];
    if (users != nullptr) *users = c->users[u];
    if (pages != nullptr) {
        if (pages_cap < (int64_t)c->pages[u].size()) return LORA_EINVAL;
        std::copy(c->pages[u].begin(), c->pages[u].end(), pages);
    }
    return LORA_OK;
}

lora_status lora_cache_stats(const lora_cache* c, int64_t* hits, int64_t* misses, int64_t* evictions,
                             int64_t* free_pages) {
    if (c == nullptr) return LORA_EINVAL;
    if (hits != nullptr) *hits = c->hits;
    if (misses != nullptr) *misses = c->misses;
    if (evictions != nullptr) *evictions = c->evictions;
    if (free_pages != nullptr) *free_pages = (int64_t)c->free_pages.size();
    return LORA_OK;
}

lora_status lora_sched_create(lora_sched** out, const lora_cache* cache) {
    if (out == nullptr) return LORA_EINVAL;
    lora_sched* s = new (std::nothrow) lora_sched;
    if (s == nullptr) return LORA_EINVAL;
    s->cache = cache;
    *out = s;
    return LORA_OK;
}

lora_status lora_sched_destroy(lora_sched* sched) {
    delete sched;
    return LORA_OK;
}

lora_status lora_sched_enqueue(lora_sched* s, int64_t id, int32_t adapter, int32_t tokens) {
    if (s == nullptr || adapter < -1 || tokens < 1) return LORA_EINVAL;
    if (s->cache != nullptr && adapter >= 0 && !valid_unit(s->cache, adapter)) return LORA_EINVAL;
    s->queue.push_back({id, adapter, tokens});
    return LORA_OK;
}

lora_status lora_sched_pick(lora_sched* s, int32_t max_tokens, int32_t max_distinct, int64_t* ids,
                            int32_t* adapters, int32_t* tokens, int32_t cap, int32_t* n, int32_t* n_tokens,
                            int32_t* n_distinct) {
    if (s == nullptr || max_tokens < 0 || max_distinct < 0 || cap < 0 || n == nullptr) return LORA_EINVAL;
    if (cap > 0 && (ids == nullptr || adapters == nullptr || tokens == nullptr)) return LORA_EINVAL;
    std::vector<size_t> take;
    std::unordered_set<int32_t> distinct;
    int64_t budget = max_tokens;
    for (size_t k = 0; k < s->queue.size() && budget > 0; ++k) {
        const lora_sched::Req& r = s->queue[k];
        if (r.tokens > budget) continue;
        if (r.adapter >= 0) {
            if (s->cache != nullptr && s->cache->state[r.adapter] != LORA_UNIT_READY) continue;
            if (!distinct.count(r.adapter)) {
                if ((int32_t)distinct.size() >= max_distinct) continue;
                distinct.insert(r.adapter);
            }
        }
        take.push_back(k);
        budget -= r.tokens;
    }
    if ((int64_t)take.size() > cap) return LORA_ETOOBIG;
    int32_t rows = 0;
    for (size_t j = 0; j < take.size(); ++j) {
        const lora_sched::Req& r = s->queue[take[j]];
        ids[j] = r.id;
        adapters[j] = r.adapter;
        tokens[j] = r.tokens;
        rows += r.tokens;
    }
    // remove the taken requests, keeping the others in arrival order
    std::deque<lora_sched::Req> rest;
    size_t t = 0;
    for (size_t k = 0; k < s->queue.size(); ++k) {
        if (t < take.size() && take[t] == k) {
            ++t;
            continue;
        }
        rest.push_back(s->queue[k]);
    }
    s->queue.swap(rest);
    *n = (int32_t)take.size();
    if (n_tokens != nullptr) *n_tokens = rows;
    if (n_distinct != nullptr) *n_distinct = (int32_t)distinct.size();
    return LORA_OK;
}

lora_status lora_sched_pending(const lora_sched* s, int64_t* n) {
    if (s == nullptr || n == nullptr) return LORA_EINVAL;
    *n = (int64_t)s->queue.size();
    return LORA_OK;
}

}  // extern "C"
