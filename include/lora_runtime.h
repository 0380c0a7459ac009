/* Host runtime of liblora.so: the adapter cache over the unified page pool and the batch
 * scheduler.  Plain host code (no GPU call, no device memory): it decides which adapters
 * are resident in which pool pages and which requests go into the next batch; the copies
 * it plans are made with lora_stage_pages (lora.h) on a side stream.
 *
 * "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work"
 * (memory management): adapter weights of the active set sit in pages of the unified GPU
 * pool; inactive adapters live in host memory, and a request for an adapter that is not
 * resident waits while its pages are copied in.  Same page, "What the engine does each
 * step": on arrival, a missing adapter takes the pages of the least recently used adapter
 * that no request is using and is copied in asynchronously; the request becomes ready when
 * the copy is done; each step the scheduler picks a batch under a token cap and a cap on
 * distinct adapters, and a request whose adapter has no slot waits.
 *
 * Units.  The cache manages "units" 0..num_units-1, each occupying a fixed number of pool
 * pages: a unit is an adapter (all its layers), or an adapter slice (e.g. one layer of it)
 * when the page table maps several blocks onto the same pages.  Pages are identified by
 * their index in the pool; the cache hands out only the pages it was given at creation
 * (the rest of the unified pool, e.g. KV-cache blocks, is the caller's).
 *
 * Threading: a cache or scheduler object must not be used from two threads at once. */
#ifndef LORA_RUNTIME_H
#define LORA_RUNTIME_H

#include <stdint.h>

#include "lora.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_cache lora_cache;
typedef struct lora_sched lora_sched;

/* Unit states. */
enum { LORA_UNIT_ABSENT = 0, LORA_UNIT_LOADING = 1, LORA_UNIT_READY = 2 };

/* Creates a cache over the pool pages managed_pages[0..n_managed) (host array, copied;
 * distinct, >= 0) for num_units units of unit_pages[u] >= 1 pages each (host array,
 * copied).  Every unit starts absent and every managed page free.  LORA_EINVAL on bad
 * arguments or duplicate pages. */
lora_status lora_cache_create(lora_cache** out, const int32_t* managed_pages, int64_t n_managed,
                              const int32_t* unit_pages, int32_t num_units);
lora_status lora_cache_destroy(lora_cache* cache);

/* A request for unit u arrives: one more user of u.
 * Hit (u loading or ready): *loaded = 0, u becomes the most recently used unit.
 * Miss (u absent): u needs unit_pages[u] pages; free pages are taken first, then the least
 * recently used ready units with no users are evicted (their pages freed) until enough are
 * free.  u becomes LOADING and its pages are written to pages[0..unit_pages[u]) in the
 * unit's page order (the order of its page-table entries); *loaded = 1.  The caller copies
 * the unit's rows from host memory into those pages and points its page-table entries at
 * them, then calls lora_cache_loaded.  The units evicted are written to evicted[] (up to
 * evicted_cap of them; *n_evicted counts all).
 * LORA_ENOSPACE (and nothing changes) if even evicting every unused ready unit would not
 * free enough pages; LORA_EINVAL for a bad unit or a pages array shorter than
 * unit_pages[u] (pages_cap). */
lora_status lora_cache_acquire(lora_cache* cache, int32_t u, int32_t* loaded, int32_t* pages,
                               int64_t pages_cap, int32_t* evicted, int32_t evicted_cap,
                               int32_t* n_evicted);

/* The copy of unit u has completed (e.g. its event has been waited on): LOADING -> READY.
 * LORA_EINVAL unless u is loading. */
lora_status lora_cache_loaded(lora_cache* cache, int32_t u);

/* A request for unit u has finished: one user fewer.  LORA_EINVAL if u has no users. */
lora_status lora_cache_release(lora_cache* cache, int32_t u);

/* State (LORA_UNIT_*), number of users, and (if pages != NULL and pages_cap is enough)
 * the pool pages of a resident unit. */
lora_status lora_cache_query(const lora_cache* cache, int32_t u, int32_t* state, int32_t* users,
                             int32_t* pages, int64_t pages_cap);

/* Counters since creation: acquires that hit, that missed, units evicted, free pages. */
lora_status lora_cache_stats(const lora_cache* cache, int64_t* hits, int64_t* misses, int64_t* evictions,
                             int64_t* free_pages);

/* Creates a scheduler.  cache may be NULL (every adapter counts as ready); otherwise a
 * request for adapter a >= 0 is ready when unit a of the cache is READY (adapters are
 * then the cache's units). */
lora_status lora_sched_create(lora_sched** out, const lora_cache* cache);
lora_status lora_sched_destroy(lora_sched* sched);

/* Queues request `id` for adapter `adapter` (-1 = base model only) with `tokens` >= 1
 * rows (a prefill chunk, or 1 for a decode step).  Requests keep their arrival order. */
lora_status lora_sched_enqueue(lora_sched* sched, int64_t id, int32_t adapter, int32_t tokens);

/* Picks the next batch: walks the queue in arrival order and takes every request that is
 * ready, fits the remaining token budget (max_tokens in total) and does not bring the
 * number of distinct adapters (>= 0) above max_distinct; a request that does not qualify
 * keeps its place and waits.  Taken requests leave the queue; their ids, adapters and
 * token counts are written in queue order to ids / adapters / tokens (capacity cap;
 * LORA_ETOOBIG if more would be taken, with nothing taken).  *n = requests taken,
 * *n_tokens = their rows, *n_distinct = their distinct adapters. */
lora_status lora_sched_pick(lora_sched* sched, int32_t max_tokens, int32_t max_distinct, int64_t* ids,
                            int32_t* adapters, int32_t* tokens, int32_t cap, int32_t* n, int32_t* n_tokens,
                            int32_t* n_distinct);

/* Requests waiting in the queue. */
lora_status lora_sched_pending(const lora_sched* sched, int64_t* n);

#ifdef __cplusplus
}
#endif

#endif /* LORA_RUNTIME_H */
