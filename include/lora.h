/*
 * lora.h - C ABI of the GB300 multi-LoRA delta library (liblora.so).
 *
 * Operation (every entry point computes this, for several projections at once):
 *
 *     y[i, :] += s_a * (x[i, :] . A_a^T) . B_a^T          for every token i with adapter a = a(i) >= 0
 *
 * where A_a is r_a x h, B_a is h x r_a and s_a = alpha / r_a is the caller's
 * per-adapter scale.  Tokens with adapter id -1 are base-only: their y rows are
 * neither read nor written.
 *   Sources, by page and section:
 *   - "Multi-LoRA serving: S-LoRA, Punica and adapter batching" (pofe.ai),
 *     "How the kernels work": the delta is a shrink v_i = A_{a(i)} x_i followed by an
 *     expand y_i += gamma B_{a(i)} v_i; BGMV serves decode (each token independent,
 *     weights gathered by a(i)), SGMV serves prefill (tokens grouped into contiguous
 *     same-adapter segments, one small GEMM per segment, one launch); an index maps
 *     each token to its adapter.  "What the engine does each step": shrink then
 *     expand per layer and LoRA target.
 *   - "S-LoRA: Serving Thousands of Concurrent LoRA Adapters" (fdeinterviews),
 *     "Unified paging" and "Kernels and tensor parallelism": one pool of pages of one
 *     hidden-size vector each; kernels gather each request's adapter from
 *     non-contiguous pages and handle mixed ranks without padding.
 *   - "S-LoRA: Serving Thousands of Concurrent Adapters in 2026" (aifetchly),
 *     "Implementation": scale = alpha / rank; A is rank x in_dim, B is out_dim x rank.
 *
 * Data layout (all device memory is owned by the caller; the library only borrows
 * pointers for the duration of a call and allocates no device memory):
 *   pool          bf16 [num_pages][h]: page q holds h contiguous values (2h bytes),
 *                 16-byte aligned.  d_in = d_out = h.
 *   page_table    int32 [page_table_len]; adapter a owns the block starting at
 *                 adapter_pt_off[a] of length L*P*2*r_a.  Entry
 *                 ((layer*P + proj)*2 + 0)*r_a + j is the page of row j of A_a and
 *                 ((layer*P + proj)*2 + 1)*r_a + j the page of column j of B_a.
 *   ranks         int32 [num_adapters], 1 <= r_a <= r_max (r_max <= LORA_MAX_RANK).
 *   scales        f32 [num_adapters] (s_a).
 *   x, y          bf16 row-major [T][ld] per problem, ld % 8 == 0, 16-byte aligned
 *                 base pointers.  y is updated in place.
 *
 * Numerics: bf16 products are exact in fp32; t = A x is accumulated in fp32 and
 * never rounded to a single bf16 before the expand (the tensor-core expand consumes
 * each fp32 value as a bf16 pair hi + lo with |t - hi - lo| <= 2^-16 |t|); the result
 * is rounded to bf16 (round to nearest even) once, when y is stored.
 *
 * Calls are asynchronous on the caller's stream (a cudaStream_t passed as void*;
 * NULL = legacy default stream) and never synchronise the host, except
 * lora_get_device_error.  Host-side argument checks return a status at once and
 * launch nothing.  Data-dependent errors found on the device (a bad adapter id, a
 * rank out of range, a page id out of range, bad segment offsets) set bits of the
 * workspace's device error word and skip the offending group; the rest of the batch
 * is still computed.  No kernel traps or spins without a bound: every wait inside a
 * kernel gives up after a time limit and reports LORA_DERR_TIMEOUT.
 *
 * Threading: a pool handle is read-only after creation (lora_pool_set_tuning aside) and
 * may be shared by calls on different streams.  A workspace must not be used by two
 * calls that may run concurrently on the GPU.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_MAX_RANK 256
/* Problems per kernel launch; a call with more problems issues several launches. */
#define LORA_MAX_PROBLEMS_PER_LAUNCH 256
/* Maximum adapter "segments" of one call: prefill segments + decode tokens. */
#define LORA_MAX_SEGMENTS 16384
#define LORA_MAX_VEC_PAGES 16           /* pages one A row or B column may span */

typedef enum {
    LORA_OK = 0,
    LORA_EINVAL = 1,      /* null pointer, non-positive size, inconsistent sizes    */
    LORA_EALIGN = 2,      /* pointer not 16-byte aligned or ld not a multiple of 8 */
    LORA_EWORKSPACE = 3,  /* workspace null, misaligned or smaller than required   */
    LORA_ETOOBIG = 4,     /* a size beyond a documented maximum                    */
    LORA_ECUDA = 5,       /* a CUDA runtime call failed (lora_last_cuda_error)     */
    LORA_EDEVICE = 6,     /* device error bits were set (lora_get_device_error)    */
    LORA_ENOSPACE = 7     /* adapter cache: no pages can be freed (all units in use) */
} lora_status;

/* Device error bits (data-dependent errors found by the kernels). */
#define LORA_DERR_ADAPTER 0x1u  /* adapter id outside [-1, num_adapters)            */
#define LORA_DERR_RANK 0x2u     /* rank outside [1, r_max]                           */
#define LORA_DERR_PTBLOCK 0x4u  /* adapter page-table block outside the table        */
#define LORA_DERR_PAGE 0x8u     /* page id outside [0, num_pages)                    */
#define LORA_DERR_SEGMENT 0x10u /* segment offsets decreasing or beyond the rows     */
#define LORA_DERR_TIMEOUT 0x20u /* a kernel wait exceeded its time limit (2 s); the
                                   kernel unwound and its outputs are incomplete      */

/* Pool description: plain device pointers and sizes (copied by lora_pool_create). */
typedef struct {
    void* pages;                   /* device bf16 [num_pages][h]                      */
    int64_t num_pages;
    int32_t h;                     /* page length in bf16 values; h % 8 == 0           */
    int32_t num_adapters;
    int32_t num_layers;            /* L                                                */
    int32_t num_proj;              /* P                                                */
    int32_t r_max;                 /* largest rank present, <= LORA_MAX_RANK           */
    int32_t reserved;
    const int32_t* page_table;     /* device int32 [page_table_len]                    */
    int64_t page_table_len;
    const int64_t* adapter_pt_off; /* device int64 [num_adapters]                      */
    const int32_t* ranks;          /* device int32 [num_adapters]                      */
    const float* scales;           /* device f32   [num_adapters]                      */
    /* host int32 [num_proj][2]: (d_in, d_out) of each projection, multiples of 8 and at
     * most LORA_MAX_VEC_PAGES * h, copied at creation; NULL: every projection is h x h.
     * "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "Worked example": the
     * adapted projections of a model have different widths (grouped-query k/v, MLP).
     * Page-table layout: a vector of length d takes ceil(d/h) pages (the last partly
     * used); adapter a's block for (layer l, projection p, A or B) holds r_a * ceil(d/h)
     * entries, page kb of every row (A) or column (B) and then page kb + 1; with
     * u(p) = ceil(d_in/h) + ceil(d_out/h), U = sum of u over the projections and
     * pre(p) = sum of u over the projections before p, the A block starts at entry
     * adapter_pt_off[a] + r_a * (l * U + pre(p)) and the B block r_a * ceil(d_in/h) later
     * (for h x h: (l * P + p) * 2 * r_a and r_a later).  Tensor-core tiles serve pools
     * whose d_in are multiples of 64 and d_out multiples of 128 (h a multiple of 128);
     * other pools run prefill segments on the CUDA-core kernels. */
    const int32_t* proj_dims;
} lora_pool_desc;

typedef struct lora_pool lora_pool; /* opaque, host memory only */

/* One projection instance: y (bf16 [T][ldy], d_out columns updated) += delta computed
 * from x (bf16 [T][ldx], d_in columns read) with the adapters' pages for (layer, proj).
 * All problems of one call share the batch (the same tokens and adapter ids).  Problems
 * may share x, but their y elements must not overlap: each problem's y is read and
 * rewritten in place by work items that run at the same time. */
typedef struct {
    const void* x;
    void* y;
    int64_t ldx;                   /* elements, % 8 == 0, >= d_in (h for h x h pools)  */
    int64_t ldy;                   /* elements, % 8 == 0, >= d_out                     */
    int32_t layer;
    int32_t proj;
} lora_problem;

/* Validates and copies the description (host-side checks only: sizes, alignment,
 * null pointers).  Device arrays are checked lazily by the kernels.  *out receives
 * a host handle; free it with lora_pool_destroy.  Returns LORA_EINVAL, LORA_EALIGN
 * or LORA_ETOOBIG on a bad description. */
lora_status lora_pool_create(lora_pool** out, const lora_pool_desc* desc);
lora_status lora_pool_destroy(lora_pool* pool);

/* Launch tuning of a pool: which kernel serves which work and the shape of its stages.
 * Every field has a measured default, which lora_pool_create installs; a field given
 * its "default" value below takes that default.  The results never depend on these
 * choices beyond the rounding order of the fp32 sums: they exist for measurement and
 * tests.  The library reads no environment variable.  Set the tuning before the pool
 * is shared between threads (calls read it from the handle). */
typedef struct {
    int32_t ring_rows_per_stage; /* CUDA-core ring: rows (pages) per shared-memory stage,
                                    4 or 8; 0 = 8 where three stages fit, else 4        */
    int32_t split_max_problems;  /* decode launches of at most this many projections run
                                    the cluster kernel (each chunk split over 8 CTAs);
                                    0 = never, 1..8; -1 = default (1)                   */
    int32_t mma_min_rows;        /* prefill segments of at least this many rows take the
                                    tensor-core tiles; 0 = never, >= 2; -1 = default:
                                    by rank, 512 / r rows under rank 32, 16 from rank
                                    32 up (the measured crossover of the two paths)     */
    int32_t mma_y_stages;        /* depth of the tensor-core kernel's y ring, 2..4;
                                    0 = default (3)                                     */
    float fused_ring_speed;      /* mixed launch: per-CTA byte rate of the CUDA-core body
                                    over the tensor-core body's (0.1 .. 10); 0 = default */
    int32_t reserved[3];         /* must be 0                                           */
} lora_tuning;

/* t == NULL restores the defaults.  Returns LORA_EINVAL for a value outside the ranges
 * above (the pool keeps its previous tuning). */
lora_status lora_pool_set_tuning(lora_pool* pool, const lora_tuning* t);
/* The effective values (defaults resolved). */
lora_status lora_pool_get_tuning(const lora_pool* pool, lora_tuning* out);

/* Bytes of device workspace needed by a call over at most max_tokens rows and at
 * most max_segments segments (prefill segments + decode tokens).  The workspace
 * holds the grouping of the batch, the work lists and the device error word; no
 * kernel keeps intermediate values (t) in it. */
lora_status lora_workspace_size(const lora_pool* pool, int32_t max_tokens, int32_t max_segments,
                                size_t* bytes);

/* Zeroes a fresh workspace (error word and queue counters).  Call once after
 * allocating it, before its first use, on the stream that will use it. */
lora_status lora_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Scheduler step: groups the batch by adapter, on the device.
 *   "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work":
 *   SGMV groups tokens into contiguous segments that share an adapter, and the engine
 *   computes, per step, an index from each token to its adapter; "S-LoRA: Serving
 *   Thousands of Concurrent Adapters in 2026", "The Three Core Pillars": the kernel
 *   groups token slices by adapter id with no CPU involvement -- here one CTA sorts the
 *   segments by (adapter, position) with no host synchronisation.
 * Rows [seg_start[s], seg_start[s+1]) form prefill segment s (adapter seg_adapter[s]),
 * for s < S, and rows seg_start[S] + d, d < Td, are decode tokens (adapter
 * dec_adapter[d]).  S may be 0 (decode only; seg_start may then be NULL and decode
 * rows start at 0); Td may be 0 (prefill only).  T = rows of x and y.
 * Result, in the workspace (see lora_workspace_view): the adapted rows ordered by
 * ascending adapter id (batch order inside an adapter), group offsets and group
 * adapter ids, and the work lists the kernels read.  All device arrays. */
lora_status lora_segment(const lora_pool* pool, const int32_t* seg_start, const int32_t* seg_adapter,
                         int32_t S, const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                         size_t ws_bytes, void* stream);

/* Device pointers into a workspace written by lora_segment, for inspection. */
typedef struct {
    uint32_t* error_word;   /* device error bits (LORA_DERR_*)                         */
    int32_t* counts;        /* [0] adapted rows T', [1] groups G, [2] FMA chunks,
                               [3] MMA tiles                                          */
    int32_t* perm;          /* [T'] adapted rows, grouped                              */
    int32_t* grp_start;     /* [G+1] offsets into perm                                 */
    int32_t* grp_adapter;   /* [G]                                                     */
} lora_ws_view;
lora_status lora_workspace_view(const lora_pool* pool, void* ws, size_t ws_bytes, int32_t max_tokens,
                                int32_t max_segments, lora_ws_view* view);

/* BGMV (decode): token_adapter[T] gives each row's adapter (-1 = base only).
 * Groups the batch (lora_segment) and applies the delta for every problem. */
lora_status lora_bgmv(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                      const int32_t* token_adapter, int32_t T, void* ws, size_t ws_bytes,
                      void* stream);

/* SGMV (prefill): S segments, rows [seg_start[s], seg_start[s+1]) use seg_adapter[s];
 * seg_start[0] >= 0, non-decreasing, seg_start[S] <= T. */
lora_status lora_sgmv(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                      const int32_t* seg_start, const int32_t* seg_adapter, int32_t S, int32_t T,
                      void* ws, size_t ws_bytes, void* stream);

/* Mixed continuous-batching step: S prefill segments followed by Td decode tokens
 * (rows seg_start[S] + d), one grouping and one delta launch per problem batch.
 *   "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "What the engine does each
 *   step": a step's batch holds requests in prefill and in decode, and every LoRA target
 *   of every layer applies shrink then expand to all of them; "How the kernels work":
 *   SGMV suits the prefill segments and BGMV the decode tokens.  Both work classes run in
 *   the same persistent launch, its CTAs split between them by the bytes each streams. */
lora_status lora_apply_mixed(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                             const int32_t* seg_start, const int32_t* seg_adapter, int32_t S,
                             const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                             size_t ws_bytes, void* stream);

/* Delta launches only, reusing the grouping already in ws (from lora_segment with the
 * same batch; T and S = the rows of x and y and the number of prefill segments given to
 * that call).  These are the kernels the other entry points run after grouping.  With
 * S == 0 every segment is a one-row decode segment, which the CUDA-core kernel serves
 * alone (the launch lora_bgmv makes); with S > 0 the tensor-core tiles are served too. */
lora_status lora_delta_grouped(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                               int32_t T, int32_t S, void* ws, size_t ws_bytes, void* stream);

/* Shrink alone: groups the batch (token_adapter[T], -1 = base only) into ws, then writes
 *     t[p][row][j] = s_a * sum_k x_p[row, k] A_a[j, k]        (fp32, j < r_a)
 * for every problem p and every adapted row, into t (device f32 [nprob][T][r_max],
 * 16-byte aligned; entries of base-only rows and entries j >= r_a are not written).
 * Expand alone: with the grouping lora_shrink left in ws (same batch, same T),
 *     y_p[row, n] = bf16_rn(y_p[row, n] + sum_j t[p][row][j] B_a[n, j]).
 * lora_shrink followed by lora_expand computes what lora_bgmv computes, up to the fp32
 * summation order.  Between the two a caller may combine t: the sum over tensor-parallel
 * shards of their partial t (an all-reduce) is the t of the whole projection.
 *   "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "What the engine does each
 *   step": per LoRA target, v = shrink(x, A_pool[proj], idx), y += expand(v, B_pool[proj],
 *   idx, scaling).  "S-LoRA: Serving Thousands of Concurrent LoRA Adapters", "Kernels and
 *   tensor parallelism": a partition of the adapters aligned with Megatron-LM's partition
 *   of the base model, whose LoRA terms add a small exchange of the B x r intermediate.
 * Both run on the CUDA-core kernels (up to 8 projections per launch; more take several
 * launches); they serve decode and prefill rows alike (no tensor-core tiles). */
lora_status lora_shrink(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                        const int32_t* token_adapter, int32_t T, void* ws, size_t ws_bytes, float* t,
                        void* stream);
lora_status lora_expand(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                        size_t ws_bytes, const float* t, void* stream);

/* Debug export of the page-table walk (a2): for problem (layer, proj), for each group
 * g of the grouping in ws, the entries of its A block then of its B block as the
 * page-table layout above orders them (r_a each for h x h pools; r_a * ceil(d/h) for a
 * vector of length d), packed in group order into out_pages (device int32, capacity
 * `cap`).  *count_dev receives the number written (device int32). */
lora_status lora_debug_page_list(const lora_pool* pool, void* ws, size_t ws_bytes, int32_t layer,
                                 int32_t proj, int32_t* out_pages, int64_t cap, int32_t* count_dev,
                                 void* stream);

/* Debug export of the fp32 shrink result: like lora_delta_grouped for ONE problem,
 * and also writes t[row][j] = s_a * sum_k x[row,k] A_a[j,k] (fp32, the value the
 * expand consumes) into t_out (device f32 [T][r_max]) for every adapted row. */
lora_status lora_debug_delta_with_t(const lora_pool* pool, const lora_problem* prob, void* ws,
                                    size_t ws_bytes, float* t_out, void* stream);

/* Self-test of the bounded device waits every kernel uses: one thread waits on a
 * shared-memory barrier that nothing completes, gives up after limit_ns nanoseconds
 * (1 ms .. 2 s, else LORA_ETOOBIG / LORA_EINVAL) and sets LORA_DERR_TIMEOUT in the
 * workspace's error word, exactly as a kernel whose wait ran out would; the context
 * stays usable.  elapsed_ns_dev (device uint64, may be NULL) receives the time waited. */
lora_status lora_debug_wait_limit(void* ws, size_t ws_bytes, uint64_t limit_ns, uint64_t* elapsed_ns_dev,
                                  void* stream);

/* Adapter staging from host memory (side-stream prefetch).
 * "S-LoRA: Serving Thousands of Concurrent LoRA Adapters", "Host memory for adapters":
 * adapters live in host memory and the ones a batch needs are copied to the GPU ahead
 * of use.  One kernel on `stream` copies npages page rows from host_rows (pinned host
 * memory; row i is h bf16 values at host_rows + i * 2h bytes, 16-byte aligned) into
 * pool pages dst_pages[i], then sets page_table[upd_index[k]] = upd_page[k], k < nupd.
 * dst_pages, upd_index and upd_page must be pinned host memory: they are validated on
 * the host before the launch (page ids in [0, num_pages), entries in
 * [0, page_table_len)) and read by the kernel through the same pointers.  page_table
 * must be the pool's page table (passed writable).  The caller keeps the host buffers
 * alive until the kernel has finished, orders consumers after it with an event, and
 * must not stage into pages that a running kernel reads. */
lora_status lora_stage_pages(const lora_pool* pool, const void* host_rows, const int32_t* dst_pages,
                             int32_t npages, int32_t* page_table, const int64_t* upd_index,
                             const int32_t* upd_page, int64_t nupd, void* stream);

/* Adapter staging through the copy engines (the host link's DMA engines, no SM), on
 * `stream`: the same prefetch as lora_stage_pages ("S-LoRA: Serving Thousands of
 * Concurrent LoRA Adapters", "Host memory for adapters").  host_rows: pinned host memory, row i = h bf16 values for pool page
 * dst_pages[i], 16-byte aligned.  Destination pages that form runs of consecutive ids
 * (dst_pages[i + 1] = dst_pages[i] + 1) are copied straight into the pool, one
 * cudaMemcpyAsync per run, when the call has at most LORA_STAGE_MAX_RUNS runs; otherwise
 * one cudaMemcpyAsync copies all rows into `staging` (caller-owned device memory of at
 * least npages * 2h bytes, 16-byte aligned) and one kernel moves staging row i into pool
 * page dst_pages[i].  Either way a kernel on `stream` then sets page_table[upd_index[k]] =
 * upd_page[k], k < nupd, as lora_stage_pages does (no kernel if nupd = 0 and every row
 * went straight into the pool).  staging may be NULL (staging_bytes ignored) when the
 * rows form at most LORA_STAGE_MAX_RUNS runs; a non-NULL staging is always checked.
 * dst_pages, upd_index and upd_page are pinned host memory, validated on the host before
 * anything is copied or launched (LORA_EINVAL: a page id or entry out of range, staging
 * missing when needed, too small or misaligned; LORA_EALIGN: host_rows misaligned).
 * The caller keeps host_rows, staging and the index arrays alive until the work on
 * `stream` has finished, orders consumers after it with an event, and must not stage
 * into pages that a running kernel reads.  copied (a cudaEvent_t passed as void*, may be
 * NULL) is recorded on `stream` right after the copies: once it has completed, host_rows
 * may be reused. */
#define LORA_STAGE_MAX_RUNS 64
lora_status lora_stage_pages_ce(const lora_pool* pool, const void* host_rows, void* staging,
                                size_t staging_bytes, const int32_t* dst_pages, int32_t npages,
                                int32_t* page_table, const int64_t* upd_index, const int32_t* upd_page,
                                int64_t nupd, void* copied, void* stream);

/* Allocation-free BGMV.  The pages this library follows have no counterpart of this
 * call.  It is for callers that have no way to obtain device memory for a workspace:
 * a serving engine that reserves all of the GPU's memory for its own pools at start-up
 * (any later cudaMalloc fails or eats into the KV cache), a plugin or operator that a
 * host framework hands only its input and output buffers, or a step loop in which a
 * cudaMalloc -- which may synchronise the device -- is not allowed.  It computes what
 * lora_bgmv computes (the same grouping and delta kernels, chosen by the same rules),
 * with the grouping and the work lists kept in a fixed array inside the library
 * instead of a caller workspace, and it calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   - T must be <= LORA_NOALLOC_MAX_TOKENS (decode rows); larger batches return
 *     LORA_ETOOBIG and launch nothing.
 *   - The array is shared by every call in the process on a given GPU and keeps the
 *     last call's contents (the call clears what must start at zero): calls whose
 *     kernels may overlap on the GPU (different streams without ordering, or several
 *     host threads) race with each other; order them on one stream.
 *   - The first call on each device (that device current) looks up the array's device
 *     address (cudaGetSymbolAddress) and zeroes its header; make that first call before
 *     any stream capture begins.  The address is kept for the life of the process: it
 *     does not survive cudaDeviceReset or a reset of the primary context, after which
 *     this entry point must not be called again in the process.
 *   - error_bits (a device uint32, may be NULL) receives this call's device error bits
 *     (LORA_DERR_*), copied on `stream` after the kernels.
 * Every GPU that loads this library holds the array (about 0.5 MB) until the process
 * exits. */
#define LORA_NOALLOC_MAX_TOKENS 4096
lora_status lora_bgmv_noalloc(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                              const int32_t* token_adapter, int32_t T, uint32_t* error_bits,
                              void* stream);

/* Synchronises `stream`, returns the device error bits accumulated in ws since the
 * last call (in *bits) and clears them.  Returns LORA_EDEVICE if any bit was set. */
lora_status lora_get_device_error(void* ws, void* stream, uint32_t* bits);

/* The last CUDA runtime error code seen by this thread's library calls (0 = none). */
int lora_last_cuda_error(void);

/* Human-readable name of a status. */
const char* lora_status_string(lora_status s);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GB300_H */
