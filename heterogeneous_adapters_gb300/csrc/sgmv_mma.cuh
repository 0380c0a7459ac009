// Tensor-core SGMV path (prefill): one 128-row tile of one segment per work item.
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work":
// SGMV groups tokens into contiguous segments sharing an adapter and runs one small
// GEMM per segment inside a single launch, reusing the adapter's weights across the
// segment.  "S-LoRA: Serving Thousands of Concurrent LoRA Adapters": the prefill kernel
// gathers the adapter from non-contiguous pages with mixed ranks.
//
// Per item (tile of <= 128 rows of one segment, adapter a of rank r <= 128, projection of
// widths d_in x d_out; h x h in most models):
//   shrink  D1[128 x r16] (TMEM, fp32) = X[128 x d_in] . A^T, K-loop over d_in in chunks of
//           64: X chunk by TMA (128-byte swizzle), the r A-row pages' chunks by TMA (four
//           rows per gather request, rows r..r16-1 read out of range = zeros); an A row
//           longer than a page continues on its next page block (chunk kc on page kc / (h/64));
//   convert the epilogue warps read D1, scale by s and split each fp32 value exactly into
//           a bf16 pair t = hi + lo (|t - hi - lo| <= 2^-16 |t|), written back to TMEM
//           as two K-major A operands;
//   expand  for every 128-column slice of y's d_out: D2[128 x 128] = T_hi . B^T + T_lo . B^T with
//           the B-column pages' slices as an MN-major operand (TMA, 128-byte swizzle),
//           double-buffered in TMEM so the epilogue of one slice overlaps the MMA of the
//           next; the epilogue adds D2 to y (fp32) and stores bf16 rows of the tile.
// Roles (one persistent CTA per SM): warp 0 takes items from a queue shared by the
// launch's CTAs (an atomic counter in the workspace), checks their pages, hands them to
// the other roles through a small queue in shared memory and streams the shrink operands
// (x and A chunks); warp 2 streams the B^T slices, warp 3 the y tiles, warp 1 owns TMEM
// and issues the MMAs -- while it expands tile k it also issues tile k+1's shrink chunks
// as they land, so the x stream of the next tile overlaps the y stream of this one -- and
// warps 4-11 convert D1 and run the epilogue.  T lives in TMEM.  Items differ in cost by
// up to 10x (rank 8 to 64, projection widths 1024 to 14336); taken from a queue, the
// CTAs of a launch end within about one item of each other, which a fixed round-robin
// deal does not give.
// All waits are bounded; a timeout sets an error bit and the CTA unwinds.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace lora {

constexpr int kMmaThreads = 384;
constexpr int kMmaEpiWarps = 8;
constexpr int kMmaMaxProbs = 64;            // problems per launch (3 tensor maps each)
constexpr int kMmaMaxRank = 128;
// Segments of at least this many rows take the tensor-core tiles by default: the measured
// crossover of the CUDA-core and tensor-core paths (h = 4096, every segment with its own
// adapter, 2,048 rows) is 64 rows at rank 8, 32 at rank 16 and 16 from rank 32 up.  A few
// rows of low rank carry too few flops per page byte for the tile's fixed latency to pay.
__host__ __device__ constexpr int mma_min_rows_for_rank(int r) { return r >= 32 ? 16 : 512 / (r > 0 ? r : 1); }
constexpr int kMmaMinRowsByRank = -1;       // the tuning value that selects the rule above
constexpr int kMmaKChunk = 64;              // elements per shrink K chunk (128 bytes)
constexpr int kMmaNTile = 128;              // y columns per expand slice
constexpr int kMmaRowBlock = 32;            // rows per x / y TMA box
constexpr int kMmaMaxStages = 8;
constexpr int kMmaQueue = 8;                // item slots of the CTA's item queue
constexpr int kMmaQueueReaders = 3 + kMmaEpiWarps;   // warps 1, 2, 3 and the epilogue warps
constexpr uint32_t kTmemCols = 512;
// TMEM columns: D1 (shrink, fp32) 0..127, D2 (expand, fp32, two buffers) 128..383, T_hi
// and T_lo (bf16 pairs, K / 2 columns each) 384..447 and 448..511.  When every rank of the
// launch is <= 64, t takes 32 columns per half (T_lo at 416) and D1 has three buffers of
// 64 columns: 0, 64 and 448.
constexpr uint32_t kD1Col = 0, kD2Col = 128, kThiCol = 384, kTloCol = 448;
constexpr int kMmaD1Half = 64;
constexpr uint32_t kTloColSmall = 416, kD1ThirdCol = 448;
__device__ __forceinline__ uint32_t mma_nbuf(int rp_max) { return rp_max <= kMmaD1Half ? 3u : 1u; }
__device__ __forceinline__ uint32_t mma_d1_col(uint32_t b) { return b < 2 ? kD1Col + b * kMmaD1Half : kD1ThirdCol; }
__device__ __forceinline__ uint32_t mma_tlo_col(int rp_max) { return rp_max <= kMmaD1Half ? kTloColSmall : kTloCol; }
constexpr uint32_t kDerrTimeoutMma = LORA_DERR_TIMEOUT;

struct MmaParams {   // about 25 KB: kernel parameters may hold up to 32 KB
    CUtensorMap pool_map;                    // {h, num_pages}, box {64, 1}, 128B swizzle
    CUtensorMap x_map[kMmaMaxProbs];         // {d_in, T}, box {64, 32}
    CUtensorMap y_map[kMmaMaxProbs];         // {d_out, T}, box {64, 32}
    CUtensorMap y1_map[kMmaMaxProbs];        // {d_out, T}, box {64, 1}
    int32_t blk[kMmaMaxProbs];               // A block offset in units of r (l * U + pre(p))
    int16_t n_kc[kMmaMaxProbs];              // shrink K chunks: d_in / 64
    int16_t n_nt[kMmaMaxProbs];              // expand column slices: d_out / 128
    uint8_t pv_in[kMmaMaxProbs];             // pages per A row: ceil(d_in / h)
    uint8_t pv_out[kMmaMaxProbs];            // pages per B column: ceil(d_out / h)
    PoolView pool;
    char* ws;
    int32_t nprob;
    int32_t s1, s2, s3;                      // depths of the shrink, B^T and y rings
    int32_t s1_bytes, s2_bytes;              // stage sizes (y stages are 32 KB)
    int32_t rp_max;
    int32_t pad;
    uint8_t xgrp_off[kMmaMaxProbs];          // position of each problem in its shared-x group
    uint8_t xgrp_size[kMmaMaxProbs];         // size of that group
};

struct MmaSmem {
    uint32_t ring1, ring2, ring3, full1, empty1, full2, empty2, full3, empty3, d1_full, t_ready, d2_full,
        d2_empty, final_bar, tmem_slot, qfull, qempty, qitem, total;
};

__host__ __device__ inline MmaSmem mma_smem_layout(int s1, int s1_bytes, int s2, int s2_bytes, int s3) {
    MmaSmem L;
    uint32_t o = 0;
    L.ring1 = o;     o += (uint32_t)s1 * s1_bytes;
    L.ring2 = o;     o += (uint32_t)s2 * s2_bytes;
    L.ring3 = o;     o += (uint32_t)s3 * 32768;
    L.full1 = o;     o += kMmaMaxStages * 8;
    L.empty1 = o;    o += kMmaMaxStages * 8;
    L.full2 = o;     o += kMmaMaxStages * 8;
    L.empty2 = o;    o += kMmaMaxStages * 8;
    L.full3 = o;     o += kMmaMaxStages * 8;
    L.empty3 = o;    o += kMmaMaxStages * 8;
    L.d1_full = o;   o += 24;
    L.t_ready = o;   o += 8;
    L.d2_full = o;   o += 16;
    L.d2_empty = o;  o += 16;
    L.final_bar = o; o += 8;
    L.tmem_slot = o; o += 8;
    L.qfull = o;     o += kMmaQueue * 8;
    L.qempty = o;    o += kMmaQueue * 8;
    L.qitem = o;     o += kMmaQueue * 4;
    L.total = o;
    return L;
}

__host__ __device__ inline int mma_rpad(int r) { return r <= 16 ? 16 : (r + 15) / 16 * 16; }

// One work item as every role reads it; warp 0 alone checks the pages (Check) and passes
// on only the items that pass.
struct MmaItem {
    Tile tile;
    int pr;
    int rp;
    int n_kc, n_nt;   // shrink K chunks and expand column slices of the projection
    int pv_in;        // page blocks of an A row
    long long blk;    // first page-table entry of the A block (B block follows at +r pv_in)
    bool ok;
};

// Item order.  Projections that read the same x (consecutive problems with the same input,
// as q, k and v of a layer) form a group; a group's items are tile-major, so the group's
// projections of one tile are neighbouring items, dealt to neighbouring CTAs at the same
// time, and each x tile comes from DRAM once and from L2 for the others.  Across groups,
// and for a projection alone in its group, items are projection-major, so consecutive
// tiles of one segment (which read the same adapter pages) run side by side.
// W: the launch has projections whose widths differ from h; W = false compiles the h x h
// case (one page block per vector, h / 64 chunks and h / 128 slices per item).
template <bool W, bool Check>
__device__ __forceinline__ MmaItem mma_item(const MmaParams& p, const Tile* tiles, int n_tiles, uint32_t item,
                                            int lane) {
    MmaItem it;
    const uint32_t p0 = item / (uint32_t)n_tiles;          // projection-major position
    const uint32_t start = p0 - p.xgrp_off[p0];           // the group's first projection
    const uint32_t local = item - (uint32_t)n_tiles * start;
    it.tile = tiles[local / p.xgrp_size[p0]];
    it.pr = start + local % p.xgrp_size[p0];
    const int r = it.tile.rank;
    it.rp = mma_rpad(r);
    it.blk = p.pool.pt_off[it.tile.adapter] + (long long)p.blk[it.pr] * r;
    it.n_kc = W ? p.n_kc[it.pr] : p.pool.h / kMmaKChunk;
    it.n_nt = W ? p.n_nt[it.pr] : p.pool.h / kMmaNTile;
    it.pv_in = W ? p.pv_in[it.pr] : 1;
    it.ok = true;
    if (Check) {
        bool bad = false;
        const int n_ent = W ? (it.pv_in + p.pv_out[it.pr]) * r : 2 * r;   // every page of the item
        for (int e = lane; e < n_ent; e += 32) {
            const int page = p.pool.pt[it.blk + e];
            bad |= (page < 0 || page >= p.pool.num_pages);
        }
        it.ok = !__any_sync(0xffffffffu, bad);
    }
    return it;
}

// Issue the four shrink MMAs of one K chunk (stage at shared address st) into D1.
__device__ __forceinline__ void mma_shrink_chunk(uint32_t d1, uint32_t st, uint32_t idesc, int kc) {
#pragma unroll
    for (int kk = 0; kk < kMmaKChunk / 16; ++kk) {
        const uint64_t da = smem_desc(st + kk * 32, 16, 1024, 2);
        const uint64_t db = smem_desc(st + 16384 + kk * 32, 16, 1024, 2);
        tc_mma_f16(d1, da, db, idesc, (kc | kk) != 0);
    }
}

// One CTA of the tensor-core kernel (all kMmaThreads threads); `ncta` CTAs of the launch
// run this body and share its item queue (the last of them to end resets the queue).
template <bool W>
__device__ __forceinline__ void mma_cta(const MmaParams& p, unsigned char* smem_raw, uint32_t ncta) {
    // 1024-byte aligned base (the 128-byte swizzle pattern repeats every 1024 bytes)
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const MmaSmem L = mma_smem_layout(p.s1, p.s1_bytes, p.s2, p.s2_bytes, p.s3);
    const uint32_t S1 = p.s1, S2 = p.s2, S3 = p.s3;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    const WsLayout WL = ws_layout(hdr->cap_tokens, hdr->cap_segments);
    const Tile* tiles = reinterpret_cast<const Tile*>(p.ws + WL.tiles);
    const int n_tiles = hdr->counts[3];
    const uint32_t total = (uint32_t)n_tiles * (uint32_t)p.nprob;
    const int h = p.pool.h;
    // chunks and slices per page: a vector longer than a page continues on its next page
    // block (page kb of every row, then kb + 1), so chunk kc reads page kc / kc_pg
    const int kc_pg = h / kMmaKChunk, nt_pg = h / kMmaNTile;
    auto bar = [&](uint32_t off) { return smem_addr(base + off); };

    if (tid == 0) {
        for (uint32_t s = 0; s < S1; ++s) {
            mbar_init(bar(L.full1 + s * 8), 1);
            mbar_init(bar(L.empty1 + s * 8), 1);
        }
        for (uint32_t s = 0; s < S2; ++s) {
            mbar_init(bar(L.full2 + s * 8), 1);
            mbar_init(bar(L.empty2 + s * 8), 1);
        }
        for (uint32_t s = 0; s < S3; ++s) {
            mbar_init(bar(L.full3 + s * 8), 1);
            mbar_init(bar(L.empty3 + s * 8), kMmaEpiWarps);
        }
        mbar_init(bar(L.d1_full), 1);
        mbar_init(bar(L.d1_full + 8), 1);
        mbar_init(bar(L.d1_full + 16), 1);
        mbar_init(bar(L.t_ready), kMmaEpiWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L.d2_full + b * 8), 1);
            mbar_init(bar(L.d2_empty + b * 8), kMmaEpiWarps);
        }
        mbar_init(bar(L.final_bar), 1);
        for (int s = 0; s < kMmaQueue; ++s) {
            mbar_init(bar(L.qfull + s * 8), 1);
            mbar_init(bar(L.qempty + s * 8), kMmaQueueReaders);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(bar(L.tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + L.tmem_slot);
    bool ok = true;
    // The CTA's item queue: warp 0 writes the ids of the items it has taken (an id >= total
    // ends the queue), every other role reads each slot once.  False on a timeout.
    auto take = [&](uint32_t& qk, uint32_t& item) -> bool {
        const uint32_t s = qk % kMmaQueue;
        if (!mbar_wait(bar(L.qfull + s * 8), (qk / kMmaQueue) & 1, kWaitLimitNs)) return false;
        item = *reinterpret_cast<volatile const uint32_t*>(base + L.qitem + s * 4);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L.qempty + s * 8));
        ++qk;
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ item queue + shrink producer
        if (lane == 0) prefetch_tmap(&p.pool_map);
        uint32_t it = 0, qp = 0;
        unsigned int* const counter = &hdr->work_counter2;
        // the launch's queue hands out item ids in order; the id after the one in use is
        // fetched ahead (lane 0), so the atomic's round trip hides under a stream
        uint32_t ahead = 0;
        if (lane == 0) ahead = atomicAdd(counter, 1u);
        // the next item whose pages are all in the pool, or total once the queue is empty
        auto fetch = [&](MmaItem& mi) -> uint32_t {
            for (;;) {
                const uint32_t id = __shfl_sync(0xffffffffu, ahead, 0);
                if (id >= total) return total;
                if (lane == 0) ahead = atomicAdd(counter, 1u);
                mi = mma_item<W, true>(p, tiles, n_tiles, id, lane);
                if (mi.ok) return id;
                if (lane == 0) set_error(&hdr->err, LORA_DERR_PAGE);
            }
        };
        auto publish = [&](uint32_t id) -> bool {
            const uint32_t s = qp % kMmaQueue;
            if (!mbar_wait(bar(L.qempty + s * 8), ((qp / kMmaQueue) & 1) ^ 1, kWaitLimitNs)) return false;
            if (lane == 0) {
                *reinterpret_cast<volatile uint32_t*>(base + L.qitem + s * 4) = id;
                mbar_arrive(bar(L.qfull + s * 8));
            }
            __syncwarp();
            ++qp;
            return true;
        };
        MmaItem mi, mn;
        uint32_t item = fetch(mi);
        ok = publish(item);
        while (item < total && ok) {
            // the next item goes out before this one streams, so a role that reads ids ahead
            // of this stream (the MMA issuer's shrink side as soon as this item's chunks are
            // issued, the B^T and y producers) finds it published
            const uint32_t next = fetch(mn);
            if (!publish(next)) { ok = false; break; }
            const int r = mi.tile.rank, rp = mi.rp, row0 = mi.tile.row0;
            const int nblk = (mi.tile.rows + kMmaRowBlock - 1) / kMmaRowBlock;
            const void* xmap = &p.x_map[mi.pr];
            int pga[4];
            for (int kc = 0; kc < mi.n_kc; ++kc) {
                if (W ? kc % kc_pg == 0 : kc == 0) {   // page ids of the A rows' page block kc / kc_pg
                    const long long b0 = mi.blk + (W ? (long long)(kc / kc_pg) * r : 0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = lane + 32 * q;
                        pga[q] = j < r ? p.pool.pt[b0 + j] : (int)p.pool.num_pages;
                    }
                }
                const int kcol = (W ? kc % kc_pg : kc) * kMmaKChunk;   // column within the A page
                const uint32_t s = it % S1;
                if (!mbar_wait(bar(L.empty1 + s * 8), ((it / S1) & 1) ^ 1, kWaitLimitNs)) { ok = false; break; }
                const uint32_t st = bar(L.ring1 + s * p.s1_bytes);
                if (lane == 0)
                    mbar_arrive_expect_tx(bar(L.full1 + s * 8), nblk * kMmaRowBlock * 128 + rp * 128);
                __syncwarp();
                if (lane < nblk)
                    tma_load_2d(st + lane * kMmaRowBlock * 128, xmap, kc * kMmaKChunk, row0 + lane * kMmaRowBlock,
                                bar(L.full1 + s * 8));
                // A rows: groups of four real rows with one gather (lane 4k issues rows
                // 4k..4k+3, page ids taken from the next three lanes); padding rows (>= r)
                // and a ragged last group one row each, read out of range (zeros)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = lane + 32 * q;
                    const int p1 = __shfl_down_sync(0xffffffffu, pga[q], 1);
                    const int p2 = __shfl_down_sync(0xffffffffu, pga[q], 2);
                    const int p3 = __shfl_down_sync(0xffffffffu, pga[q], 3);
                    if (j < rp) {
                        if ((j | 3) < r) {
                            if ((j & 3) == 0)
                                tma_gather4(st + 16384 + j * 128, &p.pool_map, kcol, pga[q], p1, p2, p3,
                                            bar(L.full1 + s * 8));
                        } else {
                            tma_load_2d(st + 16384 + j * 128, &p.pool_map, kcol, pga[q], bar(L.full1 + s * 8));
                        }
                    }
                }
                ++it;
            }
            item = next;
            mi = mn;
        }
        if (!ok && lane == 0) set_error(&hdr->err, kDerrTimeoutMma);
        if (lane == 0) {   // let every stage this warp filled land before the CTA can exit
            for (uint32_t k = it > S1 ? it - S1 : 0; k < it; ++k)
                mbar_wait(bar(L.full1 + (k % S1) * 8), (k / S1) & 1, 100000000ull);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------------ B^T producer
        uint32_t it2 = 0, qk = 0, item = 0;
        while (ok) {
            if (!take(qk, item)) { ok = false; break; }
            if (item >= total) break;
            const MmaItem mi = mma_item<W, false>(p, tiles, n_tiles, item, lane);
            const int r = mi.tile.rank, rp = mi.rp;
            int pgb[4];
            for (int nt = 0; nt < mi.n_nt; ++nt, ++it2) {
                if (W ? nt % nt_pg == 0 : nt == 0) {   // page ids of the B columns' page block nt / nt_pg
                    const long long b0 = mi.blk + (W ? (long long)(mi.pv_in + nt / nt_pg) * r : (long long)r);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = lane + 32 * q;
                        pgb[q] = j < r ? p.pool.pt[b0 + j] : (int)p.pool.num_pages;
                    }
                }
                const int ncol = (W ? nt % nt_pg : nt) * kMmaNTile;   // column within the B page
                // B^T slice: K rows = pages j, N = 128 columns as two 64-column atoms;
                // atom (j / 8, nb) at (j / 8) * 2048 + nb * 1024, row j % 8 at +128 (j % 8)
                const uint32_t s = it2 % S2;
                if (!mbar_wait(bar(L.empty2 + s * 8), ((it2 / S2) & 1) ^ 1, kWaitLimitNs)) { ok = false; break; }
                const uint32_t st = bar(L.ring2 + s * p.s2_bytes);
                if (lane == 0) mbar_arrive_expect_tx(bar(L.full2 + s * 8), rp * 256);
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = lane + 32 * q;
                    const int p1 = __shfl_down_sync(0xffffffffu, pgb[q], 1);
                    const int p2 = __shfl_down_sync(0xffffffffu, pgb[q], 2);
                    const int p3 = __shfl_down_sync(0xffffffffu, pgb[q], 3);
                    if (j < rp) {
                        const uint32_t dst = st + (j >> 3) * 2048 + (j & 7) * 128;
                        if ((j | 3) < r) {
                            if ((j & 3) == 0) {
                                tma_gather4(dst, &p.pool_map, ncol, pgb[q], p1, p2, p3, bar(L.full2 + s * 8));
                                tma_gather4(dst + 1024, &p.pool_map, ncol + 64, pgb[q], p1, p2, p3,
                                            bar(L.full2 + s * 8));
                            }
                        } else {
                            tma_load_2d(dst, &p.pool_map, ncol, pgb[q], bar(L.full2 + s * 8));
                            tma_load_2d(dst + 1024, &p.pool_map, ncol + 64, pgb[q], bar(L.full2 + s * 8));
                        }
                    }
                }
            }
        }
        if (!ok && lane == 0) set_error(&hdr->err, kDerrTimeoutMma);
        if (lane == 0) {
            for (uint32_t k = it2 > S2 ? it2 - S2 : 0; k < it2; ++k)
                mbar_wait(bar(L.full2 + (k % S2) * 8), (k / S2) & 1, 100000000ull);
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------------ y producer
        uint32_t it3 = 0, qk = 0, item = 0;
        while (ok) {
            if (!take(qk, item)) { ok = false; break; }
            if (item >= total) break;
            const MmaItem mi = mma_item<W, false>(p, tiles, n_tiles, item, lane);
            const int row0 = mi.tile.row0;
            const int nblk = (mi.tile.rows + kMmaRowBlock - 1) / kMmaRowBlock;
            const void* ymap = &p.y_map[mi.pr];
            for (int nt = 0; nt < mi.n_nt; ++nt, ++it3) {
                // y tile: half hf (64 columns) at hf * 16 KB, 32-row block b at + b * 4 KB
                const uint32_t s = it3 % S3;
                if (!mbar_wait(bar(L.empty3 + s * 8), ((it3 / S3) & 1) ^ 1, kWaitLimitNs)) { ok = false; break; }
                const uint32_t st = bar(L.ring3 + s * 32768);
                if (lane == 0) mbar_arrive_expect_tx(bar(L.full3 + s * 8), 2 * nblk * kMmaRowBlock * 128);
                __syncwarp();
                if (lane < 2 * nblk) {
                    const int hf = lane & 1, b = lane >> 1;
                    tma_load_2d(st + hf * 16384 + b * kMmaRowBlock * 128, ymap, nt * kMmaNTile + hf * 64,
                                row0 + b * kMmaRowBlock, bar(L.full3 + s * 8));
                }
            }
        }
        if (!ok && lane == 0) set_error(&hdr->err, kDerrTimeoutMma);
        if (lane == 0) {
            for (uint32_t k = it3 > S3 ? it3 - S3 : 0; k < it3; ++k)
                mbar_wait(bar(L.full3 + (k % S3) * 8), (k / S3) & 1, 100000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // Two cursors over the CTA's items, which the shrink side reads from the queue in
        // order.  The shrink side issues an item's K chunks into a D1 buffer as they land;
        // the expand side follows, starting an item once its shrink is issued and its t
        // converted (which frees that D1 buffer).  With three D1 buffers (every rank <= 64)
        // the shrink runs up to three items ahead of the expand, so the x stream of items
        // with a short expand (k and v of grouped-query attention, down) goes on under a
        // long one (gate, up); with one buffer, one item ahead.
        const uint32_t nbuf = mma_nbuf(p.rp_max);
        const uint32_t tlo = mma_tlo_col(p.rp_max);
        uint32_t it1 = 0, it2 = 0, tcount = 0, g = 0, qk = 0;
        uint32_t s_seq = 0;      // items whose shrink is issued (and committed to d1_full)
        uint32_t e_seq = 0;      // items whose expand has started
        bool s_busy = false;     // item s_seq's shrink is under way
        bool q_end = false;      // the queue's end has been read
        MmaItem sh;              // item s_seq
        int s_kc = 0;            // its chunks issued
        uint32_t s_idesc = 0;
        uint32_t f0 = 0, f1 = 0, f2 = 0;   // items e_seq .. e_seq + 2 (shrunk or under way): n_nt << 8 | rp
        // Advances the shrink side: starts the next item while a D1 buffer is free and
        // issues the chunks that have landed; `block` waits for every chunk of one item.
        // False on a timeout.
        auto shrink_step = [&](bool block) -> bool {
            for (;;) {
                if (!s_busy) {
                    if (q_end || s_seq >= e_seq + nbuf) return true;
                    uint32_t id = total;
                    if (!take(qk, id)) return false;
                    if (id >= total) {
                        q_end = true;
                        return true;
                    }
                    sh = mma_item<W, false>(p, tiles, n_tiles, id, lane);
                    s_idesc = idesc_bf16(128, sh.rp, 0, 0);
                    s_kc = 0;
                    s_busy = true;
                    const uint32_t packed = (uint32_t)sh.n_nt << 8 | (uint32_t)sh.rp;
                    const uint32_t fi = s_seq - e_seq;
                    if (fi == 0) f0 = packed;
                    else if (fi == 1) f1 = packed;
                    else f2 = packed;
                }
                const uint32_t b1 = s_seq % nbuf;
                while (s_kc < sh.n_kc) {
                    const uint32_t s1 = it1 % S1;
                    if (block) {
                        if (!mbar_wait(bar(L.full1 + s1 * 8), (it1 / S1) & 1, kWaitLimitNs)) return false;
                    } else if (!mbar_test_wait(bar(L.full1 + s1 * 8), (it1 / S1) & 1)) {
                        return true;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        mma_shrink_chunk(tmem + mma_d1_col(b1), bar(L.ring1 + s1 * p.s1_bytes), s_idesc, s_kc);
                        tc_commit(bar(L.empty1 + s1 * 8));
                    }
                    __syncwarp();
                    ++s_kc;
                    ++it1;
                }
                if (lane == 0) tc_commit(bar(L.d1_full + b1 * 8));
                __syncwarp();
                s_busy = false;
                ++s_seq;
                if (block) return true;
            }
        };
        while (ok) {
            // the next item's shrink, completed (a wait) if still under way
            while (ok && e_seq >= s_seq && (s_busy || !q_end))
                if (!shrink_step(true)) ok = false;
            if (!ok || e_seq >= s_seq) break;   // a timeout, or no item left
            // its t is in TMEM once the convert has read its D1 buffer
            if (!mbar_wait(bar(L.t_ready), tcount & 1, kWaitLimitNs)) { ok = false; break; }
            ++tcount;
            const int rp = (int)(f0 & 0xffu), n_nt = (int)(f0 >> 8);
            f0 = f1;
            f1 = f2;
            ++e_seq;
            tc_fence_after();
            const uint32_t id_expand = idesc_bf16(128, kMmaNTile, 0, 1);
            for (int nt = 0; nt < n_nt && ok; ++nt, ++g, ++it2) {
                const uint32_t s = it2 % S2;
                const uint32_t b = g & 1;
                if (!mbar_wait(bar(L.full2 + s * 8), (it2 / S2) & 1, kWaitLimitNs)) { ok = false; break; }
                if (!mbar_wait(bar(L.d2_empty + b * 8), ((g >> 1) & 1) ^ 1, kWaitLimitNs)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t st = bar(L.ring2 + s * p.s2_bytes);
                    const uint32_t d2 = tmem + kD2Col + b * kMmaNTile;
                    for (int ks = 0; ks < rp / 16; ++ks) {
                        const uint64_t dbt = smem_desc(st + ks * 4096, 1024, 2048, 2);
                        tc_mma_f16_ts(d2, tmem + kThiCol + ks * 8, dbt, id_expand, ks != 0);
                        tc_mma_f16_ts(d2, tmem + tlo + ks * 8, dbt, id_expand, 1);
                    }
                    tc_commit(bar(L.empty2 + s * 8));
                    tc_commit(bar(L.d2_full + b * 8));
                }
                __syncwarp();
                // shrink chunks that have already landed (a test, not a wait: a suspending
                // wait here would hold the expand back for a whole shrink)
                if (!shrink_step(false)) ok = false;
            }
        }
        if (!ok && lane == 0) set_error(&hdr->err, kDerrTimeoutMma);
        // every MMA issued by this thread must be complete before TMEM is freed
        if (lane == 0) {
            tc_commit(bar(L.final_bar));
            mbar_wait(bar(L.final_bar), 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ convert + epilogue
        const int e = warp - 4;                 // 0..7
        const int quad = warp & 3;              // TMEM lanes 32 quad .. 32 quad + 31
        const int half = e >> 2;                // column half of each slice
        const int m = quad * 32 + lane;         // tile row of this thread
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t nbuf = mma_nbuf(p.rp_max);   // D1 buffers and T_lo column, as the MMA issuer
        const uint32_t tlo = mma_tlo_col(p.rp_max);
        uint32_t tcount = 0, g = 0, qk = 0, item = 0;
        bool stored = false;
        while (ok) {
            if (!take(qk, item)) { ok = false; break; }
            if (item >= total) break;
            const MmaItem mi = mma_item<W, false>(p, tiles, n_tiles, item, lane);
            const int rp = mi.rp, rows = mi.tile.rows, row0 = mi.tile.row0;
            const float scale = p.pool.scales[mi.tile.adapter];
            const bool live = m < rows;
            const bool block_full = quad * kMmaRowBlock + kMmaRowBlock <= rows;
            const bool block_part = !block_full && quad * kMmaRowBlock < rows;
            // ---- convert D1 -> T_hi, T_lo in TMEM (bf16 pairs, column c / 2 holds k = c, c + 1)
            const uint32_t b1 = tcount % nbuf;
            if (!mbar_wait(bar(L.d1_full + b1 * 8), (tcount / nbuf) & 1, kWaitLimitNs)) { ok = false; break; }
            tc_fence_after();
            // the rp / 16 column chunks of D1 are split between the two warpgroups
            const int nck = rp / 16;
            const int ck_begin = half ? (nck + 1) / 2 : 0, ck_end = half ? nck : (nck + 1) / 2;
            for (int c0 = ck_begin * 16; c0 < ck_end * 16; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + lane_base + mma_d1_col(b1) + c0, v);
                tmem_ld_wait();
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float a = v[2 * i] * scale, b = v[2 * i + 1] * scale;
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
                    const float ha = __low2float(h2), hb = __high2float(h2);
                    const __nv_bfloat162 l2 = __floats2bfloat162_rn(a - ha, b - hb);
                    hi[i] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[i] = *reinterpret_cast<const uint32_t*>(&l2);
                }
                tmem_st8(tmem + lane_base + kThiCol + c0 / 2, hi);
                tmem_st8(tmem + lane_base + tlo + c0 / 2, lo);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L.t_ready));
            ++tcount;
            // ---- expand epilogue over the column slices: y (in the y ring) += D2
            for (int nt = 0; nt < mi.n_nt; ++nt, ++g) {
                const uint32_t b = g & 1;
                const uint32_t ys = g % S3;
                if (!mbar_wait(bar(L.d2_full + b * 8), (g >> 1) & 1, kWaitLimitNs)) { ok = false; break; }
                tc_fence_after();
                float acc[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[16];
                    tmem_ld16(tmem + lane_base + kD2Col + b * kMmaNTile + half * 64 + q * 16, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[q * 16 + i] = v[i];
                }
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L.d2_empty + b * 8));
                if (!mbar_wait(bar(L.full3 + ys * 8), (g / S3) & 1, kWaitLimitNs)) { ok = false; break; }
                // this warp's box: rows 32 quad .. +31 of column half `half` (128-byte swizzle)
                unsigned char* yrow = base + L.ring3 + ys * 32768 + half * 16384 + m * 128;
                if (live) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4* ptr = reinterpret_cast<uint4*>(yrow + ((c ^ (m & 7)) << 4));
                        float y8[8];
                        unpack8(*ptr, y8);
                        uint4 o;
                        o.x = pack2(y8[0] + acc[8 * c + 0], y8[1] + acc[8 * c + 1]);
                        o.y = pack2(y8[2] + acc[8 * c + 2], y8[3] + acc[8 * c + 3]);
                        o.z = pack2(y8[4] + acc[8 * c + 4], y8[5] + acc[8 * c + 5]);
                        o.w = pack2(y8[6] + acc[8 * c + 6], y8[7] + acc[8 * c + 7]);
                        *ptr = o;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                const int col = nt * kMmaNTile + half * 64;
                if (block_full) {
                    if (lane == 0) {
                        tma_store_2d(&p.y_map[mi.pr], col, row0 + quad * kMmaRowBlock,
                                     smem_addr(base + L.ring3 + ys * 32768 + half * 16384 + quad * 4096));
                        stored = true;
                    }
                } else if (block_part && live) {
                    tma_store_2d(&p.y1_map[mi.pr], col, row0 + m, smem_addr(yrow));
                    stored = true;
                }
                // one commit group per slice; the slot of the previous slice is released
                // once its stores have read shared memory, so a store overlaps the next slice
                bulk_commit();
                bulk_wait_read1();
                __syncwarp();
                if (lane == 0 && g > 0) mbar_arrive(bar(L.empty3 + ((g - 1) % S3) * 8));
            }
        }
        if (!ok && lane == 0) set_error(&hdr->err, kDerrTimeoutMma);
        if (stored) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    // the last of the launch's CTAs to end resets the queue for the next launch (every CTA
    // has taken its last id by now; the next launch on the stream starts after this one)
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&hdr->done_counter, 1u) == ncta - 1) {
            atomicExch(&hdr->work_counter2, 0u);
            atomicExch(&hdr->done_counter, 0u);
        }
    }
}

template <bool W>
__global__ void __launch_bounds__(kMmaThreads, 1) sgmv_mma_kernel(const __grid_constant__ MmaParams p) {
    extern __shared__ __align__(1024) unsigned char mma_smem_raw[];
    mma_cta<W>(p, mma_smem_raw, gridDim.x);
}

}  // namespace lora
