// Scheduler step on the device: group the batch by adapter (one CTA, no host sync).
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work":
// SGMV sorts or groups tokens so each contiguous segment shares an adapter, and
// engines precompute per step an index from tokens to adapters.  "S-LoRA: Serving
// Thousands of Concurrent Adapters in 2026", "The Three Core Pillars": the fused
// kernel groups token slices by target adapter id with no CPU intervention.
//
// Every prefill segment and every decode token is a "segment" (a decode token is a
// segment of one row).  Adapted segments are ordered by the unique key
// (adapter id, segment index); since segments are listed in row order, this is a
// stable sort of the adapted rows by adapter id.  Base-only (-1) and invalid
// segments are left out (invalid ones raise a device error bit).
//
// Outputs (workspace): perm / grp_start / grp_adapter (the grouping), the row list
// and chunk list of the CUDA-core path (segments shorter than mma_min, at most kChunk
// rows of one adapter per chunk) and the tile list of the tensor-core path (segments
// of at least mma_min rows, 128 rows per tile).
#pragma once
#include "common.cuh"
#include "sgmv_mma.cuh"

namespace lora {

constexpr int kSegThreads = 1024;
constexpr int kKeyTile = 2048;

struct SegParams {
    PoolView pool;
    const int32_t* seg_start;
    const int32_t* seg_adapter;
    const int32_t* dec_adapter;
    char* ws;
    WsLayout L;
    int32_t S;
    int32_t Td;
    int32_t T;
    int32_t mma_min;   // 0: every segment goes to the CUDA-core path; > 0: segments of at
                       // least this many rows take the tensor-core tiles; -1: the rank rule
                       // mma_min_rows_for_rank
    int32_t mma_max_rank;   // segments whose adapter rank exceeds this use the CUDA-core path
    int32_t L_tokens;  // the (max_tokens, max_segments) that L was computed from
    int32_t L_segments;
    int32_t smem_segs; // > 0: the per-segment scratch arrays live in dynamic shared memory
    int32_t pad;
};

// Dynamic shared memory of the grouping kernel when the per-segment arrays fit there
// (key 8 B + six int arrays per segment).
constexpr int kSegSmemMax = 1536;
__host__ __device__ constexpr size_t seg_smem_bytes(int n) { return (size_t)(n + 1) * 32 + 64; }

// Whether a segment of len rows of an adapter of rank r takes the tensor-core tiles.
__device__ __forceinline__ bool mma_tile(const SegParams& p, int len, int r) {
    if (p.mma_min == 0 || r > p.mma_max_rank) return false;
    return len >= (p.mma_min > 0 ? p.mma_min : mma_min_rows_for_rank(r));
}

__global__ void __launch_bounds__(kSegThreads) segment_kernel(const SegParams p) {
    __shared__ int scan_smem[33];
    __shared__ long long key_tile[kKeyTile];
    __shared__ int n_adapted_s;
    __shared__ unsigned long long weight_s[4];   // rows[2], page_rows[2] of the header

    const int tid = threadIdx.x, nthr = blockDim.x;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    // per-segment scratch: in shared memory for small batches (the phases below hand data
    // to each other through it), else in the workspace
    extern __shared__ __align__(16) unsigned char seg_smem[];
    long long* key;
    int32_t *sbeg, *slen, *sorted, *pos, *fpos, *gfirst;
    if (p.smem_segs > 0) {
        const int m = p.smem_segs + 1;
        key = reinterpret_cast<long long*>(seg_smem);
        sbeg = reinterpret_cast<int32_t*>(key + m);
        slen = sbeg + m;
        sorted = slen + m;
        pos = sorted + m;
        fpos = pos + m;
        gfirst = fpos + m;
    } else {
        key = reinterpret_cast<long long*>(p.ws + p.L.seg_key);
        sbeg = reinterpret_cast<int32_t*>(p.ws + p.L.seg_begin);
        slen = reinterpret_cast<int32_t*>(p.ws + p.L.seg_len);
        sorted = reinterpret_cast<int32_t*>(p.ws + p.L.sorted);
        pos = reinterpret_cast<int32_t*>(p.ws + p.L.pos);
        fpos = reinterpret_cast<int32_t*>(p.ws + p.L.fpos);
        gfirst = reinterpret_cast<int32_t*>(p.ws + p.L.gfirst);
    }
    int32_t* perm = reinterpret_cast<int32_t*>(p.ws + p.L.perm);
    int32_t* grp_start = reinterpret_cast<int32_t*>(p.ws + p.L.grp_start);
    int32_t* grp_adapter = reinterpret_cast<int32_t*>(p.ws + p.L.grp_adapter);
    int32_t* fma_rows = reinterpret_cast<int32_t*>(p.ws + p.L.fma_rows);
    Chunk* chunks = reinterpret_cast<Chunk*>(p.ws + p.L.chunks);
    Tile* tiles = reinterpret_cast<Tile*>(p.ws + p.L.tiles);
    const PoolView& P = p.pool;
    const long long kNone = 0x7fffffffffffffffLL;

    const int n = p.S + p.Td;
    if (tid == 0) {
        n_adapted_s = 0;
        weight_s[0] = weight_s[1] = weight_s[2] = weight_s[3] = 0;
    }
    __syncthreads();
    const int dec_base = p.S > 0 ? p.seg_start[p.S] : 0;

    // 1. per-segment validation and sort key
    uint32_t errbits = 0;
    int my_adapted = 0;
    for (int i = tid; i < n; i += nthr) {
        int b, e, a;
        if (i < p.S) {
            b = p.seg_start[i];
            e = p.seg_start[i + 1];
            a = p.seg_adapter[i];
        } else {
            b = dec_base + (i - p.S);
            e = b + 1;
            a = p.dec_adapter[i - p.S];
        }
        bool ok = true;
        if (b < 0 || e < b || e > p.T) {
            errbits |= LORA_DERR_SEGMENT;
            ok = false;
        }
        if (ok && a != -1) {
            if (a < -1 || a >= P.num_adapters) {
                errbits |= LORA_DERR_ADAPTER;
                ok = false;
            } else {
                const int r = P.ranks[a];
                if (r < 1 || r > P.r_max) {
                    errbits |= LORA_DERR_RANK;
                    ok = false;
                } else {
                    const long long off = P.pt_off[a];
                    const long long need = (long long)P.num_layers * P.units * r;
                    if (off < 0 || off + need > P.pt_len) {
                        errbits |= LORA_DERR_PTBLOCK;
                        ok = false;
                    }
                }
            }
        }
        const bool adapted = ok && a >= 0 && e > b;
        key[i] = adapted ? (((long long)a << 32) | (long long)i) : kNone;
        sbeg[i] = b;
        slen[i] = adapted ? e - b : 0;
        my_adapted += adapted;
    }
    if (errbits) set_error(&hdr->err, errbits);
    if (my_adapted) atomicAdd(&n_adapted_s, my_adapted);
    __syncthreads();
    const int n_ad = n_adapted_s;

    // 2. rank of every adapted segment = number of smaller keys (keys are unique)
    for (int i0 = 0; i0 < n; i0 += nthr) {
        const int i = i0 + tid;
        const long long my = i < n ? key[i] : kNone;
        int rank = 0;
        for (int k0 = 0; k0 < n; k0 += kKeyTile) {
            __syncthreads();
            for (int k = tid; k < kKeyTile; k += nthr) key_tile[k] = (k0 + k < n) ? key[k0 + k] : kNone;
            __syncthreads();
            if (my != kNone) {
                const int kn = min(kKeyTile, n - k0);
                for (int k = 0; k < kn; ++k) rank += key_tile[k] < my;
            }
        }
        if (my != kNone) sorted[rank] = i;
    }
    __syncthreads();

    // 3. positions of each sorted segment in the grouped row order, group starts,
    //    and positions in the CUDA-core row list
    int carry_pos = 0, carry_g = 0, carry_f = 0, carry_t = 0;
    for (int q0 = 0; q0 < n_ad; q0 += nthr) {
        const int q = q0 + tid;
        const bool valid = q < n_ad;
        const int seg = valid ? sorted[q] : 0;
        const int a = valid ? (int)(key[seg] >> 32) : 0;
        const int len = valid ? slen[seg] : 0;
        const int prev_a = (valid && q > 0) ? (int)(key[sorted[q - 1]] >> 32) : -1;
        const int flag = (valid && (q == 0 || a != prev_a)) ? 1 : 0;
        const bool is_mma = valid && mma_tile(p, len, P.ranks[a]);
        const int flen = (valid && !is_mma) ? len : 0;
        const int ntile = is_mma ? (len + kTileRows - 1) / kTileRows : 0;
        int tot_pos, tot_g, tot_f, tot_t;
        const int e_pos = block_exclusive_scan(len, scan_smem, &tot_pos) + carry_pos;
        const int e_g = block_exclusive_scan(flag, scan_smem, &tot_g) + carry_g;
        const int e_f = block_exclusive_scan(flen, scan_smem, &tot_f) + carry_f;
        const int e_t = block_exclusive_scan(ntile, scan_smem, &tot_t) + carry_t;
        if (valid) {
            pos[q] = e_pos;
            fpos[q] = e_f;
            if (flag) {
                grp_start[e_g] = e_pos;
                grp_adapter[e_g] = a;
                gfirst[e_g] = q;
            }
            const int r = P.ranks[a];
            if (ntile > 0) {   // x read + y read and write, plus the pages once per tile
                atomicAdd(&weight_s[1], (unsigned long long)len);
                atomicAdd(&weight_s[3], (unsigned long long)r * ntile);
            }
            for (int k = 0; k < ntile; ++k) {
                Tile tl;
                tl.adapter = a;
                tl.row0 = sbeg[seg] + k * kTileRows;
                tl.rows = min(kTileRows, len - k * kTileRows);
                tl.rank = r;
                tiles[e_t + k] = tl;
            }
        }
        carry_pos += tot_pos;
        carry_g += tot_g;
        carry_f += tot_f;
        carry_t += tot_t;
    }
    const int G = carry_g;
    if (tid == 0) {
        grp_start[G] = carry_pos;
        gfirst[G] = n_ad;
        fpos[n_ad] = carry_f;
    }
    __syncthreads();

    // 4. row lists: grouped order (perm) and the CUDA-core subset (fma_rows)
    const int lane = tid & 31, warp = tid >> 5, nwarp = nthr >> 5;
    for (int q = warp; q < n_ad; q += nwarp) {
        const int seg = sorted[q];
        const int b = sbeg[seg], len = slen[seg];
        const int a = (int)(key[seg] >> 32);
        const bool is_mma = mma_tile(p, len, P.ranks[a]);
        const int pq = pos[q], fq = fpos[q];
        for (int t = lane; t < len; t += 32) {
            perm[pq + t] = b + t;
            if (!is_mma) fma_rows[fq + t] = b + t;
        }
    }

    // 5. CUDA-core chunks: per group, its CUDA-core rows cut into pieces of kChunk.  Groups
    //    are listed by descending rank (ties: ascending adapter id) so that the largest
    //    work items are taken first from the queue and the tail of a launch is short.
    int32_t* gorder = sorted;   // the sorted-segment list is no longer needed
    __syncthreads();
    for (int g = tid; g < G; g += nthr)   // group keys, reusing the segment-key array
        key[g] = ((long long)(LORA_MAX_RANK - P.ranks[grp_adapter[g]]) << 32) | g;
    __syncthreads();
    for (int g0 = 0; g0 < G; g0 += nthr) {
        const int g = g0 + tid;
        const long long my = g < G ? key[g] : kNone;
        int rank = 0;
        for (int k0 = 0; k0 < G; k0 += kKeyTile) {
            __syncthreads();
            for (int k = tid; k < kKeyTile; k += nthr) key_tile[k] = (k0 + k < G) ? key[k0 + k] : kNone;
            __syncthreads();
            if (g < G) {
                const int kn = min(kKeyTile, G - k0);
                for (int k = 0; k < kn; ++k) rank += key_tile[k] < my;
            }
        }
        if (g < G) gorder[rank] = g;
    }
    __syncthreads();
    int carry_c = 0;
    for (int i0 = 0; i0 < G; i0 += nthr) {
        const int i = i0 + tid;
        const int g = i < G ? gorder[i] : 0;
        int first = 0, cnt = 0;
        if (i < G) {
            first = fpos[gfirst[g]];
            cnt = fpos[gfirst[g + 1]] - first;
        }
        const int nch = (cnt + kChunk - 1) / kChunk;
        int tot;
        const int base = block_exclusive_scan(nch, scan_smem, &tot) + carry_c;
        if (i < G) {
            const int a = grp_adapter[g];
            const int r = P.ranks[a];
            const float sc = P.scales[a];
            const long long ptb = P.pt_off[a];
            if (nch > 0) {   // rows read and written, plus the pages once per chunk
                atomicAdd(&weight_s[0], (unsigned long long)cnt);
                atomicAdd(&weight_s[2], (unsigned long long)r * nch);
            }
            for (int c = 0; c < nch; ++c) {
                Chunk ch;
                ch.adapter = a;
                ch.begin = first + c * kChunk;
                ch.count = min(kChunk, cnt - c * kChunk);
                ch.rank = r;
                ch.scale = sc;
                ch.pt_base = ptb;
                ch.pad = 0;
                for (int t = 0; t < kChunk; ++t) ch.rows[t] = t < ch.count ? fma_rows[ch.begin + t] : 0;
                chunks[base + c] = ch;
            }
        }
        carry_c += tot;
    }
    if (tid == 0) {
        hdr->counts[0] = carry_pos;
        hdr->counts[1] = G;
        hdr->counts[2] = carry_c;
        hdr->counts[3] = carry_t;
        hdr->work_counter = 0;
        hdr->work_counter2 = 0;
        hdr->done_counter = 0;
        hdr->cap_tokens = p.L_tokens;
        hdr->cap_segments = p.L_segments;
    }
    __syncthreads();
    if (tid == 0) {
        hdr->rows[0] = weight_s[0];
        hdr->rows[1] = weight_s[1];
        hdr->page_rows[0] = weight_s[2];
        hdr->page_rows[1] = weight_s[3];
    }
}

// Debug export of the page-table walk: for each group, its A-row pages then its
// B-column pages for one problem, packed in group order.  blk: the A block's offset in
// units of r (layer * U + pre(p)); vec_units: pages per A row plus pages per B column.
__global__ void __launch_bounds__(kSegThreads)
    page_list_kernel(const PoolView P, const char* ws, int32_t blk, int32_t vec_units, int32_t* out,
                     int64_t cap, int32_t* count_out) {
    __shared__ int scan_smem[33];
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    const WsLayout L = ws_layout(hdr->cap_tokens, hdr->cap_segments);
    const int32_t* grp_adapter = reinterpret_cast<const int32_t*>(ws + L.grp_adapter);
    const int G = hdr->counts[1];
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += blockDim.x) {
        const int g = g0 + threadIdx.x;
        const int a = g < G ? grp_adapter[g] : 0;
        const int r = g < G ? P.ranks[a] : 0;
        int tot;
        const int base = block_exclusive_scan(vec_units * r, scan_smem, &tot) + carry;
        if (g < G) {
            const long long src = P.pt_off[a] + (long long)blk * r;
            for (int e = 0; e < vec_units * r; ++e)
                if (base + e < cap) out[base + e] = P.pt[src + e];
        }
        carry += tot;
    }
    if (threadIdx.x == 0) *count_out = carry;
}

}  // namespace lora
