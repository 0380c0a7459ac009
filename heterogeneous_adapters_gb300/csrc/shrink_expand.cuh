// Shrink and expand as two separate launches, t in a caller buffer between them.
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "What the engine does each
// step": per LoRA target, v = shrink(x, A_pool[proj], idx) and then
// y += expand(v, B_pool[proj], idx, scaling) -- two steps with v between them.  "S-LoRA:
// Serving Thousands of Concurrent LoRA Adapters", "Kernels and tensor parallelism": with
// the model split across GPUs as Megatron-LM splits it, each GPU holds a part of every
// adapter, and the LoRA terms add a small exchange of the B x r intermediate to the base
// model's communication.  Between these two launches a caller can sum the partial t of
// several shards (an all-reduce), which the one-launch kernels cannot offer.
//
//   shrink (lora_shrink_kernel): item = (projection, chunk, 8 consecutive A rows j).
//     Warp w computes t[row][j0 + w] = s * sum_k x[row,k] A[j0+w,k] over the full row
//     (no partial sums cross CTAs) and writes it, fp32, to t.
//   expand (lora_expand_kernel): item = (projection, chunk, 512-column slice of y).
//     Every B column's slice is read once; 4 groups of threads take every 4th j, their
//     sums meet in shared memory, and y = bf16_rn(y + sum) is stored for the slice.
//     Per item, the page ids, t values and y rows come in one round trip, then the B
//     vectors, up to 16 per thread in flight.
// A chunk whose A or B pages are out of range is skipped (its t entries and y rows are
// left as they are) and reported in the device error word.
#pragma once
#include "common.cuh"

namespace lora {

constexpr int kSxMaxProbs = 8;           // projections of one launch at most
constexpr int kSxRows = 8;               // A rows per shrink item (one per warp)
constexpr int kSxVecs = 64;              // 16-byte column vectors per expand item (512 columns)
constexpr int kSxThreads = 256;

struct ShrinkExpandParams {
    PoolView pool;
    char* ws;
    float* t;             // [problem][token row][r_max] fp32 (the caller's buffer)
    int32_t T;            // rows of the batch
    int32_t nprob;
    int32_t out_blocks;   // the most output page blocks of the launch's projections
    int32_t pad;
    ProbDesc probs[kSxMaxProbs];
};

// Shrink.  Per item every lane first issues the loads of its share of its warp's A row
// (up to kSxLoads 16-byte vectors at once), the CTA meanwhile stages the chunk's x rows
// in shared memory, and the dot products are then taken from registers and shared memory.
constexpr int kSxLoads = 16;

// W: the pool has projections whose widths differ from h (see the ring kernel); W = false
// compiles the h x h case with one page block per vector.
template <bool W>
__global__ void __launch_bounds__(kSxThreads) lora_shrink_kernel(const __grid_constant__ ShrinkExpandParams p) {
    extern __shared__ __align__(16) unsigned char split_smem[];   // x rows: kChunk * h bf16
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    const WsLayout WL = ws_layout(hdr->cap_tokens, hdr->cap_segments);
    const Chunk* chunks = reinterpret_cast<const Chunk*>(p.ws + WL.chunks);
    float* tbuf = p.t;
    const int n_chunks = hdr->counts[2];
    const int T = p.T;
    const PoolView& P = p.pool;
    const int h8 = P.h >> 3, r_max = P.r_max;
    const int n_js = (r_max + kSxRows - 1) / kSxRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4* xs = reinterpret_cast<uint4*>(split_smem);
    const long long total = (long long)p.nprob * n_chunks * n_js;
    auto chunk_of = [&](long long it) { return (int)((it / n_js) % n_chunks); };
    Chunk next;
    if (blockIdx.x < total) next = chunks[chunk_of(blockIdx.x)];
    for (long long item = blockIdx.x; item < total; item += gridDim.x) {
        const int js = (int)(item % n_js);
        const int pr = (int)(item / ((long long)n_js * n_chunks));
        const Chunk ch = next;   // loaded while the previous item was being computed
        if (item + gridDim.x < total) next = chunks[chunk_of(item + gridDim.x)];
        const int r = ch.rank;
        if (js * kSxRows >= r) continue;   // this adapter has fewer rows
        const ProbDesc pd = p.probs[pr];
        const long long a0 = ch.pt_base + (long long)pd.blk * r;   // A block: page kb of row j at a0 + kb r + j
        const int pv_in = W ? vec_pages(pd.d_in, P.h) : 1;
        const int j = js * kSxRows + warp;
        // each warp checks its own A row's pages; a bad page leaves that t entry unwritten
        // (the expand of this chunk checks every page of it and skips it)
        bool live = j < r;
        float acc[kChunk] = {0.f, 0.f, 0.f, 0.f};
        for (int kb = 0; kb < pv_in; ++kb) {
            const int w8 = W ? min(h8, (pd.d_in - kb * P.h) >> 3) : h8;   // used vectors of this block
            const int page = live ? P.pt[a0 + (long long)kb * r + j] : 0;
            if (live && (page < 0 || page >= P.num_pages)) {
                if (lane == 0) set_error(&hdr->err, LORA_DERR_PAGE);
                live = false;
            }
            const __nv_bfloat16* a = P.pages + (long long)(live ? page : 0) * P.h;
            for (int v0 = 0; v0 < w8; v0 += 32 * kSxLoads) {
                uint4 av[kSxLoads];
#pragma unroll
                for (int k = 0; k < kSxLoads; ++k) {
                    const int v = v0 + lane + 32 * k;
                    av[k] = (live && v < w8) ? ld_stream16(a + v * 8) : make_uint4(0, 0, 0, 0);
                }
                if (v0 == 0) {   // the x rows' block kb, while the A loads are in flight
                    for (int e = threadIdx.x; e < ch.count * w8; e += blockDim.x) {
                        const int t = e / w8, v = e % w8;
                        xs[t * h8 + v] = ld16(pd.x + (long long)row_of(ch.rows, t) * pd.ldx + (long long)kb * P.h + v * 8);
                    }
                    __syncthreads();
                }
#pragma unroll
                for (int k = 0; k < kSxLoads; ++k) {
                    const int v = v0 + lane + 32 * k;
                    if (v < w8) {
#pragma unroll
                        for (int t = 0; t < kChunk; ++t)
                            if (t < ch.count) acc[t] = dot8_bf16(xs[t * h8 + v], av[k], acc[t]);
                    }
                }
            }
            if (kb + 1 < pv_in) __syncthreads();   // xs holds the next block's rows next
        }
        if (live) {
#pragma unroll
            for (int t = 0; t < kChunk; ++t) {
                float s = acc[t];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0 && t < ch.count)
                    tbuf[((long long)pr * T + row_of(ch.rows, t)) * r_max + j] = s * ch.scale;
            }
        }
        __syncthreads();   // xs is reused by the next item
    }
}

template <bool W>
__global__ void __launch_bounds__(kSxThreads) lora_expand_kernel(const __grid_constant__ ShrinkExpandParams p) {
    constexpr int kGroups = kSxThreads / kSxVecs;   // threads sharing one column vector
    __shared__ float ts[kChunk][LORA_MAX_RANK];
    __shared__ int32_t pg[LORA_MAX_RANK];
    __shared__ float red[kGroups - 1][kChunk][kSxVecs][8];
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    const WsLayout WL = ws_layout(hdr->cap_tokens, hdr->cap_segments);
    const Chunk* chunks = reinterpret_cast<const Chunk*>(p.ws + WL.chunks);
    const float* tbuf = p.t;
    const int n_chunks = hdr->counts[2];
    const int T = p.T;
    const PoolView& P = p.pool;
    const int h8 = P.h >> 3, r_max = P.r_max;
    // item = (projection, chunk, output page block q, slice of the block)
    const int n_slb = (h8 + kSxVecs - 1) / kSxVecs;
    const int n_sl = n_slb * (W ? p.out_blocks : 1);
    const int vl = threadIdx.x % kSxVecs, g = threadIdx.x / kSxVecs;
    const long long total = (long long)p.nprob * n_chunks * n_sl;
    auto chunk_of = [&](long long it) { return (int)((it / n_sl) % n_chunks); };
    Chunk next;
    if (blockIdx.x < total) next = chunks[chunk_of(blockIdx.x)];
    for (long long item = blockIdx.x; item < total; item += gridDim.x) {
        const int sl = (int)(item % n_sl);
        const int pr = (int)(item / ((long long)n_sl * n_chunks));
        const Chunk ch = next;   // loaded while the previous item was being computed
        if (item + gridDim.x < total) next = chunks[chunk_of(item + gridDim.x)];
        const int r = ch.rank;
        const ProbDesc pd = p.probs[pr];
        const int q = W ? sl / n_slb : 0;                // output page block
        const int pv_in = W ? vec_pages(pd.d_in, P.h) : 1, pv_out = W ? vec_pages(pd.d_out, P.h) : 1;
        if (W && q >= pv_out) continue;                  // a narrower projection
        const int w8 = W ? min(h8, (pd.d_out - q * P.h) >> 3) : h8;
        const int v = (W ? sl % n_slb : sl) * kSxVecs + vl;   // vector within the block
        __nv_bfloat16* yq = W ? pd.y + (long long)q * P.h : pd.y;
        const long long a0 = ch.pt_base + (long long)pd.blk * r;
        const long long bq = a0 + (long long)(pv_in + q) * r;   // page q of the B columns
        // one round trip: the chunk's page ids (all checked: the A rows' too, whose t a bad
        // page left unwritten), its t values and this thread's y vectors
        bool bad = false;
        for (long long e = threadIdx.x; e < (long long)(pv_in + pv_out) * r; e += blockDim.x) {
            const int page = P.pt[a0 + e];
            bad |= (page < 0 || page >= P.num_pages);
            if (!W && e >= r) pg[e - r] = page;
        }
        if (W)
            for (int e = threadIdx.x; e < r; e += blockDim.x) pg[e] = P.pt[bq + e];
        for (int e = threadIdx.x; e < kChunk * r; e += blockDim.x) {
            const int t = e / r, j = e % r;
            ts[t][j] = t < ch.count ? tbuf[((long long)pr * T + row_of(ch.rows, t)) * r_max + j] : 0.f;
        }
        uint4 yv[kChunk];
#pragma unroll
        for (int t = 0; t < kChunk; ++t)
            yv[t] = (g == 0 && v < w8 && t < ch.count) ? ld16(yq + (long long)row_of(ch.rows, t) * pd.ldy + v * 8)
                                                       : make_uint4(0, 0, 0, 0);
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) set_error(&hdr->err, LORA_DERR_PAGE);
            continue;
        }
        float acc[kChunk][8];
#pragma unroll
        for (int t = 0; t < kChunk; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;
        if (v < w8) {
#pragma unroll 16
            for (int j = g; j < r; j += kGroups) {
                float b8[8];
                unpack8(ld_stream16(P.pages + (long long)pg[j] * P.h + v * 8), b8);
#pragma unroll
                for (int t = 0; t < kChunk; ++t) {
                    const float tj = ts[t][j];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) fma2_f32(acc[t][e], acc[t][e + 1], tj, b8[e], b8[e + 1]);
                }
            }
        }
        if (g > 0) {
#pragma unroll
            for (int t = 0; t < kChunk; ++t)
#pragma unroll
                for (int e = 0; e < 8; ++e) red[g - 1][t][vl][e] = acc[t][e];
        }
        __syncthreads();
        if (g == 0 && v < w8) {
#pragma unroll
            for (int t = 0; t < kChunk; ++t) {
                if (t >= ch.count) break;
                __nv_bfloat16* yp = yq + (long long)row_of(ch.rows, t) * pd.ldy + v * 8;
                float y8[8];
                unpack8(yv[t], y8);
                float s8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float s = acc[t][e];
#pragma unroll
                    for (int k = 0; k < kGroups - 1; ++k) s += red[k][t][vl][e];
                    s8[e] = y8[e] + s;
                }
                uint4 o;
                o.x = pack2(s8[0], s8[1]);
                o.y = pack2(s8[2], s8[3]);
                o.z = pack2(s8[4], s8[5]);
                o.w = pack2(s8[6], s8[7]);
                st16(yp, o);
            }
        }
        __syncthreads();   // ts, pg and red are reused by the next item
    }
}

}  // namespace lora
