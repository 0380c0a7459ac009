// CUDA-core BGMV path: shrink + expand for chunks of up to kChunk rows of one adapter.
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work":
// BGMV treats tokens independently and gathers the adapter weights indexed by a(i);
// shrink v = A x then expand y += gamma B v.  "S-LoRA: Serving Thousands of Concurrent
// LoRA Adapters", "Kernels and tensor parallelism": weights gathered from
// non-contiguous pages, mixed ranks without padding.
//
// Persistent kernel over work items (chunk, problem), taken from a device counter.
// One CTA of 512 threads owns an item: every thread owns 8 consecutive columns per
// 4096-column pass, loads 16-byte vectors of x, of each A-row page and of each
// B-column page (the pages are read exactly once per item), and
//   shrink: partial dot products, reduced across each warp with a transposing
//           shuffle reduction and across warps in shared memory -> t (fp32, scaled)
//   expand: acc[row][col] += t[row][j] * B_j[col], then y = bf16_rn(y + acc).
#pragma once
#include "common.cuh"
#include "segment.cuh"

namespace lora {

constexpr int kFmaThreads = 512;
constexpr int kFmaWarps = kFmaThreads / 32;
constexpr int kColsPerPass = kFmaThreads * 8;

struct DeltaParams {
    PoolView pool;
    char* ws;
    float* t_out;   // debug: fp32 t per row [T][r_max] (single-problem launches only)
    int32_t nprob;
    int32_t pad;
    ProbDesc probs[LORA_MAX_PROBLEMS_PER_LAUNCH];
};

// Shared memory of one CTA (dynamic): red [warps][r_pad * kChunk], ts [r_pad * kChunk],
// pages [2 * r_pad], rows [kChunk].
// Rank padded to a multiple of 8 (the largest page batch of the kernel).
__host__ __device__ inline int fma_r_pad(int r_max) { return (r_max + 7) / 8 * 8; }
__host__ __device__ inline size_t fma_smem_bytes(int r_max) {
    const int rp = fma_r_pad(r_max);
    return (size_t)kFmaWarps * rp * kChunk * 4 + (size_t)rp * kChunk * 4 + (size_t)2 * rp * 4 +
           kChunk * 4 + 16;
}

// NV: 16-byte column vectors per thread (h <= NV * 4096); JU: pages per load batch.
template <int NV, int JU>
__global__ void __launch_bounds__(kFmaThreads, 1) fma_delta_kernel(const __grid_constant__ DeltaParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const PoolView& P = p.pool;
    const int rp = fma_r_pad(P.r_max);
    float* red = reinterpret_cast<float*>(smem_raw);
    float* ts = red + kFmaWarps * rp * kChunk;
    int32_t* pg = reinterpret_cast<int32_t*>(ts + rp * kChunk);
    int32_t* rows = pg + 2 * rp;
    int* item_s = rows + kChunk;

    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    const WsLayout L = ws_layout(hdr->cap_tokens, hdr->cap_segments);
    const Chunk* chunks = reinterpret_cast<const Chunk*>(p.ws + L.chunks);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = P.h;
    const uint32_t total = (uint32_t)hdr->counts[2] * (uint32_t)p.nprob;

    for (;;) {
        if (tid == 0) *item_s = (int)atomicAdd(&hdr->work_counter, 1u);
        __syncthreads();
        const uint32_t item = (uint32_t)*item_s;
        if (item >= total) break;
        const int q = item / p.nprob, pr = item % p.nprob;
        const Chunk ch = chunks[q];
        const ProbDesc pd = p.probs[pr];
        const int r = ch.rank;
        const long long blk = P.pt_off[ch.adapter] + (long long)pd.blk * 2 * r;
        int bad = 0;
        for (int e = tid; e < 2 * r; e += kFmaThreads) {
            const int page = P.pt[blk + e];
            bad |= (page < 0 || page >= P.num_pages);
            pg[e] = page;
        }
        if (tid < kChunk) rows[tid] = ch.rows[tid];
        if (__syncthreads_or(bad)) {
            if (tid == 0) set_error(&hdr->err, LORA_DERR_PAGE);
            continue;
        }
        const float s = P.scales[ch.adapter];

        // ---- shrink: red[warp][j * kChunk + t] = warp-partial of x_t . A_j
        uint4 xv[kChunk][NV];
#pragma unroll
        for (int t = 0; t < kChunk; ++t)
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = (v * kFmaThreads + tid) * 8;
                xv[t][v] = (t < ch.count && col < h)
                               ? ld16(pd.x + (long long)rows[t] * pd.ldx + col)
                               : make_uint4(0, 0, 0, 0);
            }
        for (int j0 = 0; j0 < r; j0 += JU) {
            uint4 av[JU][NV];
#pragma unroll
            for (int jj = 0; jj < JU; ++jj)
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int col = (v * kFmaThreads + tid) * 8;
                    av[jj][v] = (j0 + jj < r && col < h)
                                    ? ld_stream16(P.pages + (long long)pg[j0 + jj] * h + col)
                                    : make_uint4(0, 0, 0, 0);
                }
            float vals[JU * kChunk];
#pragma unroll
            for (int jj = 0; jj < JU; ++jj)
#pragma unroll
                for (int t = 0; t < kChunk; ++t) {
                    float acc = 0.f;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float a8[8], x8[8];
                        unpack8(av[jj][v], a8);
                        unpack8(xv[t][v], x8);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc = fmaf(x8[e], a8[e], acc);
                    }
                    vals[jj * kChunk + t] = acc;
                }
            const float sum = warp_transpose_reduce<JU * kChunk>(vals);
            constexpr int kLanesPer = 32 / (JU * kChunk);
            if ((lane % kLanesPer) == 0) red[warp * rp * kChunk + j0 * kChunk + lane / kLanesPer] = sum;
        }
        __syncthreads();
        for (int e = tid; e < r * kChunk; e += kFmaThreads) {
            float acc = 0.f;
#pragma unroll 4
            for (int w = 0; w < kFmaWarps; ++w) acc += red[w * rp * kChunk + e];
            ts[e] = acc * s;
            if (p.t_out != nullptr) {
                const int j = e / kChunk, t = e % kChunk;
                if (t < ch.count) p.t_out[(long long)rows[t] * P.r_max + j] = acc * s;
            }
        }
        __syncthreads();

        // ---- expand: acc[t][v][c] = sum_j ts[j][t] * B_j[col + c]
        float acc[kChunk][NV][8];
#pragma unroll
        for (int t = 0; t < kChunk; ++t)
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[t][v][c] = 0.f;
        for (int j0 = 0; j0 < r; j0 += JU) {
            uint4 bv[JU][NV];
#pragma unroll
            for (int jj = 0; jj < JU; ++jj)
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int col = (v * kFmaThreads + tid) * 8;
                    bv[jj][v] = (j0 + jj < r && col < h)
                                    ? ld_stream16(P.pages + (long long)pg[r + j0 + jj] * h + col)
                                    : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int jj = 0; jj < JU; ++jj) {
                const float4 tj = *reinterpret_cast<const float4*>(ts + (j0 + jj) * kChunk);
                const float tv[4] = {tj.x, tj.y, tj.z, tj.w};
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float b8[8];
                    unpack8(bv[jj][v], b8);
#pragma unroll
                    for (int t = 0; t < kChunk; ++t)
#pragma unroll
                        for (int c = 0; c < 8; ++c) acc[t][v][c] = fmaf(tv[t], b8[c], acc[t][v][c]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kChunk; ++t) {
            if (t >= ch.count) break;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = (v * kFmaThreads + tid) * 8;
                if (col >= h) continue;
                __nv_bfloat16* yp = pd.y + (long long)rows[t] * pd.ldy + col;
                const uint4 yv = ld16(yp);
                float y8[8];
                unpack8(yv, y8);
                uint4 o;
                o.x = pack2(y8[0] + acc[t][v][0], y8[1] + acc[t][v][1]);
                o.y = pack2(y8[2] + acc[t][v][2], y8[3] + acc[t][v][3]);
                o.z = pack2(y8[4] + acc[t][v][4], y8[5] + acc[t][v][5]);
                o.w = pack2(y8[6] + acc[t][v][6], y8[7] + acc[t][v][7]);
                st16(yp, o);
            }
        }
        // the next item's page/row writes must not race this item's reads
        __syncthreads();
    }
    // last CTA out resets the queue for the next launch on this workspace
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&hdr->done_counter, 1u);
        if (prev == gridDim.x - 1) {
            hdr->work_counter = 0;
            hdr->done_counter = 0;
            __threadfence();
        }
    }
}

}  // namespace lora
