// CUDA-core BGMV path, warp-specialised: a TMA-fed shared-memory ring.
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work":
// BGMV treats decode tokens independently, gathering the weights of each token's
// adapter; shrink v = A x, expand y += gamma B v.  "S-LoRA: Serving Thousands of
// Concurrent LoRA Adapters", "Kernels and tensor parallelism": each adapter is
// gathered from non-contiguous pages, mixed ranks without padding.
//
// Decode is HBM-bound: the work is streaming each distinct adapter's 2 r pages once
// per projection (r (ceil(d_in/h) + ceil(d_out/h)) for projections of other widths,
// whose vectors span several pages: the item then streams, per input page block, the
// x rows' block and that page of the A rows, and per output page block that page of the
// B columns).  One persistent CTA per SM:
//   warp 0 (producer)  takes work items (chunk of <= 4 rows of one adapter, projection)
//                      in a static rank-sorted round-robin order, validates the item's page ids, and streams
//                      into a ring of shared-memory stages with 1-D bulk copies
//                      (cp.async.bulk, completion counted on an mbarrier): first the x
//                      rows of the chunk, then its A-row pages, then its B-column pages,
//                      up to RP rows of 2h bytes per stage (RP = 4 or 8: the fewer,
//                      larger stages the better a bulk-copy ring streams, as long as
//                      three of them fit).  It prepares the next item while the current
//                      one's x and A stages land;
//   warps 1..CW        consume the stages in the same order: x into registers; the A
//                      pages -> t (on the tensor cores with warp-level mma.sync where the
//                      row splits into groups of four 16-byte vectors per warp, else fp32
//                      partial dot products reduced with a transposing shuffle), summed
//                      across warps in shared memory and scaled; each B page ->
//                      acc[row][col] += t[row][j] * B_j[col]; finally y = bf16_rn(y + acc)
//                      with 16-byte stores.
// Bytes in flight are bounded by the ring (about 190 KB per SM), not by registers.
// Every wait is bounded in time; a timeout sets LORA_DERR_TIMEOUT and unwinds.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace lora {

constexpr int kRingMaxConsumerWarps = 16;
constexpr int kRingPagesSmall = 4;   // pages (or x rows) per stage: the two choices
constexpr int kRingPagesLarge = 8;
constexpr uint32_t kDerrTimeout = LORA_DERR_TIMEOUT;

enum StageKind : int32_t { kStageX = 0, kStageA = 1, kStageB = 2, kStageStop = 3, kStageSkip = 4 };

struct alignas(16) StageMeta {   // written and read as three 16-byte words
    int32_t kind;
    int32_t npages;   // rows carried by this stage
    int32_t j0;       // first page index (A/B stages)
    int32_t pr;       // problem index
    int32_t count;    // rows of the chunk (X stage)
    int32_t rank;
    float scale;
    int32_t rows[kChunk];
    int32_t blk;      // page block of the input (x, A stages) or of the output (B stages)
};
static_assert(sizeof(StageMeta) == 48, "stage meta size");

template <int MAXP>
struct RingParamsT {
    PoolView pool;
    char* ws;
    float* t_out;
    int32_t nprob;
    int32_t stages;        // ring depth
    int32_t stage_bytes;   // RP * 2h
    int32_t pad;
    ProbDesc probs[MAXP];
};
using RingParams = RingParamsT<LORA_MAX_PROBLEMS_PER_LAUNCH>;

// Dynamic shared memory layout (offsets from a 1024-byte aligned base).
struct RingSmem {
    uint32_t ring, full, empty, cbar, meta, red, ts, pgbuf, probs, total;
};

// nprob: problem descriptors copied into shared memory (the last region, so that the other
// offsets do not depend on it and a host may size for more problems than a launch has).
__host__ __device__ inline RingSmem ring_smem_layout(int stages, int stage_bytes, int r_max, int cwarps,
                                                     int nprob) {
    RingSmem L;
    const int rp = (r_max + 7) / 8 * 8;
    uint32_t o = 0;
    L.ring = o;  o += (uint32_t)stages * stage_bytes;
    L.full = o;  o += stages * 8;
    L.empty = o; o += stages * 8;
    L.cbar = o;  o += 8;
    o = (o + 15) & ~15u;
    L.meta = o;  o += stages * sizeof(StageMeta);
    o = (o + 15) & ~15u;
    L.red = o;   o += cwarps * rp * kChunk * 4;
    L.ts = o;    o += rp * kChunk * 4;
    L.pgbuf = o; o += 2 * 2 * LORA_MAX_RANK * 4;   // page ids of two items
    L.probs = o; o += (uint32_t)nprob * sizeof(ProbDesc);
    L.total = o;
    return L;
}

// Column vectors (8 bf16 = 16 B) of a row handled by consumer thread c: c + 32 CW v.
template <int NV, int NT, int CW, int RP>
// h8: the 16-byte vectors of this page block that are used (a partly used last page
// stops early); accumulate: add to the partial sums of earlier page blocks of the rows.
__device__ __forceinline__ void ring_shrink_stage(const unsigned char* stage, int stage_row_bytes,
                                                  int npages, int h8, int c,
                                                  const uint4 (&xv)[kChunk][NV], float* red_w,
                                                  int j0, bool accumulate) {
    constexpr int V = RP * kChunk;   // 16 or 32 values per warp
    static_assert(V <= 32 && RP >= kChunk, "stage shape");
    float vals[V];
#pragma unroll
    for (int i = 0; i < V; ++i) vals[i] = 0.f;
#pragma unroll
    for (int jj = 0; jj < RP; ++jj) {
        if (jj < npages) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int vi = c + v * (CW * 32);
                if (vi < h8) {
                    const uint4 a = *reinterpret_cast<const uint4*>(stage + jj * stage_row_bytes + vi * 16);
#pragma unroll
                    for (int t = 0; t < NT; ++t) vals[jj * kChunk + t] = dot8_bf16(xv[t][v], a, vals[jj * kChunk + t]);
                }
            }
        }
    }
    const float sum = warp_transpose_reduce<V>(vals);
    const int lane = threadIdx.x & 31;
    constexpr int kRep = 32 / V;   // lanes holding each sum
    if (lane % kRep == 0) {   // index jj*kChunk + t; the same lane owns it in every block
        float* dst = red_w + j0 * kChunk + lane / kRep;
        *dst = accumulate ? *dst + sum : sum;
    }
}

// The shrink of one A stage on the tensor cores (warp-level mma.sync, m16n8k16, bf16 x bf16
// into fp32), for pools whose h splits into kXf groups of four 16-byte vectors per consumer
// warp.  Warp w takes the columns [w h / CW, (w + 1) h / CW) of the chunk's rows and of the
// stage's pages: the tile is rows (16, of which the chunk's <= 4 are real) x pages (8) x
// those columns.  The sum over k is order-free, so lane (g, q) feeds the k slots {2q, 2q+1,
// 2q+8, 2q+9} of two consecutive k steps from one 16-byte vector (its vector q + 4j of the
// warp's columns) -- of x row g for the A operand and of page g for the B operand, the same
// columns on both sides -- and no operand needs a shared-memory shuffle.  Accumulator lane
// (g, q) then holds the warp's partial sums for row g and pages 2q, 2q+1.
constexpr int kMmaXf = 8;   // 16-byte vectors of a row per lane, at most (h = 4096 over 16 warps)

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

template <int XF>
__device__ __forceinline__ void ring_shrink_stage_mma(const unsigned char* stage, int stage_row_bytes, int npages,
                                                      int warp_vec0, int lane, const uint4 (&xf)[kMmaXf],
                                                      float* red_w, int j0, bool accumulate) {
    const int g = lane >> 2, q = lane & 3;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    const unsigned char* pg = stage + (size_t)g * stage_row_bytes + (size_t)warp_vec0 * 16;
#pragma unroll
    for (int j = 0; j < XF; ++j) {
        const uint4 b = g < npages ? *reinterpret_cast<const uint4*>(pg + (q + 4 * j) * 16) : make_uint4(0, 0, 0, 0);
        mma_bf16_16816(c, xf[j].x, xf[j].y, b.x, b.y);
        mma_bf16_16816(c, xf[j].z, xf[j].w, b.z, b.w);
    }
    if (g < kChunk) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int page = 2 * q + e;
            if (page < npages) {
                float* dst = red_w + (j0 + page) * kChunk + g;
                *dst = accumulate ? *dst + c[e] : c[e];
            }
        }
    }
}

template <int NV, int NT, int CW, int RP>
__device__ __forceinline__ void ring_expand_stage(const unsigned char* stage, int stage_row_bytes,
                                                  int npages, int h8, int c, const float* ts, int j0,
                                                  float (&acc)[kChunk][NV][8]) {
#pragma unroll
    for (int jj = 0; jj < RP; ++jj) {
        if (jj < npages) {
            const float4 tj = *reinterpret_cast<const float4*>(ts + (j0 + jj) * kChunk);
            const float tv[4] = {tj.x, tj.y, tj.z, tj.w};
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int vi = c + v * (CW * 32);
                if (vi < h8) {
                    const uint4 b = *reinterpret_cast<const uint4*>(stage + jj * stage_row_bytes + vi * 16);
                    float b8[8];
                    unpack8(b, b8);
#pragma unroll
                    for (int t = 0; t < NT; ++t)
#pragma unroll
                        for (int e = 0; e < 8; e += 2) fma2_f32(acc[t][v][e], acc[t][v][e + 1], tv[t], b8[e], b8[e + 1]);
                }
            }
        }
    }
}

// One work item on the consumer side, specialised on the number of rows NT.
// Returns false if a wait timed out (the kernel then unwinds).
// Barrier of the consumer warps only, built on an mbarrier so that the wait is bounded
// (a plain named barrier could wait forever on a warp that gave up).
__device__ __forceinline__ bool consumer_barrier(unsigned char* base, const RingSmem& L, uint32_t& phase) {
    __syncwarp();
    const uint32_t bar = smem_addr(base + L.cbar);
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase & 1, kWaitLimitNs);
    ++phase;
    return ok;
}

// W: the pool has projections whose widths differ from h (vectors of several page blocks,
// a partly used last page); W = false compiles the h x h case with one block each.
template <int NV, int NT, int CW, int RP, bool W, class P>
__device__ __forceinline__ bool ring_consume_item(const P& p, unsigned char* base, const RingSmem& L,
                                  uint32_t& it, uint32_t& bphase, const StageMeta& mx, int c) {
    const int h = p.pool.h, h8 = h >> 3;
    const int row_bytes = h * 2;
    const int S = p.stages;
    const int warp = c >> 5, lane = c & 31;
    const int rp = (p.pool.r_max + 7) / 8 * 8;
    float* red = reinterpret_cast<float*>(base + L.red);
    float* red_w = red + warp * rp * kChunk;
    float* ts = reinterpret_cast<float*>(base + L.ts);
    const int r = mx.rank;
    const ProbDesc& pd = reinterpret_cast<const ProbDesc*>(base + L.probs)[mx.pr];

    // for each page block kb of the input: the x rows' block (the first one's stage was
    // waited by the caller), then page kb of the A rows; partial sums add up over blocks
    const int pv_in = W ? vec_pages(pd.d_in, h) : 1, pv_out = W ? vec_pages(pd.d_out, h) : 1;
    // tensor-core shrink: one vector per thread (NV = 1), h x h pages, and the row's vectors
    // split into groups of four per warp (h = 1024, 2048, 4096 with 8 or 16 warps); a 4-row
    // stage fills half of the MMA's 8 page columns, the rest read as zeros
    constexpr bool kMmaShape = (NV == 1 && !W && (RP == 8 || RP == 4));
    const int warp_vecs = h8 / CW;
    const int xgroups = warp_vecs / 4;   // k-step pairs of a warp: 1, 2, 4 or 8
    if (kMmaShape && h8 % (CW * 4) == 0 && (xgroups == 1 || xgroups == 2 || xgroups == 4 || xgroups == 8)) {
        const int g = lane >> 2, q = lane & 3;
        uint4 xf[kMmaXf];
        {
            const unsigned char* st = base + L.ring + (size_t)(it % S) * p.stage_bytes;
#pragma unroll
            for (int j = 0; j < kMmaXf; ++j)
                xf[j] = (g < mx.count && j < xgroups)
                            ? *reinterpret_cast<const uint4*>(st + g * row_bytes + (warp * warp_vecs + q + 4 * j) * 16)
                            : make_uint4(0, 0, 0, 0);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(base + L.empty + (it % S) * 8));
            ++it;
        }
        for (int j0 = 0; j0 < r; j0 += RP) {
            const uint32_t s = it % S;
            if (!mbar_wait(smem_addr(base + L.full + s * 8), (it / S) & 1, kWaitLimitNs)) return false;
            const int np = min(RP, r - j0);
            const unsigned char* st = base + L.ring + (size_t)s * p.stage_bytes;
            // exactly the warp's groups: a wider loop would read other warps' columns
            if (xgroups == 8)
                ring_shrink_stage_mma<8>(st, row_bytes, np, warp * warp_vecs, lane, xf, red_w, j0, false);
            else if (xgroups == 4)
                ring_shrink_stage_mma<4>(st, row_bytes, np, warp * warp_vecs, lane, xf, red_w, j0, false);
            else if (xgroups == 2)
                ring_shrink_stage_mma<2>(st, row_bytes, np, warp * warp_vecs, lane, xf, red_w, j0, false);
            else
                ring_shrink_stage_mma<1>(st, row_bytes, np, warp * warp_vecs, lane, xf, red_w, j0, false);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(base + L.empty + s * 8));
            ++it;
        }
    } else
    for (int kb = 0; kb < pv_in; ++kb) {
        const int w8 = W ? min(h8, (pd.d_in - kb * h) >> 3) : h8;   // used vectors of this block
        if (kb > 0 && !mbar_wait(smem_addr(base + L.full + (it % S) * 8), (it / S) & 1, kWaitLimitNs))
            return false;
        uint4 xv[kChunk][NV];
        {
            const unsigned char* st = base + L.ring + (size_t)(it % S) * p.stage_bytes;
#pragma unroll
            for (int t = 0; t < kChunk; ++t)
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int vi = c + v * (CW * 32);
                    xv[t][v] = (t < mx.count && vi < w8) ? *reinterpret_cast<const uint4*>(st + t * row_bytes + vi * 16)
                                                   : make_uint4(0, 0, 0, 0);
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(base + L.empty + (it % S) * 8));
            ++it;
        }
        for (int j0 = 0; j0 < r; j0 += RP) {
            const uint32_t s = it % S;
            if (!mbar_wait(smem_addr(base + L.full + s * 8), (it / S) & 1, kWaitLimitNs)) return false;
            const int np = min(RP, r - j0);
            ring_shrink_stage<NV, NT, CW, RP>(base + L.ring + (size_t)s * p.stage_bytes, row_bytes, np, w8, c, xv,
                                              red_w, j0, W && kb > 0);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(base + L.empty + s * 8));
            ++it;
        }
    }
    // Two barriers per item: every warp's partial sums are in red, then t is complete.
    // The next item writes red only after the second one (every warp is done reading
    // red) and t only after its own first one, which every warp reaches after its expand
    // of this item, so no barrier is needed at the end of the item.
    if (!consumer_barrier(base, L, bphase)) return false;
    // only the NT rows the expand reads (entries of t for rows >= NT are never read)
    for (int e = c; e < r * NT; e += CW * 32) {
        const int j = e / NT, t = e % NT;
        const int idx = j * kChunk + t;
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < CW; ++w) a += red[w * rp * kChunk + idx];
        ts[idx] = a * mx.scale;
        if (p.t_out != nullptr && t < mx.count)
            p.t_out[(long long)row_of(mx.rows, t) * p.pool.r_max + j] = a * mx.scale;
    }
    if (!consumer_barrier(base, L, bphase)) return false;
    // for each page block q of the output: y's block q (loaded while its B pages stream
    // in), page q of the B columns, y = bf16_rn(y + acc) for the block's used columns
    for (int q = 0; q < pv_out; ++q) {
        const int w8 = W ? min(h8, (pd.d_out - q * h) >> 3) : h8;
        __nv_bfloat16* yq = W ? pd.y + (long long)q * h : pd.y;
        uint4 yv[NT][NV];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int vi = c + v * (CW * 32);
                yv[t][v] = (t < mx.count && vi < w8) ? ld16(yq + (long long)mx.rows[t] * pd.ldy + vi * 8)
                                                     : make_uint4(0, 0, 0, 0);
            }
        float acc[kChunk][NV][8];
#pragma unroll
        for (int t = 0; t < kChunk; ++t)
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[t][v][e] = 0.f;
        for (int j0 = 0; j0 < r; j0 += RP) {
            const uint32_t s = it % S;
            if (!mbar_wait(smem_addr(base + L.full + s * 8), (it / S) & 1, kWaitLimitNs)) return false;
            const int np = min(RP, r - j0);
            ring_expand_stage<NV, NT, CW, RP>(base + L.ring + (size_t)s * p.stage_bytes, row_bytes, np, w8, c, ts,
                                              j0, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(base + L.empty + s * 8));
            ++it;
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int vi = c + v * (CW * 32);
                if (t < mx.count && vi < w8) {
                    float y8[8];
                    unpack8(yv[t][v], y8);
                    uint4 o;
                    o.x = pack2(y8[0] + acc[t][v][0], y8[1] + acc[t][v][1]);
                    o.y = pack2(y8[2] + acc[t][v][2], y8[3] + acc[t][v][3]);
                    o.z = pack2(y8[4] + acc[t][v][4], y8[5] + acc[t][v][5]);
                    o.w = pack2(y8[6] + acc[t][v][6], y8[7] + acc[t][v][7]);
                    st16(yq + (long long)mx.rows[t] * pd.ldy + vi * 8, o);
                }
            }
    }
    return true;
}

// One CTA of the ring kernel: CTA `cta` of `ncta` taking part (threads beyond the
// producer and the CW consumer warps only join the initial barrier).
// NV: 16-byte column vectors per consumer thread; CW: consumer warps (h = 8 * 32 * CW * NV
// or less); RP: rows per stage (stage_bytes = RP * 2h).
template <int NV, int CW, int RP, bool W, class P>
__device__ __forceinline__ void ring_cta(const P& p, unsigned char* base, uint32_t cta, uint32_t ncta) {
    const RingSmem L = ring_smem_layout(p.stages, p.stage_bytes, p.pool.r_max, CW, p.nprob);
    const int S = p.stages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    StageMeta* meta = reinterpret_cast<StageMeta*>(base + L.meta);
    // The problem descriptors, copied once into shared memory: read from the kernel
    // parameters by problem index, they go through the constant cache, which misses on
    // most items (about a microsecond each on the producer's path, as long as a small
    // item takes to stream).
    const ProbDesc* sprobs = reinterpret_cast<const ProbDesc*>(base + L.probs);
    {
        static_assert(sizeof(ProbDesc) % 8 == 0, "descriptor copy in 8-byte words");
        const unsigned long long* src = reinterpret_cast<const unsigned long long*>(p.probs);
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(base + L.probs);
        const int words = p.nprob * (int)(sizeof(ProbDesc) / 8);
        for (int w = tid; w < words; w += blockDim.x) dst[w] = src[w];
    }

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(base + L.full + s * 8), 1);
            mbar_init(smem_addr(base + L.empty + s * 8), CW);
        }
        mbar_init(smem_addr(base + L.cbar), CW);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        // Items (chunk q, problem pr) = (item / nprob, item % nprob) are dealt round-robin
        // over the CTAs (chunks are listed by descending rank, so every CTA gets a similar
        // mix and the last round is made of the smallest items).  The metadata of the next
        // items is loaded while the current one streams: the chunk two items ahead, the
        // page ids one item ahead.  Each item is prepared (page ids checked and written to
        // one of two id buffers, its stage metadata built) while the previous item's x and
        // A stages are in flight, before that item's B stages wait for a free stage: the
        // B stages of item k need the consumers to finish item k - 1, and the x stage of
        // item k + 1 then follows them at once.
        const PoolView& PV = p.pool;
        const WsLayout WL = ws_layout(hdr->cap_tokens, hdr->cap_segments);
        const Chunk* chunks = reinterpret_cast<const Chunk*>(p.ws + WL.chunks);
        const uint32_t total = (uint32_t)hdr->counts[2] * (uint32_t)p.nprob;
        const uint32_t row_bytes = (uint32_t)PV.h * 2;
        const uint32_t G = ncta;
        constexpr int kPg = 2 * LORA_MAX_RANK / 32;   // page ids per lane
        uint32_t it = 0;
        bool ok = true;
        auto claim = [&](void) -> int {
            const uint32_t s = it % S;
            if (!mbar_wait(smem_addr(base + L.empty + s * 8), ((it / S) & 1) ^ 1, kWaitLimitNs)) return -1;
            return (int)s;
        };
        // page ids of an item's first A block and first B block (all of them for h x h pools)
        auto load_pages = [&](const Chunk& c, uint32_t itm, int32_t (&pg)[kPg]) {
            const ProbDesc& pd = sprobs[itm % p.nprob];
            const long long a0 = c.pt_base + (long long)pd.blk * c.rank;
            const long long b0 = a0 + (long long)(W ? vec_pages(pd.d_in, PV.h) : 1) * c.rank;
#pragma unroll
            for (int k = 0; k < kPg; ++k) {
                const int e = lane + 32 * k;
                pg[k] = 0;
                if (32 * k < 2 * c.rank)   // whole groups of 32 ids past the item's are skipped
                    pg[k] = e < c.rank ? PV.pt[a0 + e] : (e < 2 * c.rank ? PV.pt[b0 + e - c.rank] : 0);
            }
        };
        struct Cur {
            Chunk ch;
            long long a0, b0;   // first A-block and B-block entries
            int pr, pv_in, pv_out;
            bool bad;
        };
        Chunk c_next, c_next2;
        int32_t pg_next[kPg];
        // item `itm`: rotate the metadata pipeline, check its page ids into id buffer `buf`
        auto prepare = [&](uint32_t itm, int buf, Cur& cu) {
            cu.ch = c_next;
            int32_t pg[kPg];
#pragma unroll
            for (int k = 0; k < kPg; ++k) pg[k] = pg_next[k];
            if (itm + G < total) {
                c_next = c_next2;
                load_pages(c_next, itm + G, pg_next);
            }
            if (itm + 2 * G < total) c_next2 = chunks[(itm + 2 * G) / p.nprob];
            const int r = cu.ch.rank;
            cu.pr = itm % p.nprob;
            const ProbDesc& pd = sprobs[cu.pr];
            cu.pv_in = W ? vec_pages(pd.d_in, PV.h) : 1;
            cu.pv_out = W ? vec_pages(pd.d_out, PV.h) : 1;
            cu.a0 = cu.ch.pt_base + (long long)pd.blk * r;
            cu.b0 = cu.a0 + (long long)cu.pv_in * r;
            int32_t* ids = reinterpret_cast<int32_t*>(base + L.pgbuf) + buf * 2 * LORA_MAX_RANK;
            bool bad = false;
#pragma unroll
            for (int k = 0; k < kPg; ++k) {
                const int e = lane + 32 * k;
                if (e < 2 * r) {
                    bad |= (pg[k] < 0 || pg[k] >= PV.num_pages);
                    ids[e] = pg[k];
                }
            }
            // vectors longer than a page: the item's other page blocks are checked too
            if (W) {
                for (long long e = lane; e < (long long)(cu.pv_in - 1) * r; e += 32) {
                    const int q = PV.pt[cu.a0 + r + e];
                    bad |= (q < 0 || q >= PV.num_pages);
                }
                for (long long e = lane; e < (long long)(cu.pv_out - 1) * r; e += 32) {
                    const int q = PV.pt[cu.b0 + r + e];
                    bad |= (q < 0 || q >= PV.num_pages);
                }
            }
            cu.bad = __any_sync(0xffffffffu, bad);
            __syncwarp();
            if (cu.bad && lane == 0) set_error(&hdr->err, LORA_DERR_PAGE);
        };
        uint32_t item = cta;
        if (item < total) {
            c_next = chunks[item / p.nprob];
            load_pages(c_next, item, pg_next);
        }
        if (item + G < total) c_next2 = chunks[(item + G) / p.nprob];
        Cur cur;
        int buf = 0;
        if (item < total) prepare(item, buf, cur);
        while (item < total) {
            const Chunk& ch = cur.ch;
            const int r = ch.rank;
            const ProbDesc& pd = sprobs[cur.pr];
            int32_t* pgbuf = reinterpret_cast<int32_t*>(base + L.pgbuf) + buf * 2 * LORA_MAX_RANK;
            StageMeta m;
            m.kind = cur.bad ? kStageSkip : kStageX;
            m.npages = ch.count;
            m.j0 = 0;
            m.pr = cur.pr;
            m.count = ch.count;
            m.rank = r;
            m.scale = ch.scale;
#pragma unroll
            for (int t = 0; t < kChunk; ++t) m.rows[t] = ch.rows[t];
            m.blk = 0;
            // Stages of the item: for each page block kb of the input, the x rows' block
            // kb then page kb of the A rows; then, for each page block q of the output,
            // page q of the B columns.  Only the used part of a partly used page is copied.
            // emit_pages: stage(s) of page block `blk_idx` (ids from pgbuf[off ..]) of kind
            auto emit_pages = [&](int kind, int blk_idx, int off, uint32_t bytes) {
                for (int j0 = 0; j0 < r; j0 += RP) {
                    const int np = min(RP, r - j0);
                    const int s = claim();
                    if (s < 0) return false;
                    if (lane == 0) {
                        StageMeta mm = m;
                        mm.kind = kind;
                        mm.npages = np;
                        mm.j0 = j0;
                        mm.blk = blk_idx;
                        meta[s] = mm;
                        mbar_arrive_expect_tx(smem_addr(base + L.full + s * 8), bytes * np);
                    }
                    __syncwarp();
                    if (lane < np) {
                        const int page = pgbuf[off + j0 + lane];
                        bulk_g2s(smem_addr(base + L.ring + (size_t)s * p.stage_bytes + lane * row_bytes),
                                 PV.pages + (long long)page * PV.h, bytes, smem_addr(base + L.full + s * 8));
                    }
                    ++it;
                }
                return true;
            };
            // page ids of block kb of a multi-page vector, into pgbuf[off ..]
            auto fetch_block = [&](long long first, int off) {
                __syncwarp();   // every lane has read the previous block's ids
                for (int e = lane; e < r; e += 32) pgbuf[off + e] = PV.pt[first + e];
                __syncwarp();
            };
            if (cur.bad) {   // a skip marker in place of the item
                const int s = claim();
                if (s < 0) { ok = false; break; }
                if (lane == 0) {
                    meta[s] = m;
                    mbar_arrive(smem_addr(base + L.full + s * 8));
                }
                __syncwarp();
                ++it;
            } else {
                for (int kb = 0; kb < cur.pv_in && ok; ++kb) {
                    const uint32_t bytes = W ? (uint32_t)min(PV.h, pd.d_in - kb * PV.h) * 2 : row_bytes;
                    const int s = claim();
                    if (s < 0) { ok = false; break; }
                    if (lane == 0) {
                        StageMeta mx = m;
                        mx.blk = kb;
                        meta[s] = mx;
                        mbar_arrive_expect_tx(smem_addr(base + L.full + s * 8), bytes * ch.count);
                    }
                    __syncwarp();
                    if (lane < ch.count)
                        bulk_g2s(smem_addr(base + L.ring + (size_t)s * p.stage_bytes + lane * row_bytes),
                                 pd.x + (long long)row_of(ch.rows, lane) * pd.ldx + (long long)kb * PV.h, bytes,
                                 smem_addr(base + L.full + s * 8));
                    ++it;
                    if (kb > 0) fetch_block(cur.a0 + (long long)kb * r, 0);
                    if (!emit_pages(kStageA, kb, 0, bytes)) ok = false;
                }
            }
            if (!ok) break;
            // the next item, prepared while this one's x and A stages land (after its B
            // stages for pools with vectors of several pages, whose longer checks would
            // otherwise keep both items' state in registers across the B stages)
            const uint32_t nxt = item + G;
            Cur nx;
            if (!W && nxt < total) prepare(nxt, buf ^ 1, nx);
            if (!cur.bad) {
                for (int q = 0; q < cur.pv_out && ok; ++q) {
                    const uint32_t bytes = W ? (uint32_t)min(PV.h, pd.d_out - q * PV.h) * 2 : row_bytes;
                    if (q > 0) fetch_block(cur.b0 + (long long)q * r, r);
                    if (!emit_pages(kStageB, q, r, bytes)) ok = false;
                }
            }
            if (!ok) break;
            if (W && nxt < total) prepare(nxt, buf ^ 1, nx);
            item = nxt;
            if (item < total) cur = nx;
            buf ^= 1;
        }
        if (ok) {
            // stop marker for the consumers
            const int s = claim();
            if (s >= 0 && lane == 0) {
                meta[s].kind = kStageStop;
                mbar_arrive(smem_addr(base + L.full + s * 8));
            }
            if (s < 0) ok = false;
            else ++it;   // the stop stage is a use of its barrier like any other
        }
        if (!ok && lane == 0) set_error(&hdr->err, kDerrTimeout);
        // wait (bounded) until every stage this warp filled has landed, so no copy into
        // this CTA's shared memory is still in flight when it exits
        if (lane == 0) {
            const uint32_t first = it > (uint32_t)S ? it - S : 0;
            for (uint32_t k = first; k < it; ++k)
                mbar_wait(smem_addr(base + L.full + (k % S) * 8), (k / S) & 1, 100000000ull);
        }
    } else if (tid < CW * 32 + 32) {
        // ------------------------------------------------------------------ consumers
        const int c = tid - 32;
        uint32_t it = 0, bphase = 0;
        for (;;) {
            const uint32_t s = it % S;
            if (!mbar_wait(smem_addr(base + L.full + s * 8), (it / S) & 1, kWaitLimitNs)) {
                if (c == 0) set_error(&hdr->err, kDerrTimeout);
                break;
            }
            const StageMeta mx = meta[s];
            if (mx.kind == kStageStop) break;
            if (mx.kind == kStageSkip) {
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(base + L.empty + s * 8));
                ++it;
                continue;
            }
            bool ok;
            if (mx.count == 1)
                ok = ring_consume_item<NV, 1, CW, RP, W, P>(p, base, L, it, bphase, mx, c);
            else if (mx.count == 2)
                ok = ring_consume_item<NV, 2, CW, RP, W, P>(p, base, L, it, bphase, mx, c);
            else
                ok = ring_consume_item<NV, kChunk, CW, RP, W, P>(p, base, L, it, bphase, mx, c);
            if (!ok) {
                if (c == 0) set_error(&hdr->err, kDerrTimeout);
                break;
            }
        }
    }
}

template <int NV, int CW, int RP, bool W>
__global__ void __launch_bounds__(CW * 32 + 32, 1) bgmv_ring_kernel(const __grid_constant__ RingParams p) {
    extern __shared__ __align__(1024) unsigned char ring_smem_raw[];
    ring_cta<NV, CW, RP, W>(p, ring_smem_raw, blockIdx.x, gridDim.x);
}

}  // namespace lora
