// CUDA-core BGMV for launches with few projections: one kernel, each chunk (up to 4 rows
// of one adapter) served by a cluster of kClusterCtas CTAs that split its columns.
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "How the kernels work" and
// "What the engine does each step": the LoRA term of each projection is a shrink v = A x
// followed by an expand y += gamma B v, and engines apply it per projection, next to that
// projection's base GEMM.  One projection of a decode batch has only a few dozen chunks,
// too few to fill the GPU one chunk per CTA, and the shrink's reduction over all of x's
// columns must finish before any column of y can be expanded.
//
// Here CTA c of a cluster takes 1/kClusterCtas of the input columns and of the output
// columns of every item (projection, chunk):
//   shrink   partial t_c[row][j] = sum over its input columns of x[row, k] A_j[k] (every
//            A page read once, in slices, by the cluster's CTAs together);
//   exchange each CTA publishes its partials in shared memory, announces them on every
//            peer's mbarrier (a remote arrive), waits for the peers' announcements (a
//            bounded wait) and sums all partials from distributed shared memory: t, scaled;
//   expand   its output columns of y: y = bf16_rn(y + sum_j t[row][j] B_j[col]).
// No t round trip through global memory, no second launch; every page is read once.
// A chunk with a page id out of range is skipped by every CTA of the cluster (each checks
// every page of the item) and reported in the device error word.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace lora {

constexpr int kClusterCtas = 8;          // CTAs of one cluster (the portable maximum)
constexpr int kClusterThreads = 256;      // three CTAs per SM (80 registers): 57 resident clusters,
                                          // enough for a one-projection launch's chunks in one round
constexpr int kClusterMaxProbs = 8;      // projections of one launch at most
constexpr int kClusterDefaultProbs = 1;  // the default limit (measured against the ring kernel)
constexpr int kClusterExpandVecs = 64;   // 16-byte column vectors per expand pass
constexpr int kClusterPg = 4;            // A rows a warp loads at once in the shrink

struct ClusterParams {
    PoolView pool;
    char* ws;
    int32_t nprob;
    int32_t ni;           // input vectors (16 bytes) per CTA: ceil(max d_in / 8 / kClusterCtas)
    int32_t no;           // output vectors per CTA
    int32_t pv_max;       // most page blocks of an A row plus a B column over the launch
    ProbDesc probs[kClusterMaxProbs];
};

// Dynamic shared memory of one CTA (offsets in bytes).
struct ClusterSmem {
    uint32_t xs, part, ts, red, pg, bars, total;
};

__host__ __device__ inline ClusterSmem cluster_smem_layout(int ni, int r_max, int pv_max) {
    ClusterSmem L;
    uint32_t o = 0;
    L.xs = o;    o += (uint32_t)kChunk * ni * 16;                       // the chunk's x rows, its slice
    L.part = o;  o += 2u * kChunk * r_max * 4;                          // partial t, two buffers
    L.ts = o;    o += (uint32_t)kChunk * r_max * 4;                     // t, summed and scaled
    L.red = o;   o += 3u * kChunk * kClusterExpandVecs * 8 * 4;         // expand: 3 groups' sums
    L.pg = o;    o += (uint32_t)r_max * pv_max * 4;                     // page ids of the item
    o = (o + 7) & ~7u;
    L.bars = o;  o += 2 * 8;                                            // exchange barriers
    L.total = o;
    return L;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// The shared-memory address `a` of this CTA seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's prior writes
// (and, through the CTA barrier before it, the CTA's) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}
// Every thread of every CTA of the cluster (an aligned hardware barrier; used once before
// the first exchange and once before exit, where every CTA takes part unconditionally).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// W: the pool has projections whose widths differ from h (vectors over several pages);
// W = false compiles the h x h case.
template <bool W>
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kClusterThreads, 3)
    bgmv_cluster_kernel(const __grid_constant__ ClusterParams p) {
    extern __shared__ __align__(16) unsigned char cl_smem[];
    const ClusterSmem L = cluster_smem_layout(p.ni, p.pool.r_max, p.pv_max);
    uint4* xs = reinterpret_cast<uint4*>(cl_smem + L.xs);
    float* part = reinterpret_cast<float*>(cl_smem + L.part);
    float* ts = reinterpret_cast<float*>(cl_smem + L.ts);
    float* red = reinterpret_cast<float*>(cl_smem + L.red);
    int32_t* pg = reinterpret_cast<int32_t*>(cl_smem + L.pg);
    const uint32_t bars = smem_addr(cl_smem + L.bars);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
    const WsLayout WL = ws_layout(hdr->cap_tokens, hdr->cap_segments);
    const Chunk* chunks = reinterpret_cast<const Chunk*>(p.ws + WL.chunks);
    const int n_chunks = hdr->counts[2];
    const PoolView& P = p.pool;
    const int h8 = P.h >> 3, r_max = P.r_max;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t cid = cluster_id_x(), ncl = cluster_count_x();

    if (tid == 0) {
        mbar_init(bars, kClusterCtas);
        mbar_init(bars + 8, kClusterCtas);
        fence_mbar_init();
    }
    cluster_sync_all();   // every CTA's barriers are initialised before any remote arrive

    const long long total = (long long)p.nprob * n_chunks;
    uint32_t k = 0;       // items of this cluster so far (exchange buffer k & 1, phase (k >> 1) & 1)
    bool ok = true;
    for (long long item = cid; item < total && ok; item += ncl) {
        const int pr = (int)(item / n_chunks);
        const Chunk ch = chunks[item % n_chunks];
        const ProbDesc pd = p.probs[pr];
        const int r = ch.rank;
        const int pv_in = W ? vec_pages(pd.d_in, P.h) : 1, pv_out = W ? vec_pages(pd.d_out, P.h) : 1;
        const long long a0 = ch.pt_base + (long long)pd.blk * r;   // page kb of A row j at a0 + kb r + j;
                                                                    // B column j's page q at a0 + (pv_in + q) r + j
        // the item's page ids (every CTA checks every one: a bad item is skipped by all)
        bool bad = false;
        for (int e = tid; e < (pv_in + pv_out) * r; e += kClusterThreads) {
            const int page = P.pt[a0 + e];
            bad |= (page < 0 || page >= P.num_pages);
            pg[e] = page;
        }
        // this CTA's input columns: vectors [v_lo, v_hi) of x's d_in / 8
        const int d_in8 = pd.d_in >> 3, d_out8 = pd.d_out >> 3;
        const int v_lo = min((int)crank * p.ni, d_in8), v_hi = min(v_lo + p.ni, d_in8);
        const int nv = v_hi - v_lo;
        for (int e = tid; e < ch.count * nv; e += kClusterThreads) {
            const int t = e / nv, v = e % nv;
            xs[t * p.ni + v] = ld16(pd.x + (long long)row_of(ch.rows, t) * pd.ldx + (long long)(v_lo + v) * 8);
        }
        if (__syncthreads_or(bad)) {
            if (tid == 0 && crank == 0) set_error(&hdr->err, LORA_DERR_PAGE);
            continue;
        }
        // this CTA's output columns
        const int o_lo = min((int)crank * p.no, d_out8), o_hi = min(o_lo + p.no, d_out8);
        // Everything the item reads after the page ids is known now: bring this CTA's slices
        // of the A rows, of the B columns and of the chunk's y rows into L2 with one bulk
        // prefetch each, so that the shrink's loads and, after the exchange, the expand's
        // find them there instead of waiting for DRAM one dependent step after another.
        for (int e = tid; e < r + ch.count; e += kClusterThreads) {
            if (e < r) {
                for (int kb = v_lo / h8; kb * h8 < v_hi; ++kb) {   // A row e: its page blocks in [v_lo, v_hi)
                    const int s0 = max(v_lo, kb * h8), s1 = min(v_hi, (kb + 1) * h8);
                    bulk_prefetch_l2(P.pages + (long long)pg[kb * r + e] * P.h + (s0 - kb * h8) * 8,
                                     (uint32_t)(s1 - s0) * 16);
                }
                for (int qb = o_lo / h8; qb * h8 < o_hi; ++qb) {   // B column e: blocks in [o_lo, o_hi)
                    const int s0 = max(o_lo, qb * h8), s1 = min(o_hi, (qb + 1) * h8);
                    bulk_prefetch_l2(P.pages + (long long)pg[(pv_in + qb) * r + e] * P.h + (s0 - qb * h8) * 8,
                                     (uint32_t)(s1 - s0) * 16);
                }
            } else if (o_hi > o_lo) {
                bulk_prefetch_l2(pd.y + (long long)row_of(ch.rows, e - r) * pd.ldy + (long long)o_lo * 8,
                                 (uint32_t)(o_hi - o_lo) * 16);
            }
        }
        const int vl = tid % kClusterExpandVecs, g = tid / kClusterExpandVecs;

        // ---- shrink partials: warp w takes A rows j = w, w + 8, ... in batches of kClusterPg
        //      rows, lane l the vectors v_lo + l, v_lo + l + 32 of its slice (64 per pass); every
        //      load of a batch is issued before the first product
        float* pb = part + (k & 1) * kChunk * r_max;
        for (int jb = warp; jb < r; jb += kClusterPg * (kClusterThreads / 32)) {
            float acc[kClusterPg][kChunk];
#pragma unroll
            for (int i = 0; i < kClusterPg; ++i)
#pragma unroll
                for (int t = 0; t < kChunk; ++t) acc[i][t] = 0.f;
            for (int v0 = 0; v0 < nv; v0 += 64) {
                uint4 av[kClusterPg][2];
#pragma unroll
                for (int i = 0; i < kClusterPg; ++i) {
                    const int j = jb + i * (kClusterThreads / 32);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int v = v0 + lane + 32 * u;
                        const int vg = v_lo + v;                      // vector of the row
                        const int kb = W ? vg / h8 : 0;               // its page block
                        av[i][u] = (j < r && v < nv)
                                       ? ld_stream16(P.pages + (long long)pg[kb * r + j] * P.h + (W ? vg - kb * h8 : vg) * 8)
                                       : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int v = v0 + lane + 32 * u;
                    if (v < nv) {
#pragma unroll
                        for (int t = 0; t < kChunk; ++t) {
                            if (t < ch.count) {
                                const uint4 xv = xs[t * p.ni + v];
#pragma unroll
                                for (int i = 0; i < kClusterPg; ++i) acc[i][t] = dot8_bf16(xv, av[i][u], acc[i][t]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kClusterPg; ++i) {
                const int j = jb + i * (kClusterThreads / 32);
#pragma unroll
                for (int t = 0; t < kChunk; ++t) {
                    float s = acc[i][t];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (lane == 0 && j < r) pb[t * r_max + j] = s;
                }
            }
        }
        __syncthreads();
        // ---- exchange: announce this CTA's partials to every CTA of the cluster, wait for all
        const uint32_t bar = bars + (k & 1) * 8;
        if (tid < kClusterCtas) mbar_arrive_remote(map_rank(bar, (uint32_t)tid));
        if (!mbar_wait_cluster(bar, (k >> 1) & 1, kWaitLimitNs)) {
            if (tid == 0) set_error(&hdr->err, LORA_DERR_TIMEOUT);
            ok = false;
            break;
        }
        const uint32_t pb_addr = smem_addr(pb);
        for (int e = tid; e < ch.count * r; e += kClusterThreads) {
            const int t = e / r, j = e % r;
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < kClusterCtas; ++c) s += ld_cluster_f32(map_rank(pb_addr + (t * r_max + j) * 4, c));
            ts[t * r_max + j] = s * ch.scale;
        }
        __syncthreads();
        // ---- expand this CTA's output vectors, kClusterExpandVecs at a time: 4 groups of
        //      threads take every 4th j and meet in shared memory
        for (int o0 = o_lo; o0 < o_hi; o0 += kClusterExpandVecs) {
            const int ov = o0 + vl;
            const bool live = ov < o_hi;
            const int qb = W ? ov / h8 : 0;                           // page block of the column vector
            const int ow = W ? ov - qb * h8 : ov;                     // vector within the page
            uint4 yv[kChunk];
#pragma unroll
            for (int t = 0; t < kChunk; ++t)
                yv[t] = (g == 0 && live && t < ch.count) ? ld16(pd.y + (long long)row_of(ch.rows, t) * pd.ldy + (long long)ov * 8)
                                                         : make_uint4(0, 0, 0, 0);
            float acc[kChunk][8];
#pragma unroll
            for (int t = 0; t < kChunk; ++t)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;
            if (live) {
                const int32_t* pgb = pg + (pv_in + qb) * r;
#pragma unroll 8
                for (int j = g; j < r; j += kClusterThreads / kClusterExpandVecs) {
                    float b8[8];
                    unpack8(ld_stream16(P.pages + (long long)pgb[j] * P.h + ow * 8), b8);
#pragma unroll
                    for (int t = 0; t < kChunk; ++t) {
                        const float tj = ts[t * r_max + j];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[t][e] = fmaf(tj, b8[e], acc[t][e]);
                    }
                }
            }
            if (g > 0) {
#pragma unroll
                for (int t = 0; t < kChunk; ++t)
#pragma unroll
                    for (int e = 0; e < 8; ++e) red[(((g - 1) * kChunk + t) * kClusterExpandVecs + vl) * 8 + e] = acc[t][e];
            }
            __syncthreads();
            if (g == 0 && live) {
#pragma unroll
                for (int t = 0; t < kChunk; ++t) {
                    if (t >= ch.count) break;
                    float y8[8];
                    unpack8(yv[t], y8);
                    float s8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float s = acc[t][e];
#pragma unroll
                        for (int q = 0; q < 3; ++q) s += red[((q * kChunk + t) * kClusterExpandVecs + vl) * 8 + e];
                        s8[e] = y8[e] + s;
                    }
                    uint4 o;
                    o.x = pack2(s8[0], s8[1]);
                    o.y = pack2(s8[2], s8[3]);
                    o.z = pack2(s8[4], s8[5]);
                    o.w = pack2(s8[6], s8[7]);
                    st16(pd.y + (long long)row_of(ch.rows, t) * pd.ldy + (long long)ov * 8, o);
                }
            }
            __syncthreads();   // red is reused by the next pass
        }
        ++k;
    }
    // no CTA leaves while a peer may still read its partials
    cluster_sync_all();
}

}  // namespace lora
