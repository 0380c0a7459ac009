// Launches of the tensor-core tile kernel (sgmv_mma.cuh) and of the fused launch of both
// work classes (fused.cuh): tensor maps, shared-memory plan, CTA split weights.
#include <string.h>

#include <algorithm>
#include <mutex>

#include "fused.cuh"
#include "host.h"

namespace lora {
namespace host {

// Segments of at least this many rows (and rank <= kMmaMaxRank) take the tensor-core
// path when h is a multiple of 128 and every projection's d_in is a multiple of 64 (the
// shrink K chunk) and d_out one of 128 (the expand slice); the pool's tuning sets the
// row count, or -1 for the rank rule mma_min_rows_for_rank (0 disables the path; one-row
// segments always stay on the CUDA-core path).
int mma_min_rows(const lora_pool* pool) {
    const lora_pool_desc& d = pool->d;
    if (d.h % kMmaNTile != 0 || !pool->mma_widths) return 0;
    return pool->tune.mma_min_rows;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

std::mutex g_encode_mu;

lora_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        lora_status st = cuda_status(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                                      cudaEnableDefault, &q));
        if (st != LORA_OK) return st;
        if (fn == nullptr || q != cudaDriverEntryPointSuccess) return LORA_ECUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return LORA_OK;
}

// 2-D bf16 tensor map {inner, rows} with row stride `ld` elements, box {64, box_rows},
// 128-byte swizzle, out-of-range elements read as zero.
lora_status make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t ld,
                     uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    lora_status st = encode_fn(&enc);
    if (st != LORA_OK) return st;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = 10000 + (int)r;
        return LORA_ECUDA;
    }
    return LORA_OK;
}

// Shared-memory plan of the tensor-core kernel for this pool.
struct MmaConfig {
    int rp_max, s1, s2, s3, s1_bytes, s2_bytes;
    size_t smem;
};

lora_status mma_config(const lora_pool* pool, int smem_optin, MmaConfig* c) {
    const lora_pool_desc& d = pool->d;
    c->rp_max = mma_rpad(d.r_max < kMmaMaxRank ? d.r_max : kMmaMaxRank);
    c->s1_bytes = (16384 + c->rp_max * 128 + 1023) / 1024 * 1024;   // x chunk + A chunk
    c->s2_bytes = (c->rp_max * 256 + 1023) / 1024 * 1024;           // B^T slice
    // the deepest y ring (<= 3) that leaves the shrink ring two stages, and the rest to
    // the shrink ring (the next tile's shrink streams under this tile's expand and must
    // end with it); B^T ring of 2.  On the Llama-7B prefill a 3-slot y ring with a 4-stage
    // shrink ring beat both 4 + 2 (13% slower) and 2 + 6 (18% slower).
    c->s2 = 2;
    const int s3_max = pool->tune.mma_y_stages;   // 3 unless the pool's tuning says otherwise
    for (c->s3 = s3_max; c->s3 >= 2; --c->s3) {
        for (c->s1 = kMmaMaxStages; c->s1 >= 2; --c->s1) {
            c->smem = mma_smem_layout(c->s1, c->s1_bytes, c->s2, c->s2_bytes, c->s3).total + 1024;
            if (c->smem <= (size_t)smem_optin) break;
        }
        if (c->s1 >= 2) break;
    }
    return c->s1 < 2 ? LORA_ETOOBIG : LORA_OK;
}

lora_status fill_mma(MmaParams& prm, const lora_pool* pool, const lora_problem* probs, int32_t n, int32_t T,
                     void* ws, const MmaConfig& c) {
    const lora_pool_desc& d = pool->d;
    memset(&prm, 0, sizeof prm);
    lora_status st = make_map(&prm.pool_map, d.pages, (uint64_t)d.h, (uint64_t)d.num_pages, (uint64_t)d.h, 1);
    if (st != LORA_OK) return st;
    for (int32_t i = 0; i < n; ++i) {
        const lora_problem& pr = probs[i];
        const int32_t di = pool->d_in[pr.proj], dq = pool->d_out[pr.proj];
        st = make_map(&prm.x_map[i], pr.x, (uint64_t)di, (uint64_t)T, (uint64_t)pr.ldx, kMmaRowBlock);
        if (st != LORA_OK) return st;
        st = make_map(&prm.y_map[i], pr.y, (uint64_t)dq, (uint64_t)T, (uint64_t)pr.ldy, kMmaRowBlock);
        if (st != LORA_OK) return st;
        st = make_map(&prm.y1_map[i], pr.y, (uint64_t)dq, (uint64_t)T, (uint64_t)pr.ldy, 1);
        if (st != LORA_OK) return st;
        prm.blk[i] = pr.layer * pool->units + pool->pre[pr.proj];
        prm.n_kc[i] = (int16_t)(di / kMmaKChunk);
        prm.n_nt[i] = (int16_t)(dq / kMmaNTile);
        prm.pv_in[i] = (uint8_t)vec_pages(di, d.h);
        prm.pv_out[i] = (uint8_t)vec_pages(dq, d.h);
    }
    // runs of consecutive problems reading the same x form the item order's groups
    for (int32_t i = 0; i < n;) {
        int32_t j = i + 1;
        while (j < n && probs[j].x == probs[i].x && probs[j].ldx == probs[i].ldx) ++j;
        for (int32_t k = i; k < j; ++k) {
            prm.xgrp_off[k] = (uint8_t)(k - i);
            prm.xgrp_size[k] = (uint8_t)(j - i);
        }
        i = j;
    }
    prm.pool = view_of(pool);
    prm.ws = reinterpret_cast<char*>(ws);
    prm.nprob = n;
    prm.s1 = c.s1;
    prm.s2 = c.s2;
    prm.s3 = c.s3;
    prm.s1_bytes = c.s1_bytes;
    prm.s2_bytes = c.s2_bytes;
    prm.rp_max = c.rp_max;
    return LORA_OK;
}

template <int MAXP>
void fill_ring(RingParamsT<MAXP>& prm, const lora_pool* pool, const lora_problem* probs, int32_t n, void* ws,
               float* t_out, int stages, int rows_per_stage) {
    const lora_pool_desc& d = pool->d;
    memset(&prm, 0, sizeof prm);
    prm.pool = view_of(pool);
    prm.ws = reinterpret_cast<char*>(ws);
    prm.t_out = t_out;
    prm.nprob = n;
    prm.stages = stages;
    prm.stage_bytes = rows_per_stage * 2 * d.h;
    for (int32_t i = 0; i < n; ++i) {
        prm.probs[i] = prob_desc(pool, probs[i]);
    }
}

// Balanced batches of at most `cap` problems (no short last launch).
int32_t batch_size(int32_t nprob, int32_t cap) {
    const int32_t nb = (nprob + cap - 1) / cap;
    return (nprob + nb - 1) / nb;
}

lora_status run_mma(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                    cudaStream_t stream) {
    if (T <= 0 || nprob <= 0) return LORA_OK;
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    MmaConfig c;
    st = mma_config(pool, di->smem_optin, &c);
    if (st != LORA_OK) return st;
    static thread_local MmaParams prm;
    static thread_local int attr_dev = -1;
    static thread_local size_t attr_smem = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = pool->square ? sgmv_mma_kernel<false> : sgmv_mma_kernel<true>;
    if (attr_dev != dev || attr_smem < c.smem) {
        for (auto k : {sgmv_mma_kernel<false>, sgmv_mma_kernel<true>}) {
            st = cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem));
            if (st != LORA_OK) return st;
        }
        attr_dev = dev;
        attr_smem = c.smem;
    }
    const int32_t per = batch_size(nprob, kMmaMaxProbs);
    for (int32_t base = 0; base < nprob; base += per) {
        const int32_t n = nprob - base < per ? nprob - base : per;
        st = fill_mma(prm, pool, probs + base, n, T, ws, c);
        if (st != LORA_OK) return st;
        kern<<<di->sm_count, kMmaThreads, c.smem, stream>>>(prm);
        st = cuda_status(cudaGetLastError());
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

// Per-CTA byte rate of the ring body relative to the tensor-core body in the fused launch,
// measured on the 13B mixed step (ring CTAs split by bytes alone ended 18% before the
// tensor-core ones; 1.0 / 1.1 / 1.22 / 1.35 / 1.5: 11.67 / 11.29 / 11.18 / 11.42 / 12.95 ms).
// Pools with projections of other widths: the ring body streams multi-page vectors (an x
// block and an A page per input page block), and the tensor-core body's wide shapes (gate,
// up, down) run at their own rate; measured on the Llama-3-8B mixed step with the tile
// items taken from a queue and three D1 buffers (0.85 / 1.0 / 1.15: 1.904 / 1.869 / 1.879
// ms on one box; 0.85 / 1.0: 1.902 / 1.855 and 1.864 / 1.852 ms on two others).
float default_fused_ring_speed(bool square) { return square ? 1.22f : 1.0f; }

// Both work classes in one launch per batch of projections (h <= 5120, h % 128 == 0); the
// ring body takes the stage shape the stand-alone ring kernel would take.
template <int NV, int CW, int RP, bool W>
lora_status launch_fused_rp(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T,
                            void* ws, const DeviceInfo* di, const MmaConfig& c, const RingShape& sh,
                            cudaStream_t stream) {
    const size_t smem = c.smem > sh.smem ? c.smem : sh.smem;
    static thread_local FusedParams prm;
    const float ring_speed = pool->tune.fused_ring_speed;   // see default_fused_ring_speed
    static thread_local int attr_dev = -1;
    static thread_local size_t attr_smem = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = delta_fused_kernel<NV, CW, RP, W>;
    lora_status st;
    if (attr_dev != dev || attr_smem < smem) {
        st = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (st != LORA_OK) return st;
        attr_dev = dev;
        attr_smem = smem;
    }
    const int32_t per = batch_size(nprob, kMmaMaxProbs);
    for (int32_t base = 0; base < nprob; base += per) {
        const int32_t n = nprob - base < per ? nprob - base : per;
        st = fill_mma(prm.mma, pool, probs + base, n, T, ws, c);
        if (st != LORA_OK) return st;
        fill_ring(prm.ring, pool, probs + base, n, ws, nullptr, sh.stages, RP);
        prm.ring_speed = ring_speed;
        prm.row_elems = prm.page_elems = 0;
        for (int32_t i = base; i < base + n; ++i) {
            const int64_t di = pool->d_in[probs[i].proj], dq = pool->d_out[probs[i].proj];
            prm.row_elems += (unsigned long long)(di + 2 * dq);
            prm.page_elems += (unsigned long long)(di + dq);
        }
        kern<<<di->sm_count, kMmaThreads, smem, stream>>>(prm);
        st = cuda_status(cudaGetLastError());
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

template <int NV, int CW>
lora_status launch_fused(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                         cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    MmaConfig c;
    st = mma_config(pool, di->smem_optin, &c);
    if (st != LORA_OK) return st;
    const RingShape sh = ring_shape(pool->d.h, pool->d.r_max, di->smem_optin, CW, pool->tune.ring_rows_per_stage,
                                    kMmaMaxProbs);
    if (sh.stages < 2) return LORA_ETOOBIG;
    if (!pool->square) {
        if (sh.rp == kRingPagesLarge)
            return launch_fused_rp<NV, CW, kRingPagesLarge, true>(pool, probs, nprob, T, ws, di, c, sh, stream);
        return launch_fused_rp<NV, CW, kRingPagesSmall, true>(pool, probs, nprob, T, ws, di, c, sh, stream);
    }
    if (sh.rp == kRingPagesLarge)
        return launch_fused_rp<NV, CW, kRingPagesLarge, false>(pool, probs, nprob, T, ws, di, c, sh, stream);
    return launch_fused_rp<NV, CW, kRingPagesSmall, false>(pool, probs, nprob, T, ws, di, c, sh, stream);
}

// One launch per batch of projections for both work classes (h <= 5120).
lora_status run_fused(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                      cudaStream_t stream) {
    const int h8 = pool->d.h / 8;
    if (h8 <= 256) return launch_fused<1, 8>(pool, probs, nprob, T, ws, stream);
    if (h8 <= 512) return launch_fused<2, 8>(pool, probs, nprob, T, ws, stream);
    return launch_fused<2, 10>(pool, probs, nprob, T, ws, stream);
}

}  // namespace host
}  // namespace lora
