// Launches of the CUDA-core decode kernel (bgmv_ring.cuh): the ring's stage shape and the
// kernel instantiation for h and for pools with or without projections of other widths.
#include <string.h>

#include "bgmv_ring.cuh"
#include "host.h"

namespace lora {
namespace host {

// Ring depth that fits the opt-in shared memory of one CTA (at most 8 stages).
int ring_stages(int smem_optin, int stage_bytes, int r_max, int cwarps, int nprob, size_t* smem) {
    for (int S = 8; S >= 2; --S) {
        const size_t need = ring_smem_layout(S, stage_bytes, r_max, cwarps, nprob).total + 1024;
        if (need <= (size_t)smem_optin) {
            *smem = need;
            return S;
        }
    }
    return 0;
}

// Rows per stage: the larger stages when three of them fit (a bulk-copy ring streams
// closer to the HBM read rate with fewer, larger stages), else the small ones.
// force = 4 or 8 (the pool's tuning) forces the choice where two such stages fit.
RingShape ring_shape(int h, int r_max, int smem_optin, int cwarps, int force, int nprob) {
    RingShape fallback{0, 0, 0};
    for (int rp : {kRingPagesLarge, kRingPagesSmall}) {
        size_t smem = 0;
        const int S = ring_stages(smem_optin, rp * 2 * h, r_max, cwarps, nprob, &smem);
        if (S < 2) continue;
        const RingShape sh{rp, S, smem};
        if (force == rp || (force == 0 && S >= 3)) return sh;
        if (fallback.stages == 0) fallback = sh;
    }
    return fallback;
}

template <int NV, int CW, int RP, bool W>
lora_status launch_ring_rp(RingParams& prm, const DeviceInfo* di, const RingShape& sh, cudaStream_t stream) {
    static thread_local int attr_dev = -1;
    static thread_local size_t attr_smem = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    prm.stage_bytes = RP * 2 * prm.pool.h;
    prm.stages = sh.stages;
    const size_t smem = sh.smem;
    auto kern = bgmv_ring_kernel<NV, CW, RP, W>;
    if (attr_dev != dev || attr_smem < smem) {
        lora_status st = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (st != LORA_OK) return st;
        attr_dev = dev;
        attr_smem = smem;
    }
    kern<<<di->sm_count, CW * 32 + 32, smem, stream>>>(prm);
    return cuda_status(cudaGetLastError());
}

template <int NV, int CW, bool W>
lora_status launch_ring_w(RingParams& prm, int force_rp, cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    const RingShape sh = ring_shape(prm.pool.h, prm.pool.r_max, di->smem_optin, CW, force_rp, prm.nprob);
    if (sh.stages < 2) return LORA_ETOOBIG;
    if (sh.rp == kRingPagesLarge) return launch_ring_rp<NV, CW, kRingPagesLarge, W>(prm, di, sh, stream);
    return launch_ring_rp<NV, CW, kRingPagesSmall, W>(prm, di, sh, stream);
}

// h x h pools take the kernels compiled for one page block per vector
template <int NV, int CW>
lora_status launch_ring(RingParams& prm, const lora_pool* pool, cudaStream_t stream) {
    const int rp = pool->tune.ring_rows_per_stage;
    return pool->square ? launch_ring_w<NV, CW, false>(prm, rp, stream) : launch_ring_w<NV, CW, true>(prm, rp, stream);
}

lora_status run_delta_ring(const lora_pool* pool, const lora_problem* probs, int32_t nprob, void* ws,
                           float* t_out, cudaStream_t stream) {
    const lora_pool_desc& d = pool->d;
    static thread_local RingParams prm;
    for (int32_t base = 0; base < nprob; base += LORA_MAX_PROBLEMS_PER_LAUNCH) {
        const int32_t n = nprob - base < LORA_MAX_PROBLEMS_PER_LAUNCH ? nprob - base
                                                                         : LORA_MAX_PROBLEMS_PER_LAUNCH;
        memset(&prm, 0, sizeof prm);
        prm.pool = view_of(pool);
        prm.ws = reinterpret_cast<char*>(ws);
        prm.t_out = t_out;
        prm.nprob = n;
        for (int32_t i = 0; i < n; ++i) {
            prm.probs[i] = prob_desc(pool, probs[base + i]);
        }
        // consumer warps x vectors per thread cover the h / 8 16-byte vectors of a row
        const int h8 = d.h / 8;
        lora_status st;
        if (h8 <= 256)
            st = launch_ring<1, 8>(prm, pool, stream);
        else if (h8 <= 512)
            st = launch_ring<1, 16>(prm, pool, stream);
        else if (h8 <= 640)
            st = launch_ring<2, 10>(prm, pool, stream);
        else if (h8 <= 768)
            st = launch_ring<2, 12>(prm, pool, stream);
        else
            st = launch_ring<2, 16>(prm, pool, stream);
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

}  // namespace host
}  // namespace lora
