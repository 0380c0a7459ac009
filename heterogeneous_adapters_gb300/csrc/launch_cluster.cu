// Launches of the cluster kernel (bgmv_cluster.cuh) for launches of few projections of a
// decode batch, and of the separate shrink and expand kernels (shrink_expand.cuh).
#include <string.h>

#include <algorithm>

#include "bgmv_cluster.cuh"
#include "host.h"
#include "shrink_expand.cuh"

namespace lora {
namespace host {

// Launches of at most the pool's split_max_problems projections: one chunk of one projection
// per CTA would leave most SMs idle, and one SM alone takes ~20 us to stream a rank-64
// chunk's pages.
bool cluster_fits(const lora_pool* pool, int32_t nprob) {
    const int max_p = std::min(pool->tune.split_max_problems, kClusterMaxProbs);
    return nprob >= 1 && nprob <= max_p;
}

template <bool W>
lora_status launch_cluster(const ClusterParams& prm, size_t smem, const DeviceInfo* di, cudaStream_t stream) {
    static thread_local int attr_dev = -1;
    static thread_local size_t attr_smem = 0;
    static thread_local int clusters = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = bgmv_cluster_kernel<W>;
    if (attr_dev != dev || attr_smem < smem) {
        lora_status st = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (st != LORA_OK) return st;
        // as many clusters as are resident at once (the kernel loops over its items)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kClusterCtas * di->sm_count, 1, 1);
        cfg.blockDim = dim3(kClusterThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        int n = 0;
        st = cuda_status(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
        if (st != LORA_OK) return st;
        clusters = n > 0 ? n : std::max(1, di->sm_count / kClusterCtas);
        attr_dev = dev;
        attr_smem = smem;
    }
    kern<<<clusters * kClusterCtas, kClusterThreads, smem, stream>>>(prm);
    return cuda_status(cudaGetLastError());
}

lora_status run_cluster(const lora_pool* pool, const lora_problem* probs, int32_t nprob, void* ws,
                        cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    static thread_local ClusterParams prm;
    memset(&prm, 0, sizeof prm);
    prm.pool = view_of(pool);
    prm.ws = reinterpret_cast<char*>(ws);
    prm.nprob = nprob;
    int in8 = 1, out8 = 1, pv = 2;
    for (int32_t i = 0; i < nprob; ++i) {
        prm.probs[i] = prob_desc(pool, probs[i]);
        in8 = std::max(in8, prm.probs[i].d_in / 8);
        out8 = std::max(out8, prm.probs[i].d_out / 8);
        pv = std::max(pv, vec_pages(prm.probs[i].d_in, pool->d.h) + vec_pages(prm.probs[i].d_out, pool->d.h));
    }
    prm.ni = (in8 + kClusterCtas - 1) / kClusterCtas;
    prm.no = (out8 + kClusterCtas - 1) / kClusterCtas;
    prm.pv_max = pv;
    const size_t smem = cluster_smem_layout(prm.ni, pool->d.r_max, pv).total;
    if (smem > (size_t)di->smem_optin) return LORA_ETOOBIG;
    return pool->square ? launch_cluster<false>(prm, smem, di, stream) : launch_cluster<true>(prm, smem, di, stream);
}

// Shrink (expand = false) or expand of up to 8 projections per launch, t in the caller's
// buffer [problem][row][r_max].
template <bool W>
lora_status launch_sx(const ShrinkExpandParams& prm, bool expand, const DeviceInfo* di, cudaStream_t stream) {
    const int grid = di->sm_count * 4;
    static thread_local int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        lora_status st = cuda_status(cudaFuncSetAttribute(lora_shrink_kernel<W>,
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                          (int)(kChunk * 8192 * 2)));   // h <= 8192
        if (st != LORA_OK) return st;
        attr_dev = dev;
    }
    if (expand)
        lora_expand_kernel<W><<<grid, kSxThreads, 0, stream>>>(prm);
    else
        lora_shrink_kernel<W><<<grid, kSxThreads, (size_t)kChunk * prm.pool.h * 2, stream>>>(prm);
    return cuda_status(cudaGetLastError());
}

lora_status run_shrink_expand(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T,
                              void* ws, float* t, bool expand, cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    static thread_local ShrinkExpandParams prm;
    for (int32_t base = 0; base < nprob; base += kSxMaxProbs) {
        const int32_t n = std::min(kSxMaxProbs, nprob - base);
        memset(&prm, 0, sizeof prm);
        prm.pool = view_of(pool);
        prm.ws = reinterpret_cast<char*>(ws);
        prm.t = t + (size_t)base * T * pool->d.r_max;
        prm.T = T;
        prm.nprob = n;
        prm.out_blocks = 1;
        for (int32_t i = 0; i < n; ++i) {
            prm.probs[i] = prob_desc(pool, probs[base + i]);
            prm.out_blocks = std::max(prm.out_blocks, vec_pages(prm.probs[i].d_out, pool->d.h));
        }
        st = pool->square ? launch_sx<false>(prm, expand, di, stream) : launch_sx<true>(prm, expand, di, stream);
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

}  // namespace host
}  // namespace lora
