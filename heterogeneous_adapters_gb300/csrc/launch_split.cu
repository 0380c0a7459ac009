// Launches of the two-phase CUDA-core kernels (bgmv_split.cuh) for launches of few
// projections of a decode-sized batch.
#include <string.h>

#include <algorithm>

#include "bgmv_split.cuh"
#include "host.h"

namespace lora {
namespace host {

// Workspace bytes the split path's t takes for batches of up to max_tokens rows (none
// above kSplitMaxTokens: larger batches never take that path).
size_t split_t_bytes(const lora_pool_desc& d, int32_t max_tokens) {
    if (max_tokens > kSplitMaxTokens) return 0;
    return (size_t)kSplitMaxProbs * (size_t)max_tokens * (size_t)d.r_max * sizeof(float);
}

// The two-phase CUDA-core path serves launches of few projections of a decode-sized batch
// (a chunk of one projection per CTA would leave most SMs idle), when the workspace has
// room for its t.  The pool's tuning sets the projection limit (0 turns the path off).
bool split_fits(const lora_pool* pool, int32_t nprob, int32_t T, size_t ws_bytes) {
    const int max_p = std::min(pool->tune.split_max_problems, kSplitMaxProbs);
    if (nprob < 1 || nprob > max_p || T < 1 || T > kSplitMaxTokens) return false;
    // the grouping laid the workspace out for (T, segments); decode segments number at most T
    return ws_bytes >= ws_layout(T, T).total + split_t_bytes(pool->d, T);
}

template <bool W>
lora_status launch_split(const SplitParams& prm, const DeviceInfo* di, cudaStream_t stream) {
    const int grid = di->sm_count * 4;
    const size_t xs_bytes = (size_t)kChunk * prm.pool.h * 2;   // the chunk's x rows
    static thread_local int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        lora_status st = cuda_status(cudaFuncSetAttribute(split_shrink_kernel<W>,
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                          (int)(kChunk * 8192 * 2)));   // h <= 8192
        if (st != LORA_OK) return st;
        attr_dev = dev;
    }
    split_shrink_kernel<W><<<grid, kSplitThreads, xs_bytes, stream>>>(prm);
    lora_status st = cuda_status(cudaGetLastError());
    if (st != LORA_OK) return st;
    split_expand_kernel<W><<<grid, kSplitThreads, 0, stream>>>(prm);
    return cuda_status(cudaGetLastError());
}

lora_status run_split(const lora_pool* pool, const lora_problem* probs, int32_t nprob, void* ws,
                      cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    static thread_local SplitParams prm;
    memset(&prm, 0, sizeof prm);
    prm.pool = view_of(pool);
    prm.ws = reinterpret_cast<char*>(ws);
    prm.nprob = nprob;
    prm.out_blocks = 1;
    for (int32_t i = 0; i < nprob; ++i) {
        prm.probs[i] = prob_desc(pool, probs[i]);
        prm.out_blocks = std::max(prm.out_blocks, vec_pages(prm.probs[i].d_out, pool->d.h));
    }
    return pool->square ? launch_split<false>(prm, di, stream) : launch_split<true>(prm, di, stream);
}

}  // namespace host
}  // namespace lora
