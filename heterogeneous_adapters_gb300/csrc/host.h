// Host-side launch plumbing shared by the translation units of liblora.so: the pool's
// host record, device facts, kernel-parameter helpers, and the launch entry points of each
// kernel family (launch_ring.cu: the CUDA-core ring kernel; launch_tile.cu: the
// tensor-core tile kernel and the fused launch; launch_cluster.cu: the cluster kernel for
// launches of few projections).  The C ABI itself lives in lora_api.cu.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "common.cuh"
#include "lora.h"

struct lora_pool {
    lora_pool_desc d;                 // proj_dims is not kept (a host array of the caller)
    std::vector<int32_t> d_in, d_out; // widths of each projection
    std::vector<int32_t> pre;         // units before each projection in a layer
    int32_t units = 0;                // units of one layer
    bool square = true;               // every projection h x h
    bool mma_widths = true;           // every d_in % 64 == 0 and d_out % 128 == 0 (tile shapes)
    lora_tuning tune{};               // launch tuning, defaults resolved (lora_pool_set_tuning)
};

namespace lora {
namespace host {

extern thread_local int g_last_cuda_error;
lora_status cuda_status(cudaError_t e);
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Kernel views of the pool and of one problem.
PoolView view_of(const lora_pool* pool);
ProbDesc prob_desc(const lora_pool* pool, const lora_problem& pr);

// Per-device launch facts, looked up once per device.
struct DeviceInfo {
    int sm_count = 0;
    int smem_optin = 0;
    bool ready = false;
};
constexpr int kMaxDevices = 64;
lora_status device_info(DeviceInfo** out);

// Shape of the ring for one launch: rows per stage, depth and the shared memory it takes.
struct RingShape {
    int rp, stages;
    size_t smem;
};
// force_rp: 4 or 8 rows per stage where two such stages fit; 0 = automatic.  nprob: the
// most problem descriptors a launch copies into shared memory.
RingShape ring_shape(int h, int r_max, int smem_optin, int cwarps, int force_rp, int nprob);

// launch_ring.cu: the CUDA-core kernel over the chunk list (t_out: debug export of t).
lora_status run_delta_ring(const lora_pool* pool, const lora_problem* probs, int32_t nprob, void* ws,
                           float* t_out, cudaStream_t stream);

// launch_tile.cu: the tensor-core kernel over the tile list, and the fused launch of both
// work classes (h <= 5120).
int mma_min_rows(const lora_pool* pool);
float default_fused_ring_speed(bool square);
lora_status run_mma(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                    cudaStream_t stream);
lora_status run_fused(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                      cudaStream_t stream);

// launch_cluster.cu: the cluster kernel for launches of few projections (no workspace
// beyond the grouping).
bool cluster_fits(const lora_pool* pool, int32_t nprob);
lora_status run_cluster(const lora_pool* pool, const lora_problem* probs, int32_t nprob, void* ws,
                        cudaStream_t stream);
// The separate shrink (expand = false: t = s * x A^T into t) or expand (y += t B^T) over the
// CUDA-core chunks of the grouping in ws; t is fp32 [nprob][T][r_max].
lora_status run_shrink_expand(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T,
                              void* ws, float* t, bool expand, cudaStream_t stream);

}  // namespace host
}  // namespace lora
