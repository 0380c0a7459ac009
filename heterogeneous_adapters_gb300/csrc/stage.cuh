// Adapter staging: copy page rows from pinned host memory into pool pages and rewrite
// the page-table entries that point at them, in one kernel on a side stream.
//
// "S-LoRA: Serving Thousands of Concurrent LoRA Adapters", "Host memory for adapters":
// adapters live in host memory and the ones the batch needs are copied to the GPU,
// prefetched during the current step.  "Multi-LoRA serving: S-LoRA, Punica and adapter
// batching", "What the engine does each step": on a miss the engine evicts an unused
// adapter and copies the new one over the host link; requests wait for that copy.
//
// The source rows are read straight from host memory (pinned host memory is addressable
// from the GPU with the same pointer), 16 bytes per thread per load, many loads in
// flight per SM; a consumer kernel on another stream orders itself after the copy with
// an event recorded after this kernel.
#pragma once
#include "common.cuh"

namespace lora {

constexpr int kStageThreads = 256;

struct StageParams {
    const uint4* host_rows;      // [npages][2h / 16]
    const int32_t* dst_pages;    // [npages] (host-pinned or device)
    __nv_bfloat16* pages;        // pool
    int32_t* pt;                 // writable page table
    const int64_t* upd_index;    // [nupd] page-table entries to rewrite
    const int32_t* upd_page;     // [nupd] their new page ids
    int64_t nupd;
    int32_t npages;
    int32_t vec_per_row;         // 2h / 16
};

__global__ void __launch_bounds__(kStageThreads) stage_kernel(const StageParams p) {
    for (int32_t i = blockIdx.x; i < p.npages; i += gridDim.x) {
        const uint4* src = p.host_rows + (size_t)i * p.vec_per_row;
        uint4* dst = reinterpret_cast<uint4*>(p.pages + (size_t)p.dst_pages[i] * (p.vec_per_row * 8));
        constexpr int kUnroll = 4;
        for (int v0 = threadIdx.x; v0 < p.vec_per_row; v0 += kStageThreads * kUnroll) {
            uint4 buf[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * kStageThreads;
                if (v < p.vec_per_row) buf[u] = src[v];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * kStageThreads;
                if (v < p.vec_per_row) dst[v] = buf[u];
            }
        }
    }
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t k = tid; k < p.nupd; k += (int64_t)gridDim.x * blockDim.x) p.pt[p.upd_index[k]] = p.upd_page[k];
}

}  // namespace lora
