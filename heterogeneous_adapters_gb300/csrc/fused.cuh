// One delta launch for a batch that holds both work classes (prefill segments long enough
// for the tensor cores, and decode tokens / short segments for the CUDA-core ring).
//
// "Multi-LoRA serving: S-LoRA, Punica and adapter batching", "What the engine does each
// step": a continuous-batching step mixes requests in prefill and in decode; SGMV suits
// the former and BGMV the latter.  Here both run in the same persistent grid: the CTAs
// are split between the two bodies in proportion to the bytes each class streams per
// projection (weights written by the grouping kernel), so the two HBM streams proceed
// side by side and end together instead of one after the other.  A CTA of the ring body
// streams bytes faster than one of the tensor-core body (it only reads pages, where the
// other also reads and writes y in place), so the split weighs the two byte counts by their
// per-CTA rates.
#pragma once
#include "bgmv_ring.cuh"
#include "sgmv_mma.cuh"

namespace lora {

struct FusedParams {
    MmaParams mma;
    RingParamsT<kMmaMaxProbs> ring;
    float ring_speed;   // bytes per CTA-second of the ring body / those of the tensor-core body
    // over the launch's projections: sum of (d_in + 2 d_out) and of (d_in + d_out), the
    // elements streamed per adapted row and per page row
    unsigned long long row_elems, page_elems;
};
static_assert(sizeof(FusedParams) <= 32764, "kernel parameters are limited to 32,764 bytes");

// CTAs given to the CUDA-core class out of G (0 if it has no work, G if the tensor-core
// class has none; otherwise at least one each), so that both classes' CTAs need about the
// same time: G * (wf / speed) / (wf / speed + wm), w the bytes each class streams.
__device__ __forceinline__ uint32_t fused_split(const WsHeader* hdr, const FusedParams& p, uint32_t G) {
    const float ring_speed = p.ring_speed;
    const unsigned long long wf = hdr->rows[0] * p.row_elems + hdr->page_rows[0] * p.page_elems;
    const unsigned long long wm = hdr->rows[1] * p.row_elems + hdr->page_rows[1] * p.page_elems;
    if (wm == 0) return G;
    if (wf == 0) return 0;
    const double tf = (double)wf / (double)ring_speed;
    uint32_t gf = (uint32_t)((double)G * tf / (tf + (double)wm) + 0.5);
    if (gf < 1) gf = 1;
    if (gf > G - 1) gf = G - 1;
    return gf;
}

// W: projections whose widths differ from h (the ring body's W instantiation).
template <int NV, int CW, int RP, bool W>
__global__ void __launch_bounds__(kMmaThreads, 1) delta_fused_kernel(const __grid_constant__ FusedParams p) {
    static_assert(CW * 32 + 32 <= kMmaThreads, "ring body must fit the fused CTA");
    extern __shared__ __align__(1024) unsigned char fused_smem_raw[];
    const uint32_t gf = fused_split(reinterpret_cast<const WsHeader*>(p.mma.ws), p, gridDim.x);
    if (blockIdx.x < gf)
        ring_cta<NV, CW, RP, W>(p.ring, fused_smem_raw, blockIdx.x, gf);
    else
        mma_cta<W>(p.mma, fused_smem_raw, gridDim.x - gf);
}

}  // namespace lora
