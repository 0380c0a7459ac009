// C ABI of liblora.so (declarations and contracts in include/lora.h).
//
// Host side: argument checks, workspace layout, launch configuration.  All compute
// runs in the kernels of segment.cuh and fma_delta.cuh (and the tensor-core kernel
// when present); nothing here touches adapter or activation values.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "fma_delta.cuh"
#include "segment.cuh"

using namespace lora;

struct lora_pool {
    lora_pool_desc d;
};

namespace {

thread_local int g_last_cuda_error = 0;

lora_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LORA_OK;
    g_last_cuda_error = (int)e;
    return LORA_ECUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

PoolView view_of(const lora_pool* pool) {
    const lora_pool_desc& d = pool->d;
    PoolView v;
    v.pages = reinterpret_cast<const __nv_bfloat16*>(d.pages);
    v.num_pages = d.num_pages;
    v.pt = d.page_table;
    v.pt_len = d.page_table_len;
    v.pt_off = d.adapter_pt_off;
    v.ranks = d.ranks;
    v.scales = d.scales;
    v.h = d.h;
    v.num_adapters = d.num_adapters;
    v.num_layers = d.num_layers;
    v.num_proj = d.num_proj;
    v.r_max = d.r_max;
    v.pad = 0;
    return v;
}

// Per-device launch facts, looked up once per device.
struct DeviceInfo {
    int sm_count = 0;
    bool ready = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

lora_status device_info(DeviceInfo** out) {
    int dev = 0;
    lora_status st = cuda_status(cudaGetDevice(&dev));
    if (st != LORA_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return LORA_ETOOBIG;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        st = cuda_status(cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev));
        if (st != LORA_OK) return st;
        di.ready = true;
    }
    *out = &di;
    return LORA_OK;
}

lora_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr || ((uintptr_t)ws & 255u) != 0) return LORA_EWORKSPACE;
    if (ws_bytes < need) return LORA_EWORKSPACE;
    return LORA_OK;
}

// Launch the CUDA-core delta kernel for one group of <= LORA_MAX_PROBLEMS_PER_LAUNCH
// problems.  The grid is persistent: (resident CTAs per SM) x (SM count).
template <int NV, int JU>
lora_status launch_fma(const DeltaParams& prm, size_t smem, cudaStream_t stream) {
    static thread_local int attr_set_dev = -1;
    static thread_local size_t attr_smem = 0;
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = fma_delta_kernel<NV, JU>;
    if (attr_set_dev != dev || attr_smem < smem) {
        st = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)smem));
        if (st != LORA_OK) return st;
        attr_set_dev = dev;
        attr_smem = smem;
    }
    int per_sm = 0;
    st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFmaThreads, smem));
    if (st != LORA_OK) return st;
    if (per_sm < 1) per_sm = 1;
    kern<<<per_sm * di->sm_count, kFmaThreads, smem, stream>>>(prm);
    return cuda_status(cudaGetLastError());
}

lora_status run_delta(const lora_pool* pool, const lora_problem* probs, int32_t nprob, void* ws,
                      float* t_out, cudaStream_t stream) {
    const lora_pool_desc& d = pool->d;
    // host-side checks of every problem before any launch
    for (int32_t i = 0; i < nprob; ++i) {
        const lora_problem& pr = probs[i];
        if (pr.x == nullptr || pr.y == nullptr) return LORA_EINVAL;
        if (!aligned16(pr.x) || !aligned16(pr.y)) return LORA_EALIGN;
        if (pr.ldx % 8 != 0 || pr.ldy % 8 != 0) return LORA_EALIGN;
        if (pr.ldx < d.h || pr.ldy < d.h || pr.ldx > INT32_MAX || pr.ldy > INT32_MAX)
            return LORA_EINVAL;
        if (pr.layer < 0 || pr.layer >= d.num_layers || pr.proj < 0 || pr.proj >= d.num_proj)
            return LORA_EINVAL;
    }
    const size_t smem = fma_smem_bytes(d.r_max);
    static thread_local DeltaParams prm;   // ~8 KiB: keep it off the stack
    for (int32_t base = 0; base < nprob; base += LORA_MAX_PROBLEMS_PER_LAUNCH) {
        const int32_t n = nprob - base < LORA_MAX_PROBLEMS_PER_LAUNCH ? nprob - base
                                                                         : LORA_MAX_PROBLEMS_PER_LAUNCH;
        memset(&prm, 0, sizeof prm);
        prm.pool = view_of(pool);
        prm.ws = reinterpret_cast<char*>(ws);
        prm.t_out = t_out;
        prm.nprob = n;
        for (int32_t i = 0; i < n; ++i) {
            const lora_problem& pr = probs[base + i];
            prm.probs[i].x = reinterpret_cast<const __nv_bfloat16*>(pr.x);
            prm.probs[i].y = reinterpret_cast<__nv_bfloat16*>(pr.y);
            prm.probs[i].ldx = (int32_t)pr.ldx;
            prm.probs[i].ldy = (int32_t)pr.ldy;
            prm.probs[i].blk = pr.layer * d.num_proj + pr.proj;
        }
        lora_status st;
        if (d.h <= 4096)
            st = launch_fma<1, 8>(prm, smem, stream);
        else
            st = launch_fma<2, 4>(prm, smem, stream);
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

}  // namespace

extern "C" {

const char* lora_status_string(lora_status s) {
    switch (s) {
        case LORA_OK: return "ok";
        case LORA_EINVAL: return "invalid argument";
        case LORA_EALIGN: return "misaligned pointer or leading dimension";
        case LORA_EWORKSPACE: return "workspace missing, misaligned or too small";
        case LORA_ETOOBIG: return "size beyond a documented maximum";
        case LORA_ECUDA: return "CUDA runtime error";
        case LORA_EDEVICE: return "device-detected data error";
    }
    return "unknown status";
}

int lora_last_cuda_error(void) { return g_last_cuda_error; }

lora_status lora_pool_create(lora_pool** out, const lora_pool_desc* desc) {
    if (out == nullptr || desc == nullptr) return LORA_EINVAL;
    *out = nullptr;
    const lora_pool_desc& d = *desc;
    if (d.pages == nullptr || d.page_table == nullptr || d.adapter_pt_off == nullptr ||
        d.ranks == nullptr || d.scales == nullptr)
        return LORA_EINVAL;
    if (d.num_pages <= 0 || d.h <= 0 || d.num_adapters <= 0 || d.num_layers <= 0 ||
        d.num_proj <= 0 || d.page_table_len <= 0 || d.r_max <= 0)
        return LORA_EINVAL;
    if (d.h % 8 != 0 || !aligned16(d.pages)) return LORA_EALIGN;
    if (d.r_max > LORA_MAX_RANK || d.h > 8192) return LORA_ETOOBIG;
    if (d.num_pages > INT32_MAX || d.num_pages > INT64_MAX / d.h) return LORA_ETOOBIG;
    if ((int64_t)d.num_layers * d.num_proj > (1 << 20)) return LORA_ETOOBIG;
    lora_pool* p = (lora_pool*)malloc(sizeof(lora_pool));
    if (p == nullptr) return LORA_EINVAL;
    p->d = d;
    *out = p;
    return LORA_OK;
}

lora_status lora_pool_destroy(lora_pool* pool) {
    free(pool);
    return LORA_OK;
}

lora_status lora_workspace_size(const lora_pool* pool, int32_t max_tokens, int32_t max_segments,
                                size_t* bytes) {
    if (pool == nullptr || bytes == nullptr || max_tokens < 0 || max_segments < 0)
        return LORA_EINVAL;
    if (max_segments > LORA_MAX_SEGMENTS || max_tokens > (1 << 28)) return LORA_ETOOBIG;
    *bytes = ws_layout(max_tokens, max_segments).total;
    return LORA_OK;
}

lora_status lora_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    return cuda_status(cudaMemsetAsync(ws, 0, sizeof(WsHeader), (cudaStream_t)stream));
}

lora_status lora_workspace_view(const lora_pool* pool, void* ws, size_t ws_bytes, int32_t max_tokens,
                                int32_t max_segments, lora_ws_view* view) {
    if (pool == nullptr || view == nullptr || max_tokens < 0 || max_segments < 0) return LORA_EINVAL;
    const WsLayout L = ws_layout(max_tokens, max_segments);
    lora_status st = check_ws(ws, ws_bytes, L.total);
    if (st != LORA_OK) return st;
    char* w = reinterpret_cast<char*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
    view->error_word = &hdr->err;
    view->counts = hdr->counts;
    view->perm = reinterpret_cast<int32_t*>(w + L.perm);
    view->grp_start = reinterpret_cast<int32_t*>(w + L.grp_start);
    view->grp_adapter = reinterpret_cast<int32_t*>(w + L.grp_adapter);
    return LORA_OK;
}

lora_status lora_segment(const lora_pool* pool, const int32_t* seg_start, const int32_t* seg_adapter,
                         int32_t S, const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                         size_t ws_bytes, void* stream) {
    if (pool == nullptr || S < 0 || Td < 0 || T < 0) return LORA_EINVAL;
    if ((int64_t)S + Td > LORA_MAX_SEGMENTS || T > (1 << 28)) return LORA_ETOOBIG;
    if (S > 0 && (seg_start == nullptr || seg_adapter == nullptr)) return LORA_EINVAL;
    if (Td > 0 && dec_adapter == nullptr) return LORA_EINVAL;
    if (S == 0 && Td > T) return LORA_EINVAL;
    const WsLayout L = ws_layout(T, S + Td);
    lora_status st = check_ws(ws, ws_bytes, L.total);
    if (st != LORA_OK) return st;
    SegParams sp;
    memset(&sp, 0, sizeof sp);
    sp.pool = view_of(pool);
    sp.seg_start = seg_start;
    sp.seg_adapter = seg_adapter;
    sp.dec_adapter = dec_adapter;
    sp.ws = reinterpret_cast<char*>(ws);
    sp.L = L;
    sp.S = S;
    sp.Td = Td;
    sp.T = T;
    sp.mma_min = 0;
    sp.L_tokens = T;
    sp.L_segments = S + Td;
    segment_kernel<<<1, kSegThreads, 0, (cudaStream_t)stream>>>(sp);
    return cuda_status(cudaGetLastError());
}

lora_status lora_delta_grouped(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                               void* ws, size_t ws_bytes, void* stream) {
    if (pool == nullptr || nprob < 0 || (nprob > 0 && probs == nullptr)) return LORA_EINVAL;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    if (nprob == 0) return LORA_OK;
    return run_delta(pool, probs, nprob, ws, nullptr, (cudaStream_t)stream);
}

lora_status lora_bgmv(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                      const int32_t* token_adapter, int32_t T, void* ws, size_t ws_bytes,
                      void* stream) {
    if (T > 0 && token_adapter == nullptr) return LORA_EINVAL;
    lora_status st = lora_segment(pool, nullptr, nullptr, 0, token_adapter, T, T, ws, ws_bytes, stream);
    if (st != LORA_OK) return st;
    return lora_delta_grouped(pool, probs, nprob, ws, ws_bytes, stream);
}

lora_status lora_sgmv(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                      const int32_t* seg_start, const int32_t* seg_adapter, int32_t S, int32_t T,
                      void* ws, size_t ws_bytes, void* stream) {
    lora_status st = lora_segment(pool, seg_start, seg_adapter, S, nullptr, 0, T, ws, ws_bytes, stream);
    if (st != LORA_OK) return st;
    return lora_delta_grouped(pool, probs, nprob, ws, ws_bytes, stream);
}

lora_status lora_apply_mixed(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                             const int32_t* seg_start, const int32_t* seg_adapter, int32_t S,
                             const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                             size_t ws_bytes, void* stream) {
    lora_status st = lora_segment(pool, seg_start, seg_adapter, S, dec_adapter, Td, T, ws, ws_bytes,
                                  stream);
    if (st != LORA_OK) return st;
    return lora_delta_grouped(pool, probs, nprob, ws, ws_bytes, stream);
}

lora_status lora_debug_page_list(const lora_pool* pool, void* ws, size_t ws_bytes, int32_t layer,
                                 int32_t proj, int32_t* out_pages, int64_t cap, int32_t* count_dev,
                                 void* stream) {
    if (pool == nullptr || out_pages == nullptr || count_dev == nullptr || cap < 0) return LORA_EINVAL;
    if (layer < 0 || layer >= pool->d.num_layers || proj < 0 || proj >= pool->d.num_proj)
        return LORA_EINVAL;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    page_list_kernel<<<1, kSegThreads, 0, (cudaStream_t)stream>>>(
        view_of(pool), reinterpret_cast<const char*>(ws), layer * pool->d.num_proj + proj, out_pages,
        cap, count_dev);
    return cuda_status(cudaGetLastError());
}

lora_status lora_debug_delta_with_t(const lora_pool* pool, const lora_problem* prob, void* ws,
                                    size_t ws_bytes, float* t_out, void* stream) {
    if (pool == nullptr || prob == nullptr || t_out == nullptr) return LORA_EINVAL;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    return run_delta(pool, prob, 1, ws, t_out, (cudaStream_t)stream);
}

lora_status lora_get_device_error(void* ws, void* stream, uint32_t* bits) {
    if (bits == nullptr) return LORA_EINVAL;
    *bits = 0;
    lora_status st = check_ws(ws, sizeof(WsHeader), sizeof(WsHeader));
    if (st != LORA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    uint32_t v = 0;
    st = cuda_status(cudaStreamSynchronize(s));
    if (st != LORA_OK) return st;
    st = cuda_status(cudaMemcpy(&v, &hdr->err, sizeof v, cudaMemcpyDeviceToHost));
    if (st != LORA_OK) return st;
    if (v != 0) {
        st = cuda_status(cudaMemsetAsync(&hdr->err, 0, sizeof v, s));
        if (st != LORA_OK) return st;
        st = cuda_status(cudaStreamSynchronize(s));
        if (st != LORA_OK) return st;
    }
    *bits = v;
    return v ? LORA_EDEVICE : LORA_OK;
}

}  // extern "C"
