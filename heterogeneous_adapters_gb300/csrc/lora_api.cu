// C ABI of liblora.so (declarations and contracts in include/lora.h).
//
// Host side: argument checks, workspace layout, the grouping launch and the choice of
// delta launches (launch_ring.cu, launch_tile.cu, launch_cluster.cu).  All compute runs in
// the kernels of segment.cuh, bgmv_ring.cuh, bgmv_cluster.cuh, sgmv_mma.cuh, fused.cuh and
// stage.cuh; nothing here touches adapter or activation values.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>

#include "bgmv_cluster.cuh"
#include "host.h"
#include "segment.cuh"
#include "sgmv_mma.cuh"
#include "stage.cuh"

using namespace lora;
using namespace lora::host;

namespace lora {
namespace host {

thread_local int g_last_cuda_error = 0;

lora_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LORA_OK;
    g_last_cuda_error = (int)e;
    return LORA_ECUDA;
}

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
    v.units = pool->units;
    return v;
}

// Kernel descriptor of one problem: pointers, strides, widths and the offset of its A
// block (in units of r_a page-table entries).
ProbDesc prob_desc(const lora_pool* pool, const lora_problem& pr) {
    ProbDesc o;
    o.x = reinterpret_cast<const __nv_bfloat16*>(pr.x);
    o.y = reinterpret_cast<__nv_bfloat16*>(pr.y);
    o.ldx = (int32_t)pr.ldx;
    o.ldy = (int32_t)pr.ldy;
    o.blk = pr.layer * pool->units + pool->pre[pr.proj];
    o.d_in = pool->d_in[pr.proj];
    o.d_out = pool->d_out[pr.proj];
    o.pad = 0;
    return o;
}

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
        st = cuda_status(
            cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        if (st != LORA_OK) return st;
        di.ready = true;
    }
    *out = &di;
    return LORA_OK;
}

}  // namespace host
}  // namespace lora

namespace {

// The measured defaults of a pool's launch tuning: stage rows chosen by shared memory,
// the cluster kernel for one projection, tensor-core tiles by the rank rule, a 3-slot y ring.
void default_tuning(const lora_pool* pool, lora_tuning* t) {
    memset(t, 0, sizeof *t);
    t->ring_rows_per_stage = 0;
    t->split_max_problems = kClusterDefaultProbs;
    t->mma_min_rows = kMmaMinRowsByRank;
    t->mma_y_stages = 3;
    t->fused_ring_speed = default_fused_ring_speed(pool->square);
}

lora_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr || ((uintptr_t)ws & 255u) != 0) return LORA_EWORKSPACE;
    if (ws_bytes < need) return LORA_EWORKSPACE;
    return LORA_OK;
}

lora_status check_problems(const lora_pool* pool, const lora_problem* probs, int32_t nprob) {
    const lora_pool_desc& d = pool->d;
    for (int32_t i = 0; i < nprob; ++i) {
        const lora_problem& pr = probs[i];
        if (pr.x == nullptr || pr.y == nullptr) return LORA_EINVAL;
        if (!aligned16(pr.x) || !aligned16(pr.y)) return LORA_EALIGN;
        if (pr.ldx % 8 != 0 || pr.ldy % 8 != 0) return LORA_EALIGN;
        if (pr.layer < 0 || pr.layer >= d.num_layers || pr.proj < 0 || pr.proj >= d.num_proj)
            return LORA_EINVAL;
        if (pr.ldx < pool->d_in[pr.proj] || pr.ldy < pool->d_out[pr.proj] || pr.ldx > INT32_MAX ||
            pr.ldy > INT32_MAX)
            return LORA_EINVAL;
    }
    return LORA_OK;
}

// The delta launches after grouping: the CUDA-core kernel over the chunk list, then
// (when the batch may hold tensor-core tiles) the tensor-core kernel over the tile list.
lora_status run_delta(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                      size_t ws_bytes, float* t_out, bool with_mma, cudaStream_t stream) {
    lora_status st = check_problems(pool, probs, nprob);
    if (st != LORA_OK) return st;
    // launches of few projections: a chunk's work is spread over a cluster of CTAs
    if (!with_mma && t_out == nullptr && cluster_fits(pool, nprob))
        return run_cluster(pool, probs, nprob, ws, stream);
    // one launch per batch of projections for both work classes
    if (with_mma && mma_min_rows(pool) != 0 && t_out == nullptr && pool->d.h / 8 <= 640 && T > 0)
        return run_fused(pool, probs, nprob, T, ws, stream);
    st = run_delta_ring(pool, probs, nprob, ws, t_out, stream);
    if (st != LORA_OK) return st;
    if (with_mma && mma_min_rows(pool) != 0) st = run_mma(pool, probs, nprob, T, ws, stream);
    return st;
}

// ---------------------------------------------------------------------------- allocation-free BGMV
// Scratch of lora_bgmv_noalloc: a workspace for up to LORA_NOALLOC_MAX_TOKENS decode
// rows, living in a file-scope device array that every GPU loading this library holds
// until the process exits.  Host code must not pass `g_noalloc_ws` itself to a kernel
// (on the host it is only a stand-in symbol): its device address is looked up once per
// device with cudaGetSymbolAddress.
constexpr size_t kNoallocWsBytes = ws_layout(LORA_NOALLOC_MAX_TOKENS, LORA_NOALLOC_MAX_TOKENS).total;
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoallocWsBytes];

void* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// First call on a device (that device current): find the array's device address and
// zero its header.  Later calls reuse the cached address.
lora_status noalloc_workspace(void** out, cudaStream_t stream) {
    int dev = 0;
    lora_status st = cuda_status(cudaGetDevice(&dev));
    if (st != LORA_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return LORA_ETOOBIG;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* ptr = nullptr;
        st = cuda_status(cudaGetSymbolAddress(&ptr, g_noalloc_ws));
        if (st != LORA_OK) return st;
        st = cuda_status(cudaMemsetAsync(ptr, 0, sizeof(WsHeader), stream));
        if (st != LORA_OK) return st;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
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
        case LORA_ENOSPACE: return "no pool pages can be freed: every resident adapter is in use";
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
    lora_pool* p = new (std::nothrow) lora_pool;
    if (p == nullptr) return LORA_EINVAL;
    p->d = d;
    p->d.proj_dims = nullptr;
    p->d_in.resize((size_t)d.num_proj);
    p->d_out.resize((size_t)d.num_proj);
    p->pre.resize((size_t)d.num_proj);
    int64_t units = 0;
    for (int32_t q = 0; q < d.num_proj; ++q) {
        const int32_t di = d.proj_dims ? d.proj_dims[2 * q] : d.h;
        const int32_t dq = d.proj_dims ? d.proj_dims[2 * q + 1] : d.h;
        if (di <= 0 || dq <= 0 || di % 8 != 0 || dq % 8 != 0 ||
            di > LORA_MAX_VEC_PAGES * d.h || dq > LORA_MAX_VEC_PAGES * d.h) {
            delete p;
            return (di <= 0 || dq <= 0 || di % 8 || dq % 8) ? LORA_EINVAL : LORA_ETOOBIG;
        }
        p->d_in[q] = di;
        p->d_out[q] = dq;
        p->pre[q] = (int32_t)units;
        units += vec_pages(di, d.h) + vec_pages(dq, d.h);
        p->square = p->square && di == d.h && dq == d.h;
        p->mma_widths = p->mma_widths && di % kMmaKChunk == 0 && dq % kMmaNTile == 0;
    }
    if (units * d.num_layers > (1 << 26)) {
        delete p;
        return LORA_ETOOBIG;
    }
    p->units = (int32_t)units;
    default_tuning(p, &p->tune);
    *out = p;
    return LORA_OK;
}

lora_status lora_pool_destroy(lora_pool* pool) {
    delete pool;
    return LORA_OK;
}

lora_status lora_pool_set_tuning(lora_pool* pool, const lora_tuning* t) {
    if (pool == nullptr) return LORA_EINVAL;
    lora_tuning v;
    default_tuning(pool, &v);
    if (t != nullptr) {
        if (t->reserved[0] != 0 || t->reserved[1] != 0 || t->reserved[2] != 0) return LORA_EINVAL;
        if (t->ring_rows_per_stage != 0 && t->ring_rows_per_stage != 4 && t->ring_rows_per_stage != 8)
            return LORA_EINVAL;
        if (t->split_max_problems < -1 || t->split_max_problems > kClusterMaxProbs) return LORA_EINVAL;
        if (t->mma_min_rows < -1 || t->mma_min_rows == 1) return LORA_EINVAL;
        if (t->mma_y_stages != 0 && (t->mma_y_stages < 2 || t->mma_y_stages > 4)) return LORA_EINVAL;
        if (t->fused_ring_speed != 0.f && !(t->fused_ring_speed >= 0.1f && t->fused_ring_speed <= 10.f))
            return LORA_EINVAL;
        v.ring_rows_per_stage = t->ring_rows_per_stage;
        if (t->split_max_problems >= 0) v.split_max_problems = t->split_max_problems;
        if (t->mma_min_rows >= 0) v.mma_min_rows = t->mma_min_rows;
        if (t->mma_y_stages != 0) v.mma_y_stages = t->mma_y_stages;
        if (t->fused_ring_speed != 0.f) v.fused_ring_speed = t->fused_ring_speed;
    }
    pool->tune = v;
    return LORA_OK;
}

lora_status lora_pool_get_tuning(const lora_pool* pool, lora_tuning* out) {
    if (pool == nullptr || out == nullptr) return LORA_EINVAL;
    *out = pool->tune;
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

// The grouping launch.
// allow_tiles = false: every row goes to the CUDA-core chunks (the separate shrink and
// expand serve chunks only).
static lora_status segment_impl(const lora_pool* pool, const int32_t* seg_start, const int32_t* seg_adapter,
                         int32_t S, const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                         size_t ws_bytes, void* stream, bool allow_tiles = true) {
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
    sp.mma_min = allow_tiles ? mma_min_rows(pool) : 0;
    sp.mma_max_rank = kMmaMaxRank;
    sp.L_tokens = T;
    sp.L_segments = S + Td;
    size_t smem = 0;
    if (S + Td <= kSegSmemMax) {
        static thread_local int attr_dev = -1;
        int dev = 0;
        st = cuda_status(cudaGetDevice(&dev));
        if (st != LORA_OK) return st;
        if (attr_dev != dev) {
            st = cuda_status(cudaFuncSetAttribute(segment_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)seg_smem_bytes(kSegSmemMax)));
            if (st != LORA_OK) return st;
            attr_dev = dev;
        }
        sp.smem_segs = S + Td;
        smem = seg_smem_bytes(S + Td);
    }
    segment_kernel<<<1, kSegThreads, smem, (cudaStream_t)stream>>>(sp);
    return cuda_status(cudaGetLastError());
}

lora_status lora_segment(const lora_pool* pool, const int32_t* seg_start, const int32_t* seg_adapter,
                         int32_t S, const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                         size_t ws_bytes, void* stream) {
    return segment_impl(pool, seg_start, seg_adapter, S, dec_adapter, Td, T, ws, ws_bytes, stream);
}

lora_status lora_delta_grouped(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T,
                               int32_t S, void* ws, size_t ws_bytes, void* stream) {
    if (pool == nullptr || nprob < 0 || T < 0 || S < 0 || (nprob > 0 && probs == nullptr))
        return LORA_EINVAL;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    if (nprob == 0) return LORA_OK;
    // without prefill segments every segment has one row: no tensor-core tile exists
    return run_delta(pool, probs, nprob, T, ws, ws_bytes, nullptr, S > 0, (cudaStream_t)stream);
}

lora_status lora_bgmv(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                      const int32_t* token_adapter, int32_t T, void* ws, size_t ws_bytes,
                      void* stream) {
    if (T > 0 && token_adapter == nullptr) return LORA_EINVAL;
    lora_status st = lora_segment(pool, nullptr, nullptr, 0, token_adapter, T, T, ws, ws_bytes, stream);
    if (st != LORA_OK) return st;
    if (nprob < 0 || (nprob > 0 && probs == nullptr)) return LORA_EINVAL;
    if (nprob == 0) return LORA_OK;
    // decode rows are one-row segments: the CUDA-core kernel serves all of them
    return run_delta(pool, probs, nprob, T, ws, ws_bytes, nullptr, false, (cudaStream_t)stream);
}

lora_status lora_sgmv(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                      const int32_t* seg_start, const int32_t* seg_adapter, int32_t S, int32_t T,
                      void* ws, size_t ws_bytes, void* stream) {
    lora_status st = lora_segment(pool, seg_start, seg_adapter, S, nullptr, 0, T, ws, ws_bytes, stream);
    if (st != LORA_OK) return st;
    return lora_delta_grouped(pool, probs, nprob, T, S, ws, ws_bytes, stream);
}

lora_status lora_apply_mixed(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                             const int32_t* seg_start, const int32_t* seg_adapter, int32_t S,
                             const int32_t* dec_adapter, int32_t Td, int32_t T, void* ws,
                             size_t ws_bytes, void* stream) {
    lora_status st = lora_segment(pool, seg_start, seg_adapter, S, dec_adapter, Td, T, ws, ws_bytes,
                                  stream);
    if (st != LORA_OK) return st;
    return lora_delta_grouped(pool, probs, nprob, T, S, ws, ws_bytes, stream);
}

lora_status lora_shrink(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                        const int32_t* token_adapter, int32_t T, void* ws, size_t ws_bytes, float* t,
                        void* stream) {
    if (pool == nullptr || nprob < 0 || T < 0 || (nprob > 0 && probs == nullptr)) return LORA_EINVAL;
    if (T > 0 && (token_adapter == nullptr || t == nullptr)) return LORA_EINVAL;
    if (((uintptr_t)t & 15u) != 0) return LORA_EALIGN;
    lora_status st = check_problems(pool, probs, nprob);
    if (st != LORA_OK) return st;
    st = segment_impl(pool, nullptr, nullptr, 0, token_adapter, T, T, ws, ws_bytes, stream, false);
    if (st != LORA_OK || nprob == 0 || T == 0) return st;
    return run_shrink_expand(pool, probs, nprob, T, ws, t, false, (cudaStream_t)stream);
}

lora_status lora_expand(const lora_pool* pool, const lora_problem* probs, int32_t nprob, int32_t T, void* ws,
                        size_t ws_bytes, const float* t, void* stream) {
    if (pool == nullptr || nprob < 0 || T < 0 || (nprob > 0 && probs == nullptr)) return LORA_EINVAL;
    if (T > 0 && t == nullptr) return LORA_EINVAL;
    if (((uintptr_t)t & 15u) != 0) return LORA_EALIGN;
    lora_status st = check_ws(ws, ws_bytes, ws_layout(T, T).total);
    if (st != LORA_OK) return st;
    st = check_problems(pool, probs, nprob);
    if (st != LORA_OK || nprob == 0 || T == 0) return st;
    return run_shrink_expand(pool, probs, nprob, T, ws, const_cast<float*>(t), true, (cudaStream_t)stream);
}

lora_status lora_debug_page_list(const lora_pool* pool, void* ws, size_t ws_bytes, int32_t layer,
                                 int32_t proj, int32_t* out_pages, int64_t cap, int32_t* count_dev,
                                 void* stream) {
    if (pool == nullptr || out_pages == nullptr || count_dev == nullptr || cap < 0) return LORA_EINVAL;
    if (layer < 0 || layer >= pool->d.num_layers || proj < 0 || proj >= pool->d.num_proj)
        return LORA_EINVAL;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    const int32_t vec_units = vec_pages(pool->d_in[proj], pool->d.h) + vec_pages(pool->d_out[proj], pool->d.h);
    page_list_kernel<<<1, kSegThreads, 0, (cudaStream_t)stream>>>(
        view_of(pool), reinterpret_cast<const char*>(ws), layer * pool->units + pool->pre[proj], vec_units,
        out_pages, cap, count_dev);
    return cuda_status(cudaGetLastError());
}

lora_status lora_debug_delta_with_t(const lora_pool* pool, const lora_problem* prob, void* ws,
                                    size_t ws_bytes, float* t_out, void* stream) {
    if (pool == nullptr || prob == nullptr || t_out == nullptr) return LORA_EINVAL;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    return run_delta(pool, prob, 1, 0, ws, ws_bytes, t_out, false, (cudaStream_t)stream);
}

namespace {
// One thread waits, bounded, on a barrier nothing arrives at (the wait kernels use).
__global__ void wait_limit_kernel(char* ws, uint64_t limit_ns, uint64_t* elapsed) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const uint64_t t0 = global_timer_ns();
    const bool done = mbar_wait(b, 0, limit_ns);
    const uint64_t t1 = global_timer_ns();
    if (!done) set_error(&reinterpret_cast<WsHeader*>(ws)->err, LORA_DERR_TIMEOUT);
    if (elapsed != nullptr) *elapsed = t1 - t0;
}
}  // namespace

lora_status lora_debug_wait_limit(void* ws, size_t ws_bytes, uint64_t limit_ns, uint64_t* elapsed_ns_dev,
                                  void* stream) {
    if (limit_ns < 1000000ull) return LORA_EINVAL;
    if (limit_ns > 2000000000ull) return LORA_ETOOBIG;
    lora_status st = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (st != LORA_OK) return st;
    wait_limit_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(reinterpret_cast<char*>(ws), limit_ns, elapsed_ns_dev);
    return cuda_status(cudaGetLastError());
}

// Host-side checks of a staging call (the index arrays are host memory).
static lora_status check_stage(const lora_pool* pool, const void* rows, const int32_t* dst_pages, int32_t npages,
                               int32_t* page_table, const int64_t* upd_index, const int32_t* upd_page, int64_t nupd) {
    if (pool == nullptr || npages < 0 || nupd < 0) return LORA_EINVAL;
    const lora_pool_desc& d = pool->d;
    if (npages > 0 && (rows == nullptr || dst_pages == nullptr)) return LORA_EINVAL;
    if (nupd > 0 && (page_table == nullptr || upd_index == nullptr || upd_page == nullptr)) return LORA_EINVAL;
    if (nupd > 0 && page_table != d.page_table) return LORA_EINVAL;
    if (npages > 0 && !aligned16(rows)) return LORA_EALIGN;
    for (int32_t i = 0; i < npages; ++i)
        if (dst_pages[i] < 0 || dst_pages[i] >= d.num_pages) return LORA_EINVAL;
    for (int64_t k = 0; k < nupd; ++k) {
        if (upd_index[k] < 0 || upd_index[k] >= d.page_table_len) return LORA_EINVAL;
        if (upd_page[k] < 0 || upd_page[k] >= d.num_pages) return LORA_EINVAL;
    }
    return LORA_OK;
}

// The staging kernel: rows (host memory read through its mapping, or device memory) into
// pool pages, then the page-table rewrite.
static lora_status launch_stage(const lora_pool* pool, const void* rows, const int32_t* dst_pages, int32_t npages,
                                int32_t* page_table, const int64_t* upd_index, const int32_t* upd_page, int64_t nupd,
                                cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    lora_status st = device_info(&di);
    if (st != LORA_OK) return st;
    StageParams sp;
    sp.host_rows = reinterpret_cast<const uint4*>(rows);
    sp.dst_pages = dst_pages;
    sp.pages = reinterpret_cast<__nv_bfloat16*>(pool->d.pages);
    sp.pt = page_table;
    sp.upd_index = upd_index;
    sp.upd_page = upd_page;
    sp.nupd = nupd;
    sp.npages = npages;
    sp.vec_per_row = pool->d.h / 8;
    int grid = di->sm_count * 4;
    if (npages > 0 && npages < grid) grid = npages;
    if (npages == 0) grid = (int)std::min<int64_t>(grid, (nupd + kStageThreads - 1) / kStageThreads);
    if (grid < 1) grid = 1;
    stage_kernel<<<grid, kStageThreads, 0, stream>>>(sp);
    return cuda_status(cudaGetLastError());
}

lora_status lora_stage_pages_ce(const lora_pool* pool, const void* host_rows, void* staging, size_t staging_bytes,
                                const int32_t* dst_pages, int32_t npages, int32_t* page_table,
                                const int64_t* upd_index, const int32_t* upd_page, int64_t nupd, void* copied,
                                void* stream) {
    lora_status st = check_stage(pool, host_rows, dst_pages, npages, page_table, upd_index, upd_page, nupd);
    if (st != LORA_OK) return st;
    const size_t row_bytes = (size_t)pool->d.h * 2;
    const size_t bytes = (size_t)npages * row_bytes;
    if (staging != nullptr && (!aligned16(staging) || staging_bytes < bytes)) return LORA_EINVAL;
    // runs of consecutive destination pages (a cache that hands out a unit's pages from a
    // free list gives one run per unit): each run is one copy straight into the pool
    int32_t runs = 0;
    for (int32_t i = 0; i < npages; ++i)
        if (i == 0 || dst_pages[i] != dst_pages[i - 1] + 1) ++runs;
    const bool direct = runs <= LORA_STAGE_MAX_RUNS;
    if (npages > 0 && !direct && staging == nullptr) return LORA_EINVAL;
    if (npages == 0 && nupd == 0) return LORA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const char* src = static_cast<const char*>(host_rows);
    if (direct) {
        char* pages = static_cast<char*>(pool->d.pages);
        for (int32_t i0 = 0; i0 < npages;) {
            int32_t i1 = i0 + 1;
            while (i1 < npages && dst_pages[i1] == dst_pages[i1 - 1] + 1) ++i1;
            st = cuda_status(cudaMemcpyAsync(pages + (size_t)dst_pages[i0] * row_bytes, src + (size_t)i0 * row_bytes,
                                             (size_t)(i1 - i0) * row_bytes, cudaMemcpyHostToDevice, s));
            if (st != LORA_OK) return st;
            i0 = i1;
        }
    } else {
        st = cuda_status(cudaMemcpyAsync(staging, host_rows, bytes, cudaMemcpyHostToDevice, s));
        if (st != LORA_OK) return st;
    }
    if (copied != nullptr) {
        st = cuda_status(cudaEventRecord((cudaEvent_t)copied, s));
        if (st != LORA_OK) return st;
    }
    if (direct) {   // the pages are in place: only the page-table rewrite is left
        if (nupd == 0) return LORA_OK;
        return launch_stage(pool, nullptr, nullptr, 0, page_table, upd_index, upd_page, nupd, s);
    }
    return launch_stage(pool, staging, dst_pages, npages, page_table, upd_index, upd_page, nupd, s);
}

lora_status lora_stage_pages(const lora_pool* pool, const void* host_rows, const int32_t* dst_pages,
                             int32_t npages, int32_t* page_table, const int64_t* upd_index,
                             const int32_t* upd_page, int64_t nupd, void* stream) {
    lora_status st = check_stage(pool, host_rows, dst_pages, npages, page_table, upd_index, upd_page, nupd);
    if (st != LORA_OK) return st;
    if (npages == 0 && nupd == 0) return LORA_OK;
    return launch_stage(pool, host_rows, dst_pages, npages, page_table, upd_index, upd_page, nupd,
                        (cudaStream_t)stream);
}

lora_status lora_bgmv_noalloc(const lora_pool* pool, const lora_problem* probs, int32_t nprob,
                              const int32_t* token_adapter, int32_t T, uint32_t* error_bits,
                              void* stream) {
    if (pool == nullptr || T < 0 || nprob < 0) return LORA_EINVAL;
    if (T > LORA_NOALLOC_MAX_TOKENS) return LORA_ETOOBIG;
    if ((T > 0 && token_adapter == nullptr) || (nprob > 0 && probs == nullptr)) return LORA_EINVAL;
    lora_status st = check_problems(pool, probs, nprob);
    if (st != LORA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    void* ws = nullptr;
    st = noalloc_workspace(&ws, s);
    if (st != LORA_OK) return st;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    // the error word is per call; the grouping kernel re-initialises everything else
    st = cuda_status(cudaMemsetAsync(&hdr->err, 0, sizeof(uint32_t), s));
    if (st != LORA_OK) return st;
    st = segment_impl(pool, nullptr, nullptr, 0, token_adapter, T, T, ws, kNoallocWsBytes, stream);
    if (st != LORA_OK) return st;
    if (nprob > 0) {
        st = run_delta(pool, probs, nprob, T, ws, kNoallocWsBytes, nullptr, false, s);
        if (st != LORA_OK) return st;
    }
    if (error_bits != nullptr)
        st = cuda_status(cudaMemcpyAsync(error_bits, &hdr->err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s));
    return st;
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
