// Device helpers shared by the multi-LoRA kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora.h"

namespace lora {

constexpr int kWarp = 32;
constexpr int kChunk = 4;        // rows per CUDA-core work item
constexpr int kTileRows = 128;   // rows per tensor-core tile
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait

// ---------------------------------------------------------------------------- workspace
// The workspace header lives at offset 0 of the caller's workspace.
struct WsHeader {
    uint32_t err;            // LORA_DERR_* bits, sticky until lora_get_device_error
    int32_t counts[4];       // adapted rows, groups, FMA chunks, MMA tiles
    uint32_t work_counter;   // dynamic work queue of the delta kernels
    uint32_t done_counter;   // CTAs finished (the last one resets both counters)
    uint32_t work_counter2;  // second queue (tensor-core items)
    int32_t cap_tokens;      // layout of the arrays below the header (set by grouping)
    int32_t cap_segments;
    // per work class (0: CUDA-core chunks, 1: tensor-core tiles): adapted rows, and page
    // rows (rank x items: an item reads its adapter's pages once); a projection of widths
    // (d_in, d_out) streams (d_in + 2 d_out) bf16 per row and (d_in + d_out) per page row
    unsigned long long rows[2];
    unsigned long long page_rows[2];
    uint32_t pad[46];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

// Work item of the CUDA-core path: up to 4 rows of one adapter, with everything the
// delta kernels need about it except the projection (48 bytes, read with 3 vector loads).
struct Chunk {
    int32_t adapter;
    int32_t count;     // rows, 1..4
    int32_t rank;
    float scale;
    int64_t pt_base;   // adapter's page-table offset
    int32_t begin;     // offset into the CUDA-core row list
    int32_t pad;
    int32_t rows[4];   // x / y rows (unused slots 0)
};
static_assert(sizeof(Chunk) == 48, "chunk is 48 bytes");

// Work item of the tensor-core path: up to 128 contiguous rows of one segment.
struct Tile {
    int32_t adapter;
    int32_t row0;
    int32_t rows;
    int32_t rank;
};

// Byte offsets of the workspace arrays for (max_tokens, max_segments).
struct WsLayout {
    size_t seg_key, seg_begin, seg_len, sorted, pos, fpos, gfirst, perm, grp_start, grp_adapter,
        fma_rows, chunks, tiles, total;
};

__host__ __device__ constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

__host__ __device__ constexpr WsLayout ws_layout(int32_t max_tokens, int32_t max_segments) {
    WsLayout L{};
    size_t o = sizeof(WsHeader);
    const size_t n = (size_t)max_segments + 1, t = (size_t)max_tokens + 1;
    L.seg_key = o;      o = align256(o + n * 8);
    L.seg_begin = o;    o = align256(o + n * 4);
    L.seg_len = o;      o = align256(o + n * 4);
    L.sorted = o;       o = align256(o + n * 4);
    L.pos = o;          o = align256(o + n * 4);
    L.fpos = o;         o = align256(o + n * 4);
    L.gfirst = o;       o = align256(o + n * 4);
    L.perm = o;         o = align256(o + t * 4);
    L.grp_start = o;    o = align256(o + (t + 1) * 4);
    L.grp_adapter = o;  o = align256(o + t * 4);
    L.fma_rows = o;     o = align256(o + t * 4);
    L.chunks = o;       o = align256(o + t * sizeof(Chunk));
    L.tiles = o;        o = align256(o + (t / 128 + n + 1) * sizeof(Tile));
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------- pool view
struct PoolView {
    const __nv_bfloat16* pages;
    int64_t num_pages;
    const int32_t* pt;
    int64_t pt_len;
    const int64_t* pt_off;
    const int32_t* ranks;
    const float* scales;
    int32_t h;
    int32_t num_adapters;
    int32_t num_layers;
    int32_t num_proj;
    int32_t r_max;
    int32_t units;   // U: page-table entries of one layer, in units of r_a (2 P for h x h)
};

// One projection instance inside a launch (32 bytes; many fit in kernel parameters).
struct ProbDesc {
    const __nv_bfloat16* x;
    __nv_bfloat16* y;
    int32_t ldx;
    int32_t ldy;
    int32_t blk;     // the A block's offset in units of r_a entries: l * U + pre(p)
    int32_t d_in;    // x columns read (h for h x h pools)
    int32_t d_out;   // y columns updated
    int32_t pad;
};

// rows[i] for a run-time i < kChunk, by selection: an array indexed by a run-time value
// would be placed in local memory, and with it every other field of its struct.
__device__ __forceinline__ int32_t row_of(const int32_t (&rows)[kChunk], int i) {
    static_assert(kChunk == 4, "selection over four rows");
    return i == 0 ? rows[0] : i == 1 ? rows[1] : i == 2 ? rows[2] : rows[3];
}

// Pages one vector of length d spans on pages of h values.
__host__ __device__ __forceinline__ int vec_pages(int d, int h) { return (d + h - 1) / h; }

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) { atomicOr(err, bits); }

// ---------------------------------------------------------------------------- bf16 helpers
// bf16 is the upper half of an IEEE binary32: widening is a shift.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// s + x.lo * a.lo + x.hi * a.hi for two packed bf16 pairs, accumulated in fp32 in that
// order with the mixed-precision FMA (bf16 inputs, fp32 addend and result): the products
// are exact and each FMA rounds once, as fmaf on the widened values does, but the bf16
// halves feed the FMA directly instead of being widened first.
// Two fp32 FMAs in one instruction (packed f32x2, sm_100 and later): c0 += a * b0 and
// c1 += a * b1, each rounded as fmaf would round it.  The expands multiply one fp32 t value
// by the columns of a B vector, so pairs of neighbouring columns share the multiplier.
__device__ __forceinline__ void fma2_f32(float& c0, float& c1, float a, float b0, float b1) {
    unsigned long long c, av, bv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(a), "f"(a));
    asm("mov.b64 %0, {%1, %2};" : "=l"(bv) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(c) : "f"(c0), "f"(c1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c) : "l"(av), "l"(bv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(c0), "=f"(c1) : "l"(c));
}

__device__ __forceinline__ float fma_bf16x2(uint32_t x, uint32_t a, float s) {
    asm("{\n\t.reg .b16 xl, xh, al, ah;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.bf16 %0, xl, al, %0;\n\t"
        "fma.rn.f32.bf16 %0, xh, ah, %0;\n\t}"
        : "+f"(s)
        : "r"(x), "r"(a));
    return s;
}

// s + the dot product of eight bf16 pairs (x, a), element by element in order.
__device__ __forceinline__ float dot8_bf16(const uint4& x, const uint4& a, float s) {
    s = fma_bf16x2(x.x, a.x, s);
    s = fma_bf16x2(x.y, a.y, s);
    s = fma_bf16x2(x.z, a.z, s);
    return fma_bf16x2(x.w, a.w, s);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

// Streaming 16-byte load of read-only data (adapter pages): no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void st16(void* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }

// ---------------------------------------------------------------------------- warp reductions
// Reduces V per-lane values across the warp with V-1 + log2(32/V) shuffles.  Lane l
// returns the full sum of value index l / (32 / V).
template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[V]) {
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int n = V, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float s = v[0];
#pragma unroll
    for (int o = 16 / V; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// ---------------------------------------------------------------------------- block scan
// Exclusive scan of one int per thread over the whole block (blockDim.x multiple of 32,
// <= 1024).  `smem` holds >= 33 ints.  Returns the exclusive prefix; *total = block sum.
__device__ inline int block_exclusive_scan(int v, int* smem, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) smem[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? smem[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < nw) smem[lane] = wi - w;
        if (lane == 31) smem[32] = wi;
    }
    __syncthreads();
    const int res = smem[warp] + incl - v;
    *total = smem[32];
    __syncthreads();
    return res;
}

}  // namespace lora
