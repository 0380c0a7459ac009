// Device side of the seeded value generator (see valuegen.h for the definition).
// It produces the same bf16 bits as valuegen_host.c: the only floating-point
// steps are one round-to-nearest double multiply (__dmul_rn, never contracted)
// and the double->float->bf16 conversions, done with CUDA's own RN intrinsics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include "valuegen.h"

#define WL_GAMMA 0x9E3779B97F4A7C15ULL

__device__ __forceinline__ uint64_t wl_mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

__global__ void wl_fill_rows_kernel(__nv_bfloat16* __restrict__ dst, int64_t h,
                                    const int64_t* __restrict__ row_ids,
                                    const uint64_t* __restrict__ keys, int64_t n, uint64_t seed,
                                    int dist, double param) {
    for (int64_t r = blockIdx.x; r < n; r += gridDim.x) {
        const uint64_t state0 = wl_mix64(seed ^ wl_mix64(keys[r]));
        __nv_bfloat16* out = dst + row_ids[r] * h;
        for (int64_t k = threadIdx.x; k < h; k += blockDim.x) {
            const uint64_t z = wl_mix64(state0 + (uint64_t)(k + 1) * WL_GAMMA);
            double v;
            if (dist == WL_DIST_UNIFORM) {
                const int64_t m = (int64_t)(2 * (z >> 40) + 1) - (int64_t)(1LL << 24);
                v = __dmul_rn((double)m, param);
            } else {
                const int64_t s = (int64_t)(z & 0xFFFFu) + (int64_t)((z >> 16) & 0xFFFFu) +
                                  (int64_t)((z >> 32) & 0xFFFFu) + (int64_t)(z >> 48);
                v = __dmul_rn((double)(s - 131070), param);
            }
            out[k] = __float2bfloat16_rn(__double2float_rn(v));
        }
    }
}

// Fill `n` rows of the device bf16 matrix `dst` (row length h). row_ids and
// keys are device arrays. Asynchronous on `stream`; returns a cudaError_t.
extern "C" int wl_fill_rows_dev(void* dst, int64_t h, const int64_t* row_ids, const uint64_t* keys,
                                int64_t n, uint64_t seed, int dist, double param, void* stream) {
    if (n <= 0) return 0;
    int blocks = (int)(n < 65536 ? n : 65536);
    wl_fill_rows_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(
        (__nv_bfloat16*)dst, h, row_ids, keys, n, seed, dist, param);
    return (int)cudaGetLastError();
}
