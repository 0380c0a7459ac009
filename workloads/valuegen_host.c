/* Host side of the seeded value generator (see valuegen.h for the definition).
 * Built with -ffp-contract=off so that x86-64 and aarch64 hosts give the same bits. */
#include <stdint.h>
#include <string.h>
#include "valuegen.h"

#define WL_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t wl_mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

/* IEEE binary32 -> bfloat16, round to nearest, ties to even (finite inputs only:
 * the generator never produces NaN or infinity). */
static inline uint16_t wl_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline double wl_value(uint64_t z, int dist, double param) {
    if (dist == WL_DIST_UNIFORM) {
        int64_t m = (int64_t)(2 * (z >> 40) + 1) - (int64_t)(1LL << 24);
        return (double)m * param;
    }
    int64_t s = (int64_t)(z & 0xFFFFu) + (int64_t)((z >> 16) & 0xFFFFu) +
                (int64_t)((z >> 32) & 0xFFFFu) + (int64_t)(z >> 48);
    return (double)(s - 131070) * param;
}

/* Fill rows of a bf16 matrix: row row_ids[r] of dst (row length h, stored as
 * raw uint16 bf16 bits) receives the h values of the stream keyed by keys[r]. */
void wl_fill_rows_host(uint16_t* dst, int64_t h, const int64_t* row_ids, const uint64_t* keys,
                       int64_t n, uint64_t seed, int dist, double param) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        uint64_t state0 = wl_mix64(seed ^ wl_mix64(keys[r]));
        uint16_t* out = dst + row_ids[r] * h;
        for (int64_t k = 0; k < h; ++k) {
            uint64_t z = wl_mix64(state0 + (uint64_t)(k + 1) * WL_GAMMA);
            out[k] = wl_f32_to_bf16((float)wl_value(z, dist, param));
        }
    }
}
