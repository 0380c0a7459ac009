/* Seeded synthetic values for the multi-LoRA workloads (inputs only).
 *
 * Shared by both sides of the parity check: the CPU oracle's harness fills the
 * rows it needs with the host routine, the GPU harness fills device buffers with
 * the device routine, and both produce the same bf16 bits for the same
 * (seed, row key, element index).  Nothing here computes any part of the LoRA
 * delta.
 *
 * Counter-based generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014): the output finaliser
 *     z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 * applied to state0 + (k+1)*0x9E3779B97F4A7C15 gives the k-th output of the
 * stream whose state starts at state0.  Each row gets its own stream:
 *     state0 = mix64(seed ^ mix64(row_key)),  z_k = mix64(state0 + (k+1)*GAMMA).
 *
 * Value mapping (exact integer work, then ONE rounded double multiply, then
 * double -> float -> bf16, each round-to-nearest-even):
 *   WL_DIST_UNIFORM: m = 2*(z>>40) + 1 - 2^24 (odd integer, |m| < 2^24),
 *                    v = m * param, param = bound * 2^-24   ->  U(-bound, bound)
 *   WL_DIST_NORMAL : s = sum of the four 16-bit fields of z (Irwin-Hall, n=4),
 *                    v = (s - 131070) * param, param = sigma / sqrt(4*(2^32-1)/12)
 *                    -> mean 0, standard deviation sigma, support +-3.46 sigma.
 */
#ifndef WORKLOADS_VALUEGEN_H
#define WORKLOADS_VALUEGEN_H
#include <stdint.h>

#define WL_DIST_UNIFORM 0
#define WL_DIST_NORMAL 1

#endif
