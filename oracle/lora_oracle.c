/*
 * ORACLE — test infrastructure only.  Plain, slow, fp64 CPU restatement of the
 * multi-LoRA delta.  Only the tests, the package's smoke check and the bench's
 * CPU-baseline leg may load it; the GPU product path never calls it.
 *
 * What it computes (the plain definition; the GPU method reaches the same
 * result up to rounding order):
 *
 *   For problem (layer l, projection p) and each token i with adapter a = a(i):
 *     a == -1                 : y_ref[i,:] = y0[i,:] exactly (base-only token).
 *     otherwise, r = r_a, s = s_a,
 *       A row j   = page pt[off[a] + ((l*P + p)*2 + 0)*r + j],   j < r
 *       B col j   = page pt[off[a] + ((l*P + p)*2 + 1)*r + j],   j < r
 *       t_j       = sum_k x[i,k] * A_j[k]                  (shrink, k in order)
 *       delta_n   = s * sum_j t_j * Bcol_j[n]              (expand, j in order)
 *       y_ref[i,n]= y0[i,n] + delta_n                      (kept in double)
 *
 * Sources, by page and section:
 *   - "Multi-LoRA serving: S-LoRA, Punica and adapter batching", section "How the
 *     kernels work": shrink v_i = A_{a(i)} x_i in R^r, expand y_i += gamma B_{a(i)} v_i,
 *     one adapter index per token; section "Implementation sketch": the gathered
 *     bmm form (shrink over A_pool[idx], expand over B_pool[idx], times scale).
 *   - "S-LoRA: Serving Thousands of Concurrent Adapters in 2026", section
 *     "Implementation": per-token loop, scale = alpha / rank, A is rank x in_dim,
 *     B is out_dim x rank, delta = (x A^T) B^T * scale, un-adapted tokens untouched.
 *   - "S-LoRA: Serving Thousands of Concurrent LoRA Adapters" (unified paging): one
 *     pool of pages, each one hidden-size vector; adapters gathered from
 *     non-contiguous pages with mixed ranks and no padding.
 *   Readings where the pages are silent: each A row and each B column takes one
 *   page; the page-table block layout above; s applied after the j-sum.
 *
 * Values are raw bf16 bit patterns widened exactly to double.  Every
 * multiply-add of the shrink and expand is counted in *madds (two flops each).
 *
 * Return value: 0 on success, otherwise the first data error found
 * (1 adapter id out of range, 2 rank out of range, 3 page-table block out of
 * range, 4 page id out of range); outputs are then unspecified.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_lora_delta(const uint16_t* pool, int64_t num_pages, int32_t h,
                      const int32_t* pt, int64_t pt_len, const int64_t* pt_off,
                      const int32_t* ranks, const float* scales, int32_t num_adapters,
                      int32_t num_layers, int32_t num_proj, int32_t r_max,
                      int32_t layer, int32_t proj,
                      const uint16_t* x, int64_t ldx, const double* y0, int64_t ldy0,
                      const int32_t* token_adapter, int32_t T,
                      double* y_out, int64_t ldyo, double* t_out, int64_t* madds) {
    int err = 0;
    int64_t count = 0;
    if (layer < 0 || layer >= num_layers || proj < 0 || proj >= num_proj) return 3;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : count)
    for (int32_t i = 0; i < T; ++i) {
        const int32_t a = token_adapter[i];
        double* yo = y_out + (int64_t)i * ldyo;
        const double* yi = y0 + (int64_t)i * ldy0;
        if (t_out)
            for (int32_t j = 0; j < r_max; ++j) t_out[(int64_t)i * r_max + j] = 0.0;
        if (a == -1) {
            for (int32_t n = 0; n < h; ++n) yo[n] = yi[n];
            continue;
        }
        int e = 0;
        int32_t r = 0;
        int64_t blk_a = 0, blk_b = 0;
        if (a < -1 || a >= num_adapters) {
            e = 1;
        } else {
            r = ranks[a];
            if (r < 1 || r > r_max) {
                e = 2;
            } else {
                blk_a = pt_off[a] + ((int64_t)(layer * num_proj + proj) * 2 + 0) * r;
                blk_b = pt_off[a] + ((int64_t)(layer * num_proj + proj) * 2 + 1) * r;
                if (pt_off[a] < 0 || blk_b + r > pt_len) e = 3;
            }
        }
        if (!e) {
            for (int32_t j = 0; j < r && !e; ++j) {
                int32_t pa = pt[blk_a + j], pb = pt[blk_b + j];
                if (pa < 0 || pa >= num_pages || pb < 0 || pb >= num_pages) e = 4;
            }
        }
        if (e) {
#pragma omp critical
            if (!err) err = e;
            continue;
        }
        const double s = (double)scales[a];
        const uint16_t* xi = x + (int64_t)i * ldx;
        double* t = (double*)malloc(sizeof(double) * (size_t)r);
        /* shrink: t_j = sum_k x[i,k] * A_j[k] */
        for (int32_t j = 0; j < r; ++j) {
            const uint16_t* arow = pool + (int64_t)pt[blk_a + j] * h;
            double acc = 0.0;
            for (int32_t k = 0; k < h; ++k) acc += bf16_to_double(xi[k]) * bf16_to_double(arow[k]);
            t[j] = acc;
            count += h;
        }
        /* expand: delta_n = s * sum_j t_j * Bcol_j[n]; y_ref = y0 + delta */
        for (int32_t n = 0; n < h; ++n) {
            double acc = 0.0;
            for (int32_t j = 0; j < r; ++j)
                acc += t[j] * bf16_to_double(pool[(int64_t)pt[blk_b + j] * h + n]);
            yo[n] = yi[n] + s * acc;
        }
        count += (int64_t)h * r;
        if (t_out)
            for (int32_t j = 0; j < r; ++j) t_out[(int64_t)i * r_max + j] = t[j];
        free(t);
    }
    if (madds) *madds = count;
    return err;
}
