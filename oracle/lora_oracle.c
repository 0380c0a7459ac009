/*
 * ORACLE — test infrastructure only.  Plain, slow, fp64 CPU restatement of the
 * multi-LoRA delta.  Only the tests, the package's smoke check and the bench's
 * CPU-baseline leg may load it; the GPU product path never calls it.
 *
 * What it computes (the plain definition; the GPU method reaches the same
 * result up to rounding order):
 *
 *   For problem (layer l, projection p) of widths d_in x d_out and each token i with
 *   adapter a = a(i):
 *     a == -1                 : y_ref[i,:] = y0[i,:] exactly (base-only token).
 *     otherwise, r = r_a, s = s_a,
 *       A row j   : d_in values, B col j : d_out values, each vector of length d taking
 *                   pv(d) = ceil(d / h) pages; element k of A row j is element k % h of
 *                   page pt[blkA + (k / h) * r + j] (B col j likewise from blkB), where
 *                   blkA = off[a] + r * (l * U + pre(p)), blkB = blkA + r * pv(d_in),
 *                   u(p) = pv(d_in) + pv(d_out), U = sum_p u(p), pre(p) = sum_{p'<p} u(p')
 *                   (with d_in = d_out = h: blkA = off[a] + ((l*P + p)*2 + 0)*r, blkB =
 *                   off[a] + ((l*P + p)*2 + 1)*r, one page per vector)
 *       t_j       = sum_{k < d_in} x[i,k] * A_j[k]          (shrink, k in order)
 *       delta_n   = s * sum_j t_j * Bcol_j[n], n < d_out     (expand, j in order)
 *       y_ref[i,n]= y0[i,n] + delta_n                        (kept in double)
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
 *   - "Multi-LoRA serving: S-LoRA, Punica and adapter batching", section "Worked
 *     example: a thousand adapters on one 8B base": projections of different in and
 *     out widths (grouped-query k/v, the MLP), every one of them adapted.
 *   Readings where the pages are silent: a vector longer than a page continues on
 *   further pages (the last one partly used), one page per h values; the page-table
 *   block layout above; s applied after the j-sum.
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
                      const int32_t* proj_dims,
                      int32_t layer, int32_t proj,
                      const uint16_t* x, int64_t ldx, const double* y0, int64_t ldy0,
                      const int32_t* token_adapter, int32_t T,
                      double* y_out, int64_t ldyo, double* t_out, int64_t* madds) {
    int err = 0;
    int64_t count = 0;
    if (layer < 0 || layer >= num_layers || proj < 0 || proj >= num_proj) return 3;
    /* widths of every projection (all h when proj_dims is NULL) and the block layout */
    int64_t U = 0, pre = 0;
    for (int32_t q = 0; q < num_proj; ++q) {
        const int32_t di = proj_dims ? proj_dims[2 * q] : h, dq = proj_dims ? proj_dims[2 * q + 1] : h;
        const int64_t u = (di + h - 1) / h + (dq + h - 1) / h;
        if (q < proj) pre += u;
        U += u;
    }
    const int32_t d_in = proj_dims ? proj_dims[2 * proj] : h;
    const int32_t d_out = proj_dims ? proj_dims[2 * proj + 1] : h;
    const int64_t pv_in = (d_in + h - 1) / h, pv_out = (d_out + h - 1) / h;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : count)
    for (int32_t i = 0; i < T; ++i) {
        const int32_t a = token_adapter[i];
        double* yo = y_out + (int64_t)i * ldyo;
        const double* yi = y0 + (int64_t)i * ldy0;
        if (t_out)
            for (int32_t j = 0; j < r_max; ++j) t_out[(int64_t)i * r_max + j] = 0.0;
        if (a == -1) {
            for (int32_t n = 0; n < d_out; ++n) yo[n] = yi[n];
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
                blk_a = pt_off[a] + (int64_t)r * ((int64_t)layer * U + pre);
                blk_b = blk_a + (int64_t)r * pv_in;
                if (pt_off[a] < 0 || blk_b + (int64_t)r * pv_out > pt_len) e = 3;
            }
        }
        if (!e) {
            for (int64_t k = 0; k < (pv_in + pv_out) * r && !e; ++k) {
                const int32_t pg = pt[blk_a + k];
                if (pg < 0 || pg >= num_pages) e = 4;
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
        /* shrink: t_j = sum_k x[i,k] * A_j[k], A_j[k] on page (k / h) of row j */
        for (int32_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int32_t k = 0; k < d_in; ++k) {
                const uint16_t* pg = pool + (int64_t)pt[blk_a + (int64_t)(k / h) * r + j] * h;
                acc += bf16_to_double(xi[k]) * bf16_to_double(pg[k % h]);
            }
            t[j] = acc;
            count += d_in;
        }
        /* expand: delta_n = s * sum_j t_j * Bcol_j[n]; y_ref = y0 + delta */
        for (int32_t n = 0; n < d_out; ++n) {
            double acc = 0.0;
            for (int32_t j = 0; j < r; ++j) {
                const uint16_t* pg = pool + (int64_t)pt[blk_b + (int64_t)(n / h) * r + j] * h;
                acc += t[j] * bf16_to_double(pg[n % h]);
            }
            yo[n] = yi[n] + s * acc;
        }
        count += (int64_t)d_out * r;
        if (t_out)
            for (int32_t j = 0; j < r; ++j) t_out[(int64_t)i * r_max + j] = t[j];
        free(t);
    }
    if (madds) *madds = count;
    return err;
}
