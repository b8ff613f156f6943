/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for paged MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant table with the
 * CUDA path.
 *
 * What it computes (FlashMLA-PyTorch page, flash_mla_interface.py, docstring
 * of flash_mla_with_kvcache; vLLM page "vllm.attention.ops.flashmla",
 * flash_mla_with_kvcache parameter table):
 *
 *   q        (B, s_q, h_q, D)            D = head_dim = 576
 *   k_cache  (num_blocks, P, h_k, D)     P = page_block_size
 *   V        = the first Dv = head_dim_v dims of the same cache rows (the
 *              interface passes no separate V cache, "None" in the
 *              fwd_kvcache_mla call)
 *   block_table (B, max_blocks) int32: logical block j of sequence b lives in
 *              physical block block_table[b][j]
 *   cache_seqlens (B) int32
 *   out      (B, s_q, h_q, Dv)
 *   softmax_lse (B, h_q, s_q): natural-log sum of exp of the scaled logits.
 *
 * For every (b, i, h):
 *   hk   = h / (h_q / h_k)                      (query heads grouped per KV head)
 *   n    = causal ? L_b - s_q + 1 + i : L_b,    clamped to [0, L_b]
 *          (bottom-right causal alignment: the last query of the step sees
 *           the whole cache; the pages only say "whether to apply a causal
 *           mask", this is the reading adopted)
 *   s_t  = scale * sum_d q[b,i,h,d] * k[t,d]    for t < n
 *   lse  = log(sum_t exp(s_t))                  (computed max-shifted)
 *   out  = sum_t exp(s_t - lse) * k[t, 0:Dv]
 * With n == 0 the row has no visible key: out = 0, lse = -inf.
 *
 * Everything is evaluated in double precision from the exact bf16 inputs.
 * The loops follow the definition directly: no blocking, no online softmax.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of threads the parallel loop will use (1 in a build without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Returns 0 on success, -1 on a bad shape, -2 when a block_table entry that
 * a sequence needs lies outside [0, num_blocks).
 *
 * Strides are in elements.  q_stride = {b, i, h} (last dim contiguous);
 * k_stride = {block, row-in-page, kv-head} (last dim contiguous).
 * Only the rows listed in row_sel (flattened b*s_q*h_q + i*h_q + h) are
 * computed when n_sel >= 0; n_sel < 0 means all rows.
 */
int oracle_mla_decode(int B, int s_q, int h_q, int h_k, int D, int Dv, int P,
                      int num_blocks, int max_blocks,
                      const uint16_t *q, const int64_t *q_stride,
                      const uint16_t *k_cache, const int64_t *k_stride,
                      const int32_t *block_table, int64_t bt_stride,
                      const int32_t *cache_seqlens, double scale, int causal,
                      const int64_t *row_sel, int64_t n_sel,
                      double *out, double *lse, int nthreads) {
    if (B < 0 || s_q < 1 || h_q < 1 || h_k < 1 || h_q % h_k != 0 || Dv > D || P < 1)
        return -1;
    const int hpk = h_q / h_k;
    const int64_t total = (int64_t)B * s_q * h_q;
    const int64_t nrows = n_sel >= 0 ? n_sel : total;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t rr = 0; rr < nrows; ++rr) {
        const int64_t row = n_sel >= 0 ? row_sel[rr] : rr;
        const int b = (int)(row / ((int64_t)s_q * h_q));
        const int i = (int)((row / h_q) % s_q);
        const int h = (int)(row % h_q);
        const int hk = h / hpk;
        const int L = cache_seqlens[b] > 0 ? cache_seqlens[b] : 0;
        int n = causal ? L - s_q + 1 + i : L;
        if (n < 0) n = 0;
        if (n > L) n = L;

        double *o = out + row * (int64_t)Dv;
        double *lse_out = lse + ((int64_t)b * h_q + h) * s_q + i;
        for (int d = 0; d < Dv; ++d) o[d] = 0.0;
        if (n == 0) {
            *lse_out = -INFINITY;
            continue;
        }
        const uint16_t *qr = q + b * q_stride[0] + i * q_stride[1] + h * q_stride[2];

        /* logits s_t = scale * q . k_t over all D dims (latent + RoPE) */
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        if (!s) { bad = 1; continue; }
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
            if (t / P >= max_blocks) { bad = 1; s[t] = -INFINITY; continue; }
            const int32_t phys = block_table[b * bt_stride + t / P];
            if (phys < 0 || phys >= num_blocks) { bad = 1; s[t] = -INFINITY; continue; }
            const uint16_t *kr = k_cache + phys * k_stride[0] + (t % P) * k_stride[1] + hk * k_stride[2];
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_bits_to_double(qr[d]) * bf16_bits_to_double(kr[d]);
            s[t] = scale * dot;
            if (s[t] > m) m = s[t];
        }
        /* softmax denominator (max-shifted) and the weighted sum of V rows */
        double denom = 0.0;
        for (int t = 0; t < n; ++t) denom += exp(s[t] - m);
        const double lse_row = m + log(denom);
        for (int t = 0; t < n; ++t) {
            if (t / P >= max_blocks) continue;
            const int32_t phys = block_table[b * bt_stride + t / P];
            if (phys < 0 || phys >= num_blocks) continue;
            const uint16_t *kr = k_cache + phys * k_stride[0] + (t % P) * k_stride[1] + hk * k_stride[2];
            const double w = exp(s[t] - lse_row);
            for (int d = 0; d < Dv; ++d) o[d] += w * bf16_bits_to_double(kr[d]);
        }
        *lse_out = lse_row;
        free(s);
    }
    return bad ? -2 : 0;
}

/* The logits of one row, for the tests: s[t] = scale * q . k_t, t < n. */
int oracle_mla_logits(int s_q, int h_q, int h_k, int D, int P, int num_blocks,
                      const uint16_t *q, const int64_t *q_stride,
                      const uint16_t *k_cache, const int64_t *k_stride,
                      const int32_t *block_table, int64_t bt_stride,
                      int b, int i, int h, int n, double scale, double *s) {
    const int hk = h / (h_q / h_k);
    (void)s_q;
    const uint16_t *qr = q + b * q_stride[0] + i * q_stride[1] + h * q_stride[2];
    for (int t = 0; t < n; ++t) {
        const int32_t phys = block_table[b * bt_stride + t / P];
        if (phys < 0 || phys >= num_blocks) return -2;
        const uint16_t *kr = k_cache + phys * k_stride[0] + (t % P) * k_stride[1] + hk * k_stride[2];
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_bits_to_double(qr[d]) * bf16_bits_to_double(kr[d]);
        s[t] = scale * dot;
    }
    return 0;
}
