/*
 * capi_decode.c -- the decode driven from C through include/libmla.h alone
 * (no Python): schedule, decode with the library's own workspace, device
 * error check, shutdown; the result is held to the fp64 oracle (linked in
 * from oracle/mla_oracle.c, test infrastructure) within the parity bar
 * |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 2e-3.
 *
 * Problem: batch 3, s_q 2 (causal), 16 query heads, 1 KV head, cache lengths
 * {100, 1, 300} in a pool of 9 shuffled 64-row blocks.  The same values
 * rounded to e4m3 then go through mla_decode_fwd_fp8 (bmm1_scale, bmm2_scale),
 * held to the oracle on the decoded values with a coarse bar
 * |out - ref| <= 0.03 + 0.03 |ref| (the probabilities are rounded to e4m3;
 * the Python tests hold the derived bar), |lse - ref| <= 2e-3.  Exit status 0
 * on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "libmla.h"

int oracle_mla_decode(int B, int s_q, int h_q, int h_k, int D, int Dv, int P, int num_blocks, int max_blocks,
                      const uint16_t *q, const int64_t *q_stride, const uint16_t *k_cache, const int64_t *k_stride,
                      const int32_t *block_table, int64_t bt_stride, const int32_t *cache_seqlens, double scale,
                      int causal, const int64_t *row_sel, int64_t n_sel, double *out, double *lse, int nthreads);

enum { B = 3, SQ = 2, HQ = 16, HK = 1, D = 576, DV = 512, P = 64, NB = 9, MAXB = 5 };

static uint64_t rng_state = 88172645463325252ull;
static double uniform01(void) {   /* xorshift64 */
    rng_state ^= rng_state << 13;
    rng_state ^= rng_state >> 7;
    rng_state ^= rng_state << 17;
    return (double)(rng_state >> 11) * (1.0 / 9007199254740992.0);
}
static uint16_t to_bf16(float f) {   /* round to nearest even */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
/* e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; subnormals m * 2^-9;
 * largest finite 448): round to nearest even, saturating; and back. */
static uint8_t to_e4m3(float f) {
    const uint8_t sign = signbit(f) ? 0x80 : 0;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                           /* subnormal range */
        const double m = nearbyint(a * 512.0);          /* units of 2^-9, ties to even */
        return sign | (uint8_t)(m >= 8.0 ? 0x08 : m);  /* 8 * 2^-9 is the smallest normal */
    }
    int e;
    const double fr = frexp(a, &e);                     /* a = fr * 2^e, fr in [0.5, 1) */
    e -= 1;                                             /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
    double m = nearbyint((2.0 * fr - 1.0) * 8.0);
    if (m >= 8.0) { m = 0.0; e += 1; }
    if (e > 8 || (e == 8 && m > 6.0)) return sign | 0x7E;
    return sign | (uint8_t)((e + 7) << 3) | (uint8_t)m;
}
static float from_e4m3(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    const double mag = e == 0 ? m * ldexp(1.0, -9) : (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return (float)((c & 0x80) ? -mag : mag);
}

#define CUDA_OK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 2; } } while (0)
#define MLA_OK_(x) do { int s_ = (x); if (s_ != MLA_OK) { \
    fprintf(stderr, "%s: %s (%s)\n", #x, mla_status_string(s_), mla_last_error()); return 3; } } while (0)

int main(void) {
    const int32_t L[B] = {100, 1, 300};
    const size_t nq = (size_t)B * SQ * HQ * D, nk = (size_t)NB * P * HK * D;
    uint16_t *q = malloc(nq * 2), *k = malloc(nk * 2), *out = malloc((size_t)B * SQ * HQ * DV * 2);
    float *lse = malloc((size_t)B * HQ * SQ * 4);
    double *ref_o = malloc((size_t)B * SQ * HQ * DV * 8), *ref_l = malloc((size_t)B * HQ * SQ * 8);
    int32_t bt[B * MAXB];
    for (size_t i = 0; i < nq; ++i) q[i] = to_bf16((float)(uniform01() + uniform01() + uniform01() - 1.5) * 2.0f);
    for (size_t i = 0; i < nk; ++i) k[i] = to_bf16((float)(uniform01() + uniform01() + uniform01() - 1.5) * 2.0f);
    const int32_t perm[NB] = {7, 2, 5, 0, 8, 3, 1, 6, 4};   /* physical blocks, handed out in order */
    for (int b = 0, used = 0; b < B; ++b)
        for (int j = 0; j < MAXB; ++j) bt[b * MAXB + j] = j < (L[b] + P - 1) / P ? perm[used++] : -1;

    void *q_d, *k_d, *out_d;
    int32_t *bt_d, *L_d, *md_d, *ns_d;
    float *lse_d;
    CUDA_OK(cudaMalloc(&q_d, nq * 2));
    CUDA_OK(cudaMalloc(&k_d, nk * 2));
    CUDA_OK(cudaMalloc((void **)&bt_d, sizeof bt));
    CUDA_OK(cudaMalloc((void **)&L_d, sizeof L));
    CUDA_OK(cudaMalloc(&out_d, (size_t)B * SQ * HQ * DV * 2));
    CUDA_OK(cudaMalloc((void **)&lse_d, (size_t)B * HQ * SQ * 4));
    CUDA_OK(cudaMemcpy(q_d, q, nq * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(k_d, k, nk * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(bt_d, bt, sizeof bt, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(L_d, L, sizeof L, cudaMemcpyHostToDevice));

    int parts = 0;
    MLA_OK_(mla_get_num_sm_parts(0, SQ * HQ / HK, HK, &parts));
    CUDA_OK(cudaMalloc((void **)&md_d, (size_t)parts * MLA_METADATA_SIZE * 4));
    CUDA_OK(cudaMalloc((void **)&ns_d, (B + 1) * 4));
    MLA_OK_(mla_get_metadata(L_d, B, SQ * HQ / HK, HK, parts, md_d, ns_d, NULL));

    mla_shape_t sh;
    memset(&sh, 0, sizeof sh);
    sh.batch = B; sh.s_q = SQ; sh.h_q = HQ; sh.h_k = HK; sh.head_dim = D; sh.head_dim_v = DV;
    sh.page_block_size = P; sh.num_blocks = NB; sh.max_blocks_per_seq = MAXB; sh.num_sm_parts = parts;
    sh.q_stride[0] = SQ * HQ * D; sh.q_stride[1] = HQ * D; sh.q_stride[2] = D;
    sh.k_stride[0] = P * HK * D; sh.k_stride[1] = HK * D; sh.k_stride[2] = D;
    sh.bt_stride = MAXB;
    sh.out_stride[0] = SQ * HQ * DV; sh.out_stride[1] = HQ * DV; sh.out_stride[2] = DV;
    /* softmax_scale 0 selects 1/sqrt(576); NULL workspace selects the library's own */
    MLA_OK_(mla_decode_fwd(&sh, q_d, k_d, bt_d, L_d, md_d, ns_d, 0.0f, 1, out_d, lse_d, NULL, 0, NULL));
    CUDA_OK(cudaDeviceSynchronize());
    int bits = -1;
    MLA_OK_(mla_check_device_error(&bits, 1));
    if (bits != 0) { fprintf(stderr, "device error bits %d\n", bits); return 4; }
    CUDA_OK(cudaMemcpy(out, out_d, (size_t)B * SQ * HQ * DV * 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(lse, lse_d, (size_t)B * HQ * SQ * 4, cudaMemcpyDeviceToHost));

    /* ---- the same values rounded to e4m3, through mla_decode_fwd_fp8 */
    const float bmm1 = 0.8f / 24.0f, bmm2 = 1.5f;
    uint8_t *q8 = malloc(nq), *k8 = malloc(nk);
    uint16_t *q8v = malloc(nq * 2), *k8v = malloc(nk * 2), *out8 = malloc((size_t)B * SQ * HQ * DV * 2);
    float *lse8 = malloc((size_t)B * HQ * SQ * 4);
    for (size_t i = 0; i < nq; ++i) { q8[i] = to_e4m3(from_bf16(q[i])); q8v[i] = to_bf16(from_e4m3(q8[i])); }
    for (size_t i = 0; i < nk; ++i) { k8[i] = to_e4m3(from_bf16(k[i])); k8v[i] = to_bf16(from_e4m3(k8[i])); }
    void *q8_d, *k8_d;
    CUDA_OK(cudaMalloc(&q8_d, nq));
    CUDA_OK(cudaMalloc(&k8_d, nk));
    CUDA_OK(cudaMemcpy(q8_d, q8, nq, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(k8_d, k8, nk, cudaMemcpyHostToDevice));
    MLA_OK_(mla_decode_fwd_fp8(&sh, q8_d, k8_d, bt_d, L_d, md_d, ns_d, bmm1, bmm2, 1, out_d, lse_d, NULL, 0, NULL));
    CUDA_OK(cudaDeviceSynchronize());
    MLA_OK_(mla_check_device_error(&bits, 1));
    if (bits != 0) { fprintf(stderr, "device error bits %d (e4m3)\n", bits); return 4; }
    CUDA_OK(cudaMemcpy(out8, out_d, (size_t)B * SQ * HQ * DV * 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(lse8, lse_d, (size_t)B * HQ * SQ * 4, cudaMemcpyDeviceToHost));
    MLA_OK_(mla_shutdown());

    const int64_t qs[3] = {SQ * HQ * D, HQ * D, D}, ks[3] = {P * HK * D, HK * D, D};
    if (oracle_mla_decode(B, SQ, HQ, HK, D, DV, P, NB, MAXB, q, qs, k, ks, bt, MAXB, L, 1.0 / sqrt((double)D), 1,
                          NULL, -1, ref_o, ref_l, 1) != 0) {
        fprintf(stderr, "oracle failed\n");
        return 5;
    }
    double max_o = 0.0, max_l = 0.0;
    for (size_t i = 0; i < (size_t)B * SQ * HQ * DV; ++i) {
        const double e = fabs((double)from_bf16(out[i]) - ref_o[i]);
        if (e > 1e-2 + 1e-2 * fabs(ref_o[i])) { fprintf(stderr, "out %zu: %g vs %g\n", i, from_bf16(out[i]), ref_o[i]); return 6; }
        if (e > max_o) max_o = e;
    }
    for (size_t i = 0; i < (size_t)B * HQ * SQ; ++i) {
        if (isinf(ref_l[i]) && isinf(lse[i]) && lse[i] < 0) continue;
        const double e = fabs((double)lse[i] - ref_l[i]);
        if (!(e <= 2e-3)) { fprintf(stderr, "lse %zu: %g vs %g\n", i, lse[i], ref_l[i]); return 7; }
        if (e > max_l) max_l = e;
    }
    /* e4m3: the oracle on the decoded values (exact in bf16) with scale bmm1, output times bmm2 */
    if (oracle_mla_decode(B, SQ, HQ, HK, D, DV, P, NB, MAXB, q8v, qs, k8v, ks, bt, MAXB, L, (double)bmm1, 1,
                          NULL, -1, ref_o, ref_l, 1) != 0) {
        fprintf(stderr, "oracle failed (e4m3)\n");
        return 5;
    }
    double max_o8 = 0.0, max_l8 = 0.0;
    for (size_t i = 0; i < (size_t)B * SQ * HQ * DV; ++i) {
        const double r = bmm2 * ref_o[i], e = fabs((double)from_bf16(out8[i]) - r);
        if (!(e <= 0.03 + 0.03 * fabs(r))) { fprintf(stderr, "e4m3 out %zu: %g vs %g\n", i, from_bf16(out8[i]), r); return 8; }
        if (e > max_o8) max_o8 = e;
    }
    for (size_t i = 0; i < (size_t)B * HQ * SQ; ++i) {
        if (isinf(ref_l[i]) && isinf(lse8[i]) && lse8[i] < 0) continue;
        const double e = fabs((double)lse8[i] - ref_l[i]);
        if (!(e <= 2e-3)) { fprintf(stderr, "e4m3 lse %zu: %g vs %g\n", i, lse8[i], ref_l[i]); return 9; }
        if (e > max_l8) max_l8 = e;
    }
    printf("capi ok: parts %d, max |out err| %.3g, max |lse err| %.3g; e4m3 max |out err| %.3g, |lse err| %.3g\n",
           parts, max_o, max_l, max_o8, max_l8);
    return 0;
}
