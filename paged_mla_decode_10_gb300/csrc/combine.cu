// combine.cu -- merge of the split-KV partial results.
//
// The split-KV decode leaves, for every (split sequence, KV head, query row)
// and every part s that touched the sequence, a normalised partial output
// o_s (fp32, 512 dims) and its natural-log lse_s.  The exact merge is the
// log-sum-exp identity: lse = ln sum_s exp(lse_s), out = sum_s
// exp(lse_s - lse) o_s (softmax_lse semantics of the FlashMLA-PyTorch page,
// flash_mla_with_kvcache docstring; the partial layout is this library's).
// Sequences the schedule gave a single part were finished by the decode
// kernel and are skipped; empty sequences get out = 0, lse = -inf.
//
// One warp per query row; lane l owns output dims [16 l, 16 l + 16).
// HBM-bound: reads splits * 2052 B and writes 1028 B per row.
#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "sm103.cuh"
#include "decode_common.cuh"

namespace mla {

__global__ void __launch_bounds__(256) mla_combine_kernel(const __grid_constant__ DecodeParams p) {
    const int b = blockIdx.x, hk = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_g = blockIdx.z * 8 + warp;
    if (row_g >= p.rows) return;
    const int ns0 = __ldg(p.num_splits + b);
    const int ns = __ldg(p.num_splits + b + 1) - ns0;
    if (ns == 1) return;
    const int qi = row_g / p.hpk, qh = hk * p.hpk + row_g % p.hpk;
    uint4 *orow = reinterpret_cast<uint4 *>(p.out + (int64_t)b * p.o_s0 + (int64_t)qi * p.o_s1 +
                                            (int64_t)qh * p.o_s2) + 2 * lane;
    float *lse_out = p.lse + ((int64_t)b * p.h_q + qh) * p.s_q + qi;
    const bool in_range = ns0 >= 0 && ns0 + ns <= p.max_slots;

    float mx = -INFINITY;
    if (ns > 0 && in_range)
        for (int s = lane; s < ns; s += 32)
            mx = fmaxf(mx, __ldg(p.ws_lse + ((int64_t)(ns0 + s) * p.h_k + hk) * p.rows + row_g));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    if (mx == -INFINITY) {   // empty sequence, or no part saw a visible key
        orow[0] = make_uint4(0u, 0u, 0u, 0u);
        orow[1] = make_uint4(0u, 0u, 0u, 0u);
        if (lane == 0) *lse_out = -INFINITY;
        return;
    }
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
    float sum = 0.f;
    for (int s = lane; s < ns; s += 32) {
        const float l = __ldg(p.ws_lse + ((int64_t)(ns0 + s) * p.h_k + hk) * p.rows + row_g);
        sum += ex2_approx((l - mx) * kLog2e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    float lg;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(sum));
    const float lse = mx + lg * kLn2;

    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const int64_t prow = ((int64_t)(ns0 + s) * p.h_k + hk) * p.rows + row_g;
        const float w = ex2_approx((__ldg(p.ws_lse + prow) - lse) * kLog2e);
        const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + prow * kDv) + 4 * lane;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float4 x = __ldg(src + v);
            acc[4 * v] += w * x.x; acc[4 * v + 1] += w * x.y; acc[4 * v + 2] += w * x.z; acc[4 * v + 3] += w * x.w;
        }
    }
    orow[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    orow[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                         pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
    if (lane == 0) *lse_out = lse;
}

}  // namespace mla
