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
// One 128-thread block per (query row, sequence, KV head).  Rows of
// sequences split over at most kWarpSplits parts (the common case) are
// merged by the block's first warp alone, lane l owning dims [16 l, 16 l + 16);
// longer split lists use the whole block, thread t owning dims [4t, 4t + 4),
// so each split is one coalesced 2 KB read.  Split loops are unrolled so
// several splits' loads are in flight.  HBM/L2-bound: splits * 2052 B read
// and 1028 B written per row.
#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "sm103.cuh"
#include "decode_common.cuh"

namespace mla {

namespace {
constexpr int kThreadsCombine = 128;
constexpr int kWarpSplits = 16;
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float block_reduce_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    v = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    return v;
}
__device__ __forceinline__ float block_reduce_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    v = (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();
    return v;
}
}  // namespace

__global__ void __launch_bounds__(kThreadsCombine) mla_combine_kernel(const __grid_constant__ DecodeParams p) {
    __shared__ float red[4];
    const int row_g = blockIdx.x, b = blockIdx.y, hk = blockIdx.z;
    const int t = threadIdx.x;
    const int ns0 = __ldg(p.num_splits + b);
    const int ns = __ldg(p.num_splits + b + 1) - ns0;
    if (ns == 1) return;
    const int qi = row_g / p.hpk, qh = hk * p.hpk + row_g % p.hpk;
    uint2 *orow = reinterpret_cast<uint2 *>(p.out + (int64_t)b * p.o_s0 + (int64_t)qi * p.o_s1 +
                                            (int64_t)qh * p.o_s2) + t;
    float *lse_out = p.lse + ((int64_t)b * p.h_q + qh) * p.s_q + qi;
    const bool in_range = ns0 >= 0 && ns0 + ns <= p.max_slots;
    const int64_t stride = (int64_t)p.h_k * p.rows;                    // between consecutive slots
    const int64_t prow0 = ((int64_t)ns0 * p.h_k + hk) * p.rows + row_g; // first partial of this row

    if (ns <= kWarpSplits) {
        // ---- one warp: lane s < ns holds lse_s; lane l owns dims [16 l, 16 l + 16)
        if (t >= 32) return;
        const float ls = (t < ns && in_range) ? __ldg(p.ws_lse + prow0 + t * stride) : -INFINITY;
        float mx = ls;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        uint4 *orow4 = reinterpret_cast<uint4 *>(p.out + (int64_t)b * p.o_s0 + (int64_t)qi * p.o_s1 +
                                                 (int64_t)qh * p.o_s2) + 2 * t;
        if (mx == -INFINITY) {
            orow4[0] = make_uint4(0u, 0u, 0u, 0u);
            orow4[1] = make_uint4(0u, 0u, 0u, 0u);
            if (t == 0) *lse_out = -INFINITY;
            return;
        }
        float e = t < ns ? ex2_approx((ls - mx) * kLog2e) : 0.f;
        float sum = e;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.f / sum;
        float lg;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(sum));
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + prow0 * kDv) + 4 * t;
        const int64_t sstride = stride * (kDv / 4);
#pragma unroll 4
        for (int s = 0; s < ns; ++s) {
            const float w = __shfl_sync(0xffffffffu, e, s) * inv;   // exp(lse_s - lse)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 x = __ldg(src + s * sstride + v);
                acc[4 * v] = fmaf(w, x.x, acc[4 * v]); acc[4 * v + 1] = fmaf(w, x.y, acc[4 * v + 1]);
                acc[4 * v + 2] = fmaf(w, x.z, acc[4 * v + 2]); acc[4 * v + 3] = fmaf(w, x.w, acc[4 * v + 3]);
            }
        }
        orow4[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                              pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
        orow4[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                              pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
        if (t == 0) *lse_out = mx + lg * kLn2;
        return;
    }

    // ---- whole block

    float mx = -INFINITY;
    if (ns > 0 && in_range)
        for (int s = t; s < ns; s += kThreadsCombine) mx = fmaxf(mx, __ldg(p.ws_lse + prow0 + s * stride));
    mx = block_reduce_max(mx, red);
    if (mx == -INFINITY) {   // empty sequence, or no part saw a visible key
        *orow = make_uint2(0u, 0u);
        if (t == 0) *lse_out = -INFINITY;
        return;
    }
    float sum = 0.f;
    for (int s = t; s < ns; s += kThreadsCombine) sum += ex2_approx((__ldg(p.ws_lse + prow0 + s * stride) - mx) * kLog2e);
    sum = block_reduce_sum(sum, red);
    float lg;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(sum));
    const float lse = mx + lg * kLn2;

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + prow0 * kDv) + t;
    const int64_t sstride = stride * (kDv / 4);                        // float4s between slots
#pragma unroll 4
    for (int s = 0; s < ns; ++s) {
        const float w = ex2_approx((__ldg(p.ws_lse + prow0 + s * stride) - lse) * kLog2e);
        const float4 x = __ldg(src + s * sstride);
        acc.x = fmaf(w, x.x, acc.x); acc.y = fmaf(w, x.y, acc.y);
        acc.z = fmaf(w, x.z, acc.z); acc.w = fmaf(w, x.w, acc.w);
    }
    *orow = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    if (t == 0) *lse_out = lse;
}

uint32_t combine_threads() { return kThreadsCombine; }

}  // namespace mla
