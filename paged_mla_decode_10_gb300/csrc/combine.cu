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
// One 128-thread block per four query rows of one (sequence, KV head): warp
// w merges row 4 blockIdx.x + w, lane l owning dims [16 l, 16 l + 16).  The
// split list is merged in one pass, kChunk splits at a time: every load of a
// chunk (its lse values and 16 dims of each partial row per lane) is issued
// before any is used, and the running max, sum and weighted sum are rescaled
// from chunk to chunk (the same log-sum-exp identity, evaluated online).
// A sequence split over at most kChunk parts -- nearly every one -- costs a
// single round trip to memory.  HBM/L2-bound: splits * 2052 B read and
// 1028 B written per row.
//
// The kernel is launched as a programmatic dependent of the split-KV kernel:
// its blocks may become resident while that kernel still runs, and
// griddepcontrol.wait holds them until its results are complete and visible.
#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "sm103.cuh"
#include "decode_common.cuh"

namespace mla {

namespace {
constexpr int kThreadsCombine = 128;
constexpr int kRowsPerCombineBlock = kThreadsCombine / 32;
constexpr int kChunk = 4;                      // splits whose loads are in flight together
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
}  // namespace

__global__ void __launch_bounds__(kThreadsCombine, 4) mla_combine_kernel(const __grid_constant__ DecodeParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_g = blockIdx.x * kRowsPerCombineBlock + warp, b = blockIdx.y, hk = blockIdx.z;
    // num_splits comes from the schedule, which completed before the decode kernel began, so it
    // is read before waiting for the decode; only the partial results need the wait
    const int ns0 = __ldg(p.num_splits + b);
    const int ns = __ldg(p.num_splits + b + 1) - ns0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (row_g >= p.rows) return;
    if (ns == 1) return;   // finished by the decode kernel
    const bool in_range = ns0 >= 0 && ns0 + ns <= p.max_slots;
    const int n = in_range ? ns : 0;
    const int qi = row_g / p.hpk, qh = hk * p.hpk + row_g % p.hpk;
    uint4 *orow = reinterpret_cast<uint4 *>(p.out + (int64_t)b * p.o_s0 + (int64_t)qi * p.o_s1 +
                                            (int64_t)qh * p.o_s2) + 2 * lane;
    float *lse_out = p.lse + ((int64_t)b * p.h_q + qh) * p.s_q + qi;
    const int64_t stride = (int64_t)p.h_k * p.rows;                    // between consecutive slots
    const int64_t prow0 = ((int64_t)ns0 * p.h_k + hk) * p.rows + row_g; // first partial of this row
    const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + prow0 * kDv) + 4 * lane;
    const int64_t sstride = stride * (kDv / 4);                        // float4s between slots

    // running state, log2 domain: m = max of lse_s * log2(e) so far, l = sum 2^(. - m), acc = sum 2^(. - m) o_s
    float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int s0 = 0; s0 < n; s0 += kChunk) {
        float ls[kChunk];
        float4 x[kChunk][4];
#pragma unroll
        for (int sp = 0; sp < kChunk; ++sp) {
            const bool in = s0 + sp < n;
            ls[sp] = in ? __ldg(p.ws_lse + prow0 + (s0 + sp) * stride) * kLog2e : -INFINITY;
            // the lane's 64 bytes of the partial row as two 32-byte (one-sector) loads
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = 0u;
            if (in) {
                ldg_nc_v8(src + (s0 + sp) * sstride, &w[0]);
                ldg_nc_v8(src + (s0 + sp) * sstride + 2, &w[8]);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v)
                x[sp][v] = make_float4(__uint_as_float(w[4 * v]), __uint_as_float(w[4 * v + 1]),
                                       __uint_as_float(w[4 * v + 2]), __uint_as_float(w[4 * v + 3]));
        }
        float mc = m;
#pragma unroll
        for (int sp = 0; sp < kChunk; ++sp) mc = fmaxf(mc, ls[sp]);
        if (mc == -INFINITY) continue;   // no visible key in any split so far
        const float scale = m == -INFINITY ? 0.f : ex2_approx(m - mc);
        l *= scale;
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] *= scale;
#pragma unroll
        for (int sp = 0; sp < kChunk; ++sp) {
            const float e = ls[sp] == -INFINITY ? 0.f : ex2_approx(ls[sp] - mc);
            l += e;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                acc[4 * v] = fmaf(e, x[sp][v].x, acc[4 * v]); acc[4 * v + 1] = fmaf(e, x[sp][v].y, acc[4 * v + 1]);
                acc[4 * v + 2] = fmaf(e, x[sp][v].z, acc[4 * v + 2]); acc[4 * v + 3] = fmaf(e, x[sp][v].w, acc[4 * v + 3]);
            }
        }
        m = mc;
    }
    if (m == -INFINITY) {   // empty sequence, or no part saw a visible key
        orow[0] = make_uint4(0u, 0u, 0u, 0u);
        orow[1] = make_uint4(0u, 0u, 0u, 0u);
        if (lane == 0) *lse_out = -INFINITY;
        return;
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] *= inv;
    orow[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    orow[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                         pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
    float lg;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l));
    if (lane == 0) *lse_out = (m + lg) * kLn2;
}

uint32_t combine_threads() { return kThreadsCombine; }
uint32_t combine_rows_per_block() { return kRowsPerCombineBlock; }

}  // namespace mla
