// decode_epilogue.cuh -- coalesced store of a CTA's normalised O half.
//
// After the last PV of a segment, thread r of softmax warp w holds query row
// 32 w + r of the 128-row block in TMEM lane 32 w + r.  Stored straight from
// registers, each store instruction of a warp would touch 32 rows with 16
// bytes apiece.  Here each warp passes its rows through a 32 x 64-byte staging
// tile in shared memory (16-byte chunks XOR-swizzled by row bits 1-2, so neither
// the row-wise writes nor the segment-wise reads conflict on banks), so that a
// store instruction writes eight 64-byte row segments (whole 32-byte sectors):
// bf16 to `out` when the sequence was not split, fp32 partial rows to the
// workspace otherwise.
#pragma once

#include <cstdint>

#include "sm103.cuh"
#include "decode_common.cuh"

namespace mla {

constexpr uint32_t kEpiPitch = 64;                    // bytes per staged row
constexpr uint32_t kEpiWarpBytes = 32 * kEpiPitch;    // staging tile of one warp

// Byte offset of 16-byte chunk c of staged row r.
static __device__ __forceinline__ uint32_t epi_offset(uint32_t r, uint32_t c) {
    return r * kEpiPitch + ((c ^ ((r >> 1) & 3u)) << 4);
}

// tmem_o: TMEM address of the warp's lane quadrant at the O columns.
// stage:  the warp's staging tile (16-byte aligned, kEpiWarpBytes).
// row0:   row (within the KV head's R rows) of the warp's lane 0.
// inv:    1 / denominator of this thread's row (0 for a row with no visible key).
static __device__ __forceinline__ void store_o_half(const DecodeParams &p, uint32_t tmem_o, uint8_t *stage, int lane,
                                                    int row0, int b, int hk, int cta, bool direct, bool slot_ok,
                                                    int slot, float inv) {
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t o[64];
        tmem_ld_32x32b_x64(tmem_o + 64u * q4, o);
        tmem_ld_wait();
        if (direct) {
            // 64 dims of bf16 per row: two passes of 32 dims (64 bytes)
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int j = 32 * sub + 8 * v;
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(o[j + 0]) * inv, __uint_as_float(o[j + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
                    *reinterpret_cast<uint4 *>(stage + epi_offset(lane, v)) = w;
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int f = lane + 32 * i, rr = f >> 2, cc = f & 3;
                    const int row_g = row0 + rr;
                    if (row_g < p.rows) {
                        const int qi = row_g / p.hpk, qh = hk * p.hpk + row_g % p.hpk;
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + (int64_t)b * p.o_s0 + (int64_t)qi * p.o_s1 +
                                                               (int64_t)qh * p.o_s2 + 256 * cta + 64 * q4 + 32 * sub) + cc;
                        *dst = *reinterpret_cast<const uint4 *>(stage + epi_offset(rr, cc));
                    }
                }
                __syncwarp();
            }
        } else if (slot_ok) {
            // 64 dims of fp32 per row: four passes of 16 dims (64 bytes)
#pragma unroll
            for (int sub = 0; sub < 4; ++sub) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int j = 16 * sub + 4 * v;
                    const float2 lo = __fmul2_rn(make_float2(__uint_as_float(o[j]), __uint_as_float(o[j + 1])),
                                                 make_float2(inv, inv));
                    const float2 hi = __fmul2_rn(make_float2(__uint_as_float(o[j + 2]), __uint_as_float(o[j + 3])),
                                                 make_float2(inv, inv));
                    *reinterpret_cast<float4 *>(stage + epi_offset(lane, v)) = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int f = lane + 32 * i, rr = f >> 2, cc = f & 3;
                    const int row_g = row0 + rr;
                    if (row_g < p.rows) {
                        const int64_t prow = ((int64_t)slot * p.h_k + hk) * p.rows + row_g;
                        float4 *dst = reinterpret_cast<float4 *>(p.ws_o + prow * kDv + 256 * cta + 64 * q4 + 16 * sub) + cc;
                        *dst = *reinterpret_cast<const float4 *>(stage + epi_offset(rr, cc));
                    }
                }
                __syncwarp();
            }
        }
    }
}

}  // namespace mla
