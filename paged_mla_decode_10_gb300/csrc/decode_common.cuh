// decode_common.cuh -- parameters and schedule walk shared by the decode kernels.
#pragma once

#include <cstdint>

namespace mla {

constexpr int kPage = 64;          // cache rows per physical block
constexpr int kDqk = 576;          // q / cache row dims (512 latent + 64 RoPE)
constexpr int kDv = 512;           // V dims (prefix of each cache row)
constexpr int kMdSize = 8;         // int32 per scheduler record
// Schedule: the cost of opening a segment, in 64-row blocks -- a part's fixed work
// for each sequence it takes up (the query load, the pipeline refill and the output
// store), measured on the decode kernel against its page time: about 6 pages with 64
// or more query rows per KV head, about 4 with fewer; one more with an e4m3 cache,
// whose pages take less time than bf16 ones.
__host__ __device__ constexpr int segment_cost(int rows_per_head_k, int kv_bytes) {
    return (rows_per_head_k >= 64 ? 6 : 4) + (kv_bytes == 1 ? 1 : 0);
}
constexpr int kRowsPerBlock = 128; // query rows per CTA (tcgen05 M)

// Device-side error bits (mirror MLA_DEVERR_* of the public header).
constexpr int kErrTimeout = 1;
constexpr int kErrBadBlock = 2;

struct DecodeParams {
    const uint16_t *q;             // bf16 latent dims of q: (B, s_q, h_q, >= 512)
    int64_t q_s0, q_s1, q_s2;
    const uint16_t *q_rope;        // bf16 RoPE dims of q: (B, s_q, h_q, 64); q + 512 when q holds all 576
    int64_t qr_s0, qr_s1, qr_s2;
    const int32_t *block_table;
    int64_t bt_stride;
    const int32_t *seqlens;
    const int32_t *md;             // (num_parts, 8)
    const int32_t *num_splits;     // (B + 1)
    uint16_t *out;                 // bf16 (B, s_q, h_q, 512)
    int64_t o_s0, o_s1, o_s2;
    float *lse;                    // (B, h_q, s_q)
    float *ws_o;                   // (slots, h_k, R, 512) fp32 partial outputs
    float *ws_lse;                 // (slots, h_k, R) fp32 partial lse
    int *err;                      // device error word
    int batch, s_q, h_q, h_k, hpk, rows;   // rows = R = s_q * h_q / h_k
    int num_blocks, max_blocks, num_parts, max_slots;
    int causal;
    int q_concat;                  // q_rope == q + 512 with q's strides: one 576-dim row per query
    int rope_x0;                   // first RoPE dim in the RoPE tensor map (512 over a 576-dim cache, else 0)
    float scale_log2;              // softmax_scale * log2(e) (bmm1_scale * log2(e) for e4m3 inputs)
    const uint8_t *q8;             // e4m3 q (B, s_q, h_q, 576), strides q_s0..2 in bytes (e4m3 kernel only)
    float out_scale;               // bmm2_scale: factor on the output of the e4m3 kernel
    // Q by TMA (q_tma = 1): the tensor maps of the latent and RoPE query dims
    // {dims, h_q, s_q, batch}; a latent box covers a 128-row block (q_hb heads x
    // q_tb tokens), a RoPE box 64 rows; the RoPE boxes start at dim qr_x0.
    int q_tma;
    int q_hb, q_tb, qr_x0;
};

// One contiguous run of blocks of one sequence assigned to a part.
struct Segment {
    int b, lo, hi, L, slot, nsplit;
};

// Walks a part's record exactly as the schedule defines it.  Every role of
// a CTA runs its own copy and sees the same segments.
struct SegmentWalk {
    int b, b0, k0, b1, k1, first_slot;
    bool first;

    __device__ __forceinline__ void init(const int32_t *rec) {
        b0 = rec[0]; k0 = rec[1]; b1 = rec[2]; k1 = rec[3]; first_slot = rec[4];
        b = b0 < 0 ? 0 : b0;
        first = true;
    }
    __device__ __forceinline__ bool next(const DecodeParams &p, Segment &s) {
        while (b <= b1 && b < p.batch) {
            const int cb = b++;
            int L = __ldg(p.seqlens + cb);
            L = L < 0 ? 0 : L;
            int nb = (L + kPage - 1) / kPage;
            if (nb > p.max_blocks) {          // block table shorter than the sequence
                atomicOr(p.err, kErrBadBlock);
                nb = p.max_blocks;
                L = nb * kPage;
            }
            const int lo = cb == b0 ? k0 : 0;
            int hi = cb == b1 ? k1 : nb;
            hi = hi > nb ? nb : hi;
            if (lo >= hi || lo < 0) continue;
            s.b = cb; s.lo = lo; s.hi = hi; s.L = L;
            const int ns0 = __ldg(p.num_splits + cb), ns1 = __ldg(p.num_splits + cb + 1);
            s.slot = first ? first_slot : ns0;
            s.nsplit = ns1 - ns0;
            first = false;
            return true;
        }
        return false;
    }
};

// Page-by-page cursor over a part's segments (used to run ahead of the
// consumer, e.g. for L2 prefetch).
struct PageCursor {
    SegmentWalk walk;
    Segment s;
    int blk;
    bool valid;

    __device__ __forceinline__ void init(const int32_t *rec, const DecodeParams &p) {
        walk.init(rec);
        valid = walk.next(p, s);
        blk = valid ? s.lo : 0;
    }
    __device__ __forceinline__ void advance(const DecodeParams &p) {
        if (!valid) return;
        if (++blk >= s.hi) {
            valid = walk.next(p, s);
            blk = valid ? s.lo : 0;
        }
    }
};

}  // namespace mla
