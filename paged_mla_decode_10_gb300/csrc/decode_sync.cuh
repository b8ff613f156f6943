// decode_sync.cuh -- bounded mbarrier waits and the page gather check shared
// by the split-KV decode kernels.
//
// Every wait is bounded: after kWaitLimitCycles a role sets the CTA's abort
// flag and MLA_DEVERR_TIMEOUT in the device error word and returns false, and
// the other roles of the CTA see the flag and stop too.  Teardown waits
// (drain_bar) ignore the flag, so copies and MMAs already in flight complete
// before shared memory and TMEM are released; they are bounded as well
// (kTimeoutCycles).
#pragma once

#include <cstdint>

#include "sm103.cuh"
#include "decode_common.cuh"

namespace mla {

// Limit of the waits of the main loops.  A test build sets MLA_WAIT_LIMIT_CYCLES
// far below a page's latency, so that the first wait runs out and the timeout
// path (error bit, drain, exit) is exercised; the library is built without it.
#ifndef MLA_WAIT_LIMIT_CYCLES
#define MLA_WAIT_LIMIT_CYCLES 4000000000ll
#endif
constexpr long long kWaitLimitCycles = MLA_WAIT_LIMIT_CYCLES;
// Limit of the teardown waits (drains): long in every build, so that each copy
// and MMA in flight has landed before shared memory and TMEM are released.
constexpr long long kTimeoutCycles = 4000000000ll;

struct Ctx {
    uint32_t base;              // shared address of the 1024-byte aligned smem base
    uint32_t bars;              // shared address of the mbarrier array
    volatile int *abort_flag;
    int *err;
};

static __device__ __forceinline__ uint32_t bar_addr(const Ctx &c, int i) { return c.bars + 8u * (uint32_t)i; }

static __device__ __noinline__ void raise_timeout(const Ctx &c) {
    *c.abort_flag = 1;
    atomicOr(c.err, kErrTimeout);
}

// Bounded wait; false when it timed out or another role already aborted.
static __device__ __forceinline__ bool wait_bar(const Ctx &c, uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_test(bar, parity)) {
        if (*c.abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) { raise_timeout(c); return false; }
    }
    return true;
}

// Teardown wait: ignores the abort flag (drains what is in flight), still bounded.
static __device__ __forceinline__ void drain_bar(const Ctx &c, uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_test(bar, parity)) {
        if (clock64() - t0 > kTimeoutCycles) { raise_timeout(c); return; }
    }
}

// Physical block of logical block `blk` of sequence `b`; an entry outside
// [0, num_blocks) raises MLA_DEVERR_BAD_BLOCK and reads block 0 instead, so no
// copy ever leaves the cache.
static __device__ __forceinline__ int checked_phys(const DecodeParams &p, int b, int blk) {
    int phys = __ldg(p.block_table + (int64_t)b * p.bt_stride + blk);
    if (phys < 0 || phys >= p.num_blocks) {
        atomicOr(p.err, kErrBadBlock);
        phys = 0;
    }
    return phys;
}

// Asks L2 for the query rows [64 half, 64 half + 64) of row block rb of KV head
// hk of sequence b (their 512 latent and 64 RoPE dims), so that the loads of
// the next segment's Q hit L2.  Warp-wide; rows that are not 16-byte aligned
// are skipped.
static __device__ __forceinline__ void prefetch_q_rows(const DecodeParams &p, int b, int rb, int hk, int half,
                                                       int lane) {
    for (int i = lane; i < 64; i += 32) {
        const int row_g = rb * kRowsPerBlock + half * 64 + i;
        if (row_g >= p.rows) break;
        const int qi = row_g / p.hpk, qh = hk * p.hpk + row_g % p.hpk;
#if MLA_F8
        const uint8_t *row8 = p.q8 + (int64_t)b * p.q_s0 + (int64_t)qi * p.q_s1 + (int64_t)qh * p.q_s2;
        if ((reinterpret_cast<uintptr_t>(row8) & 15u) == 0) bulk_prefetch_l2(row8, kDqk);   // the 576-byte e4m3 row
        continue;
#endif
        const uint16_t *row = p.q + (int64_t)b * p.q_s0 + (int64_t)qi * p.q_s1 + (int64_t)qh * p.q_s2;
        if ((reinterpret_cast<uintptr_t>(row) & 15u) != 0) continue;
        if (p.q_concat) {
            bulk_prefetch_l2(row, kDqk * 2);   // one request per whole row
        } else {
            bulk_prefetch_l2(row, kDv * 2);
            const uint16_t *rope = p.q_rope + (int64_t)b * p.qr_s0 + (int64_t)qi * p.qr_s1 + (int64_t)qh * p.qr_s2;
            if ((reinterpret_cast<uintptr_t>(rope) & 15u) == 0) bulk_prefetch_l2(rope, (kDqk - kDv) * 2);
        }
    }
}

}  // namespace mla
