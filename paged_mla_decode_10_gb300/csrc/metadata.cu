// metadata.cu -- split-KV schedule (get_mla_metadata) on the device.
//
// Output shapes follow the FlashMLA-PyTorch page (flash_mla_interface.py,
// get_mla_metadata docstring): tile_scheduler_metadata (num_sm_parts,
// TileSchedulerMetaDataSize) int32 and num_splits (batch_size + 1) int32.
// The record and policy are this library's:
//
//   record of part p: [begin_b, begin_blk, end_b, end_blk, first_slot, num_blocks, 0, 0]
//   n_b = ceil(max(L_b, 0) / 64); c = cost of opening a segment, in blocks
//   (segment_cost: 6 with >= 64 query rows per KV head, 4 with fewer, +1 for e4m3)
//   W = sum_{n_b > 0} (n_b + c);  T = max(1, ceil((W + (parts - 1) c) / parts))
//   parts walk the (b, blk) sequence in order; a part stops opening segments
//   when T - load - c <= 0, takes min(remaining, T - load - c) blocks when it
//   opens one, and the last part takes the rest.
//   num_splits = exclusive prefix sum of the per-sequence segment counts;
//   first_slot = num_splits[b] + (number of earlier parts that touched b)
//   for the part's first sequence b.
//
// One CTA.  All threads compute the block counts and, with one block-wide
// scan, the cost prefix C[b] = (blocks before b) + c (non-empty sequences
// before b) -- the load a part would carry from sequence 0 up to b if it
// opened every segment -- and E[b], the count of non-empty sequences before b.
// A part that starts at cost position g (block k of sequence b: g = C[b] + k)
// carries load C[j] - g on reaching a later sequence j, so it stops in the
// first sequence j with C[j + 1] >= g + T, and where inside j it stops
// follows from C[j], C[j + 1], g and T alone: it ends at the start of j (no
// budget left to open j: a "snap"), at the start of j + 1 (it takes exactly
// the rest of j: also a snap), or inside j at g + T - c.  Between snaps the
// parts' starts are therefore g0, g0 + (T - c), g0 + 2 (T - c), ...
//
// One warp walks the parts in rounds: lane m takes the m-th part after the
// current start g0 as if none before it snapped (start g0 + m (T - c)),
// binary-searches its stop sequence and computes its end; a ballot finds the
// first lane whose part snaps, the ends up to it are final, and the next
// round starts from there.  After a round that advanced a single part, the
// next part is tried first against a window of 32 sequences (one load per
// lane instead of a binary search); runs of snapping parts go that way.  The
// records, the per-sequence split counts, num_splits and the first slots
// follow from the boundaries in parallel (binary searches over the block
// prefix sums and over the parts' first blocks).  The result is exactly the
// sequential walk's.
#include <cuda_runtime.h>
#include <cstdint>

#include "decode_common.cuh"

namespace mla {

namespace {

constexpr int kThreadsMd = 256;
// A scanned value packs (non-empty sequences << 48) | blocks: at most 16384
// sequences and fewer than 2^48 blocks in all.
constexpr int kPackShift = 48;

// Block-wide exclusive scan of one value per thread (+ total), 256 threads.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long *warp_tot, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    long long off = 0, tot = 0;
    for (int w = 0; w < kThreadsMd / 32; ++w) {
        if (w < warp) off += warp_tot[w];
        tot += warp_tot[w];
    }
    __syncthreads();
    *total = tot;
    return off + incl - v;
}

// Index of the last i in [0, n) with at(i) <= x, for a nondecreasing at() with at(0) <= x.
template <class F>
__device__ __forceinline__ int last_le(int n, long long x, F at) {
    int lo = 0, hi = n;   // at(lo) <= x, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (at(mid) <= x) lo = mid; else hi = mid;
    }
    return lo;
}

// Where a part that starts at cost position g stops, given its stop sequence
// j (C[j] = cj, C[j + 1] = cj1): end (eb, ek), the end's cost position eg and
// whether it is a snap (ends at a sequence start).
__device__ __forceinline__ void part_end(long long g, long long T, long long c, int j, long long cj, long long cj1,
                                         int &eb, int &ek, long long &eg, bool &snap) {
    const long long start = cj > g ? cj : g;                 // cost position where the part enters j
    const long long avail = g + T - c - start;               // blocks it may take from j
    const long long rem = cj1 - c - start;                   // blocks of j left
    eb = j; ek = 0; eg = cj; snap = true;                    // no budget to open j
    if (avail > 0) {
        if (rem == avail) { eb = j + 1; eg = cj1; }          // takes the rest of j exactly
        else { ek = (int)(start + avail - cj); eg = start + avail; snap = false; }   // stops inside j
    }
}

}  // namespace

// Shared memory: C[batch + 1] (cost prefix), gs[parts + 1] (first global
// block of each part), E[batch + 1] (non-empty sequences before each
// sequence), pb/pk[parts + 1] (part boundaries as (sequence, block)).
__global__ void __launch_bounds__(kThreadsMd) mla_metadata_kernel(const int32_t *__restrict__ seqlens, int batch,
                                                                  int parts, int cost, int32_t *__restrict__ md,
                                                                  int32_t *__restrict__ num_splits) {
    extern __shared__ long long smd[];
    long long *C = smd;                                            // batch + 1
    long long *gs = C + batch + 1;                                 // parts + 1
    int32_t *E = reinterpret_cast<int32_t *>(gs + parts + 1);      // batch + 1
    int32_t *pb = E + batch + 1;                                   // parts + 1
    int32_t *pk = pb + parts + 1;                                  // parts + 1
    __shared__ long long warp_tot[kThreadsMd / 32];
    const int tid = threadIdx.x, lane = tid & 31;
    constexpr long long kMask = (1ll << kPackShift) - 1;
    // first global block of sequence i
    const long long c = cost;   // cost of opening a segment, in blocks
    auto pre = [&](int i) -> long long { return C[i] - c * E[i]; };

    // ---- block counts; one scan gives the block prefix and the non-empty count prefix
    const int per = (batch + kThreadsMd - 1) / kThreadsMd;
    const int b0 = tid * per, b1 = min(batch, b0 + per);
    long long local = 0;
    for (int b = b0; b < b1; ++b) {
        const int L = max(seqlens[b], 0);
        const long long n = ((long long)L + kPage - 1) / kPage;
        local += n + (n > 0 ? (1ll << kPackShift) : 0);
    }
    long long total = 0;
    long long off = block_exclusive_scan(local, warp_tot, &total);
    for (int b = b0; b < b1; ++b) {
        const int L = max(seqlens[b], 0);
        const long long n = ((long long)L + kPage - 1) / kPage;
        E[b] = (int32_t)(off >> kPackShift);
        C[b] = (off & kMask) + (long long)c * E[b];
        off += n + (n > 0 ? (1ll << kPackShift) : 0);
    }
    const long long W = (total & kMask) + (long long)c * (total >> kPackShift);
    if (tid == 0) { E[batch] = (int32_t)(total >> kPackShift); C[batch] = W; }
    __syncthreads();
    const long long Tl = (W + (long long)(parts - 1) * c + parts - 1) / parts;
    const long long T = Tl < 1 ? 1 : Tl;

    // ---- part boundaries: warp 0
    if (tid < 32) {
        int p = 0, cb = 0;             // part p starts in sequence cb, at cost position g0
        long long g0 = 0;
        bool window_first = false;
        if (lane == 0) { pb[0] = 0; pk[0] = 0; }
        while (p < parts - 1 && cb < batch) {
            if (window_first) {
                // part p alone, its stop sequence searched among cb .. cb + 31
                const int j = cb + lane;
                const long long cj1 = j < batch ? C[j + 1] : 0;
                const unsigned mask = __ballot_sync(0xffffffffu, j < batch && cj1 >= g0 + T);
                if (mask == 0 && cb + 32 < batch) { window_first = false; continue; }
                int eb = batch, ek = 0;
                long long eg = W;
                bool snap = true;      // no stop: the part takes everything left
                if (mask) {
                    const int i = __ffs(mask) - 1;
                    part_end(g0, T, c, j, j < batch ? C[j] : 0, cj1, eb, ek, eg, snap);
                    eb = __shfl_sync(0xffffffffu, eb, i);
                    ek = __shfl_sync(0xffffffffu, ek, i);
                    eg = __shfl_sync(0xffffffffu, eg, i);
                    snap = __shfl_sync(0xffffffffu, snap, i);
                }
                if (lane == 0) { pb[p + 1] = eb; pk[p + 1] = ek; }
                ++p;
                cb = eb;
                g0 = eg;
                window_first = snap;
                continue;
            }
            // a round: lane m takes part p + m (parts p .. parts - 2 are walked; the last takes the rest)
            const int lim = parts - 1 - p;
            const long long g = g0 + (long long)lane * (T - c);
            int lo = cb + 1, hi = batch + 1;   // first i with C[i] >= g + T; the stop sequence is i - 1
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (C[mid] >= g + T) hi = mid; else lo = mid + 1;
            }
            // the part's end, computed by every lane (no divergent branch around the loads):
            // a lane whose part takes everything left keeps the end (batch, 0)
            const bool stops = lo <= batch;
            const int j = stops ? lo - 1 : batch - 1;   // cb < batch, so batch >= 1
            int eb, ek;
            long long eg;
            bool snap;
            part_end(g, T, c, j, C[j], C[j + 1], eb, ek, eg, snap);
            if (!stops) { eb = batch; ek = 0; eg = W; snap = true; }
            const unsigned mask = __ballot_sync(0xffffffffu, lane < lim && snap);
            const int last = mask ? __ffs(mask) - 1 : min(31, lim - 1);
            if (lane <= last) { pb[p + lane + 1] = eb; pk[p + lane + 1] = ek; }
            cb = __shfl_sync(0xffffffffu, eb, last);
            g0 = __shfl_sync(0xffffffffu, eg, last);
            p += last + 1;
            window_first = last == 0;
        }
        // after the walk: the last part, or every part once the sequences ran out, ends at (batch, 0)
        for (int q = p + 1 + lane; q <= parts; q += 32) { pb[q] = batch; pk[q] = 0; }
    }
    __syncthreads();
    for (int q = tid; q <= parts; q += kThreadsMd) gs[q] = pre(pb[q]) + pk[q];
    __syncthreads();

    // ---- split counts per sequence and num_splits (exclusive prefix sum)
    auto gs_at = [&](int i) -> long long { return gs[i]; };
    auto splits_of = [&](int b) -> int {
        const long long first = pre(b), end = pre(b + 1);
        return end > first ? last_le(parts, end - 1, gs_at) - last_le(parts, first, gs_at) + 1 : 0;
    };
    long long cnt_local = 0;
    for (int b = b0; b < b1; ++b) cnt_local += splits_of(b);
    long long total_splits = 0;
    long long soff = block_exclusive_scan(cnt_local, warp_tot, &total_splits);
    for (int b = b0; b < b1; ++b) {
        num_splits[b] = (int32_t)soff;
        soff += splits_of(b);
    }
    if (tid == 0) num_splits[batch] = (int32_t)total_splits;
    __syncthreads();   // num_splits visible to the whole block (global memory, same CTA)

    // ---- records
    for (int q = tid; q < parts; q += kThreadsMd) {
        const long long blocks = gs[q + 1] - gs[q];
        int first_slot = 0;
        if (blocks > 0) {
            // sequence of the part's first block (the last sequence whose first block is <= it is non-empty)
            const int f = last_le(batch + 1, gs[q], pre);
            first_slot = num_splits[f] + (q - last_le(parts, pre(f), gs_at));
        }
        int32_t *rec = md + (int64_t)q * kMdSize;
        rec[0] = pb[q]; rec[1] = pk[q]; rec[2] = pb[q + 1]; rec[3] = pk[q + 1];
        rec[4] = first_slot; rec[5] = (int32_t)blocks; rec[6] = 0; rec[7] = 0;
    }
}

// Dynamic shared memory of mla_metadata_kernel.
size_t metadata_smem_bytes(int batch, int parts) {
    return (size_t)(batch + 1 + parts + 1) * sizeof(long long) + (size_t)(batch + 1 + 2 * (parts + 1)) * sizeof(int32_t);
}

}  // namespace mla
