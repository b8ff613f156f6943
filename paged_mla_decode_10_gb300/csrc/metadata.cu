// metadata.cu -- split-KV schedule (get_mla_metadata) on the device.
//
// Output shapes follow the FlashMLA-PyTorch page (flash_mla_interface.py,
// get_mla_metadata docstring): tile_scheduler_metadata (num_sm_parts,
// TileSchedulerMetaDataSize) int32 and num_splits (batch_size + 1) int32.
// The record and policy are this library's:
//
//   record of part p: [begin_b, begin_blk, end_b, end_blk, first_slot, num_blocks, 0, 0]
//   n_b = ceil(max(L_b, 0) / 64); c = 6 (cost of opening a segment, in blocks)
//   W = sum_{n_b > 0} (n_b + c);  T = max(1, ceil((W + (parts - 1) c) / parts))
//   parts walk the (b, blk) sequence in order; a part stops opening segments
//   when T - load - c <= 0, takes min(remaining, T - load - c) blocks when it
//   opens one, and the last part takes the rest.
//   num_splits = exclusive prefix sum of the per-sequence segment counts;
//   first_slot = num_splits[b] + (number of earlier parts that touched b)
//   for the part's first sequence b.
//
// One CTA: the per-sequence block counts and W are computed in parallel, the
// walk itself (O(batch + parts) steps) by one thread from shared memory.
#include <cuda_runtime.h>
#include <cstdint>

#include "decode_common.cuh"

namespace mla {

__global__ void __launch_bounds__(256) mla_metadata_kernel(const int32_t *__restrict__ seqlens, int batch,
                                                           int parts, int32_t *__restrict__ md,
                                                           int32_t *__restrict__ num_splits) {
    extern __shared__ int32_t sm[];
    int32_t *nb = sm;            // blocks per sequence
    int32_t *cnt = sm + batch;   // segments per sequence
    __shared__ unsigned long long w_total;
    if (threadIdx.x == 0) w_total = 0ull;
    __syncthreads();
    unsigned long long w = 0ull;
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        int L = seqlens[b];
        L = L < 0 ? 0 : L;
        const int n = (L + kPage - 1) / kPage;
        nb[b] = n;
        cnt[b] = 0;
        if (n > 0) w += (unsigned long long)(n + kFixedCost);
    }
    atomicAdd(&w_total, w);
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long W = (long long)w_total;
        long long Tl = (W + (long long)(parts - 1) * kFixedCost + parts - 1) / parts;
        const int T = Tl < 1 ? 1 : (int)Tl;
        int b = 0, k = 0;
        for (int p = 0; p < parts; ++p) {
            const int begin_b = b, begin_k = k;
            const bool last = p == parts - 1;
            int load = 0, total = 0, first_b = -1, first_idx = 0;
            while (b < batch) {
                const int n = nb[b];
                if (n == 0) { ++b; k = 0; continue; }
                const int rem = n - k;
                int take;
                if (last) {
                    take = rem;
                } else {
                    const int avail = T - load - kFixedCost;
                    if (avail <= 0) break;
                    take = rem < avail ? rem : avail;
                }
                if (first_b < 0) { first_b = b; first_idx = cnt[b]; }
                cnt[b] += 1;
                load += kFixedCost + take;
                total += take;
                k += take;
                if (k == n) { ++b; k = 0; }
                if (!last && load >= T) break;
            }
            int32_t *rec = md + (int64_t)p * kMdSize;
            rec[0] = begin_b; rec[1] = begin_k; rec[2] = b; rec[3] = k;
            rec[4] = first_b;        // resolved to a slot below
            rec[5] = total;
            rec[6] = first_idx;      // cleared below
            rec[7] = 0;
        }
        int acc = 0;
        for (int i = 0; i < batch; ++i) { num_splits[i] = acc; acc += cnt[i]; }
        num_splits[batch] = acc;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < parts; p += blockDim.x) {
        int32_t *rec = md + (int64_t)p * kMdSize;
        const int fb = rec[4];
        rec[4] = fb >= 0 ? num_splits[fb] + rec[6] : 0;
        rec[6] = 0;
    }
}

}  // namespace mla
