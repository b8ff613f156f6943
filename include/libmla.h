/*
 * libmla.h -- C ABI of libmla: Multi-head Latent Attention (MLA) decode over
 * a paged latent KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The two operations follow the interface on the FlashMLA-PyTorch page
 * (flash_mla_interface.py: get_mla_metadata and flash_mla_with_kvcache) and
 * the vLLM page "vllm.attention.ops.flashmla" (same functions, parameter
 * and return tables):
 *
 *   mla_get_metadata  -- split-KV load-balancing schedule over the SMs
 *                        (get_mla_metadata: tile_scheduler_metadata of shape
 *                        (num_sm_parts, TileSchedulerMetaDataSize) and
 *                        num_splits of shape (batch_size + 1), both int32)
 *   mla_decode_fwd    -- the decode (flash_mla_with_kvcache / fwd_kvcache_mla):
 *                        out (batch, s_q, h_q, head_dim_v) and the fp32
 *                        softmax_lse (batch, h_q, s_q)
 *
 * Conventions shared by every call
 *   - Every tensor argument is a plain pointer owned by the caller (device
 *     memory, except the host buffers of mla_decode_fwd_host); libmla keeps
 *     no reference to it after the call returns.  libmla allocates device
 *     memory only for calls that pass no workspace and for
 *     mla_decode_fwd_host (stream-ordered, released by mla_shutdown).
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and runs asynchronously; no call synchronizes the host
 *     except mla_check_device_error.
 *   - Every call returns an int status (MLA_OK or one of MLA_ERR_*); the
 *     detail of the last failure on the calling thread is available from
 *     mla_last_error().  A failing call enqueues nothing.
 *   - Layouts use element strides; the last dimension of every tensor must
 *     be contiguous.  bf16 tensors are IEEE bfloat16 bit patterns.
 *
 * The workspace convention (query the size, then pass caller-owned scratch)
 * mirrors the two-phase C API on the Ascend ATB "MLA" page
 * (AtbMLAGetWorkspaceSize, then AtbMLA).
 */
#ifndef LIBMLA_H
#define LIBMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mla_stream_t; /* same handle as cudaStream_t */

/* Status codes. */
enum {
    MLA_OK = 0,
    MLA_ERR_ARG = 1,         /* invalid argument: shape, stride, alignment or NULL pointer   */
    MLA_ERR_UNSUPPORTED = 2, /* valid request outside what libmla implements (see each call) */
    MLA_ERR_ARCH = 3,        /* current device is not compute capability 10.3 (sm_103)       */
    MLA_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed                          */
    MLA_ERR_WORKSPACE = 5,   /* workspace pointer NULL or smaller than mla_workspace_size     */
    MLA_ERR_DEVICE = 6       /* a kernel reported an error (see mla_check_device_error)       */
};

/* Device-side error bits, reported by mla_check_device_error. */
enum {
    MLA_DEVERR_TIMEOUT = 1,     /* a bounded wait inside a kernel gave up; outputs are invalid */
    MLA_DEVERR_BAD_BLOCK = 2    /* a needed block_table entry was outside [0, num_blocks)       */
};

/* int32 entries per tile_scheduler_metadata row (TileSchedulerMetaDataSize). */
#define MLA_METADATA_SIZE 8

/* Fixed dimensions of the MLA decode this library implements. */
#define MLA_HEAD_DIM 576        /* 512 latent + 64 RoPE dims of q and of each cache row */
#define MLA_HEAD_DIM_V 512      /* V = the first 512 dims of each cache row             */
#define MLA_PAGE_BLOCK_SIZE 64  /* cache rows per physical block                        */

/*
 * Problem description for mla_decode_fwd / mla_workspace_size.
 *
 *   q            (batch, s_q, h_q, head_dim) bf16;        q_stride   = {batch, token, head}
 *   k_cache      (num_blocks, page_block_size, h_k, head_dim) bf16;
 *                                                          k_stride   = {block, row, kv-head}
 *   block_table  (batch, max_blocks_per_seq) int32;        bt_stride  = elements per row
 *   out          (batch, s_q, h_q, head_dim_v) bf16;       out_stride = {batch, token, head}
 *   softmax_lse  (batch, h_q, s_q) fp32, contiguous.
 *
 * Requirements (else MLA_ERR_ARG): batch >= 0, s_q >= 1, h_k >= 1,
 * h_q % h_k == 0, head_dim == 576, head_dim_v == 512, page_block_size == 64,
 * num_blocks >= 1, max_blocks_per_seq >= 1, num_sm_parts >= 1; every stride a
 * multiple of 8 elements and every bf16 base pointer 16-byte aligned.
 * Limits (else MLA_ERR_UNSUPPORTED): s_q * h_q / h_k <= 1024 query rows per
 * KV head; batch <= 65535.
 */
typedef struct {
    int32_t batch;
    int32_t s_q;
    int32_t h_q;
    int32_t h_k;
    int32_t head_dim;
    int32_t head_dim_v;
    int32_t page_block_size;
    int32_t num_blocks;
    int32_t max_blocks_per_seq;
    int32_t num_sm_parts;      /* rows of tile_scheduler_metadata */
    int64_t q_stride[3];
    int64_t k_stride[3];
    int64_t bt_stride;
    int64_t out_stride[3];
} mla_shape_t;

/*
 * Number of scheduler parts (rows of tile_scheduler_metadata) that fill
 * `device` for the given head configuration: the number of two-CTA clusters
 * of the decode kernel that can be resident at once, divided by the number
 * of 128-row blocks per KV head and by num_heads_k (at least 1).
 * num_heads_per_head_k = s_q * h_q / h_k (vLLM page, get_mla_metadata
 * parameter table).  Errors: MLA_ERR_ARG (non-positive argument),
 * MLA_ERR_ARCH, MLA_ERR_CUDA.
 */
int mla_get_num_sm_parts(int device, int num_heads_per_head_k, int num_heads_k, int *num_sm_parts);

/*
 * Split-KV schedule (get_mla_metadata).  Reads cache_seqlens (device, int32,
 * `batch` entries) on the device and writes
 *   tile_scheduler_metadata  (num_sm_parts, MLA_METADATA_SIZE) int32, device
 *   num_splits               (batch + 1) int32, device: exclusive prefix sum
 *                            of the number of parts each sequence is split over
 * Record of part p: [begin_b, begin_blk, end_b, end_blk, first_slot,
 * num_blocks, 0, 0]; the part processes, for b in [begin_b, end_b], blocks
 * [b == begin_b ? begin_blk : 0, b == end_b ? end_blk : ceil(L_b / 64)).
 * Policy: greedy contiguous walk over (sequence, block) with a fixed cost of
 * c blocks per segment and a per-part target of
 * ceil((W + (num_sm_parts - 1) * c) / num_sm_parts), W = sum(n_b + c), where
 * c (the decode kernel's fixed work per segment in page times) is 6 for
 * num_heads_per_head_k >= 64 and 4 below, for a bf16 cache.
 * Errors: MLA_ERR_ARG (NULL pointer, batch < 0, num_sm_parts < 1,
 * num_heads_per_head_k < 1, num_heads_k < 1), MLA_ERR_UNSUPPORTED
 * (batch > 16384 or num_sm_parts > 1024), MLA_ERR_CUDA.
 */
int mla_get_metadata(const int32_t *cache_seqlens, int batch, int num_heads_per_head_k,
                     int num_heads_k, int num_sm_parts, int32_t *tile_scheduler_metadata,
                     int32_t *num_splits, mla_stream_t stream);

/*
 * mla_get_metadata for a cache of kv_bytes-byte elements (2: bf16, 1: e4m3,
 * for mla_decode_fwd_fp8): the segment cost c is one block more for e4m3,
 * whose pages take less time against the same fixed work.  Any schedule is
 * valid for either call; this one balances the parts for that cache.
 * Errors: as mla_get_metadata, and MLA_ERR_ARG for kv_bytes other than 1 or 2.
 */
int mla_get_metadata_ex(const int32_t *cache_seqlens, int batch, int num_heads_per_head_k,
                        int num_heads_k, int kv_bytes, int num_sm_parts, int32_t *tile_scheduler_metadata,
                        int32_t *num_splits, mla_stream_t stream);

/*
 * Bytes of workspace mla_decode_fwd needs for `shape`: fp32 partial outputs
 * and log-sum-exps of the sequences the schedule splits, for up to
 * batch + num_sm_parts splits.  Errors: MLA_ERR_ARG.
 */
int mla_workspace_size(const mla_shape_t *shape, size_t *bytes);

/*
 * Paged MLA decode (flash_mla_with_kvcache / fwd_kvcache_mla).  For every
 * sequence b, query token i < s_q and head h, with hk = h / (h_q / h_k),
 * L = cache_seqlens[b] and n = causal ? L - s_q + 1 + i : L (clamped to
 * [0, L]; bottom-right alignment):
 *   s_t = softmax_scale * q[b,i,h,:] . k[t, hk, :]       t < n, all 576 dims
 *   out[b,i,h,:]      = sum_t softmax(s)_t * k[t, hk, 0:512]   (V aliases K)
 *   softmax_lse[b,h,i] = ln sum_t exp(s_t)
 * where k[t] is row t % 64 of physical block block_table[b][t / 64].
 * Rows with n == 0 get out = 0 and softmax_lse = -inf.
 * softmax_scale <= 0 or NaN selects the default 1/sqrt(head_dim) (the
 * interface's default of q.shape[-1] ** -0.5).
 *
 * tile_scheduler_metadata / num_splits must come from mla_get_metadata on
 * the same cache_seqlens and num_sm_parts (not checked).  block_table
 * entries past ceil(L / 64) are never read; needed entries outside
 * [0, num_blocks) are not dereferenced and raise MLA_DEVERR_BAD_BLOCK.
 * workspace: device scratch of at least mla_workspace_size bytes, 256-byte
 * aligned, not used concurrently by another call.  workspace == NULL with
 * workspace_bytes == 0 selects the library's own stream-ordered workspace:
 * one buffer per (device, stream), allocated and grown with cudaMallocAsync
 * on `stream` (calls on one stream share it; calls on different streams get
 * different buffers) and released by mla_shutdown (the workspace
 * convention of the FlashMLA-PyTorch / vLLM pages leaves the scratch to the
 * library; the Ascend ATB page's size query plus caller buffer is the
 * explicit form).
 * Errors: MLA_ERR_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_ARCH, MLA_ERR_WORKSPACE,
 * MLA_ERR_CUDA.  Launches two kernels: mla_decode_splitkv then
 * mla_decode_combine, with the same arguments.
 */
int mla_decode_fwd(const mla_shape_t *shape, const void *q, const void *k_cache,
                   const int32_t *block_table, const int32_t *cache_seqlens,
                   const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                   float softmax_scale, int causal, void *out, float *softmax_lse,
                   void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * The first of the two launches of mla_decode_fwd: the persistent split-KV
 * decode.  Sequences the schedule does not split are finished here (out and
 * softmax_lse written); split ones leave fp32 partials in the workspace.
 */
int mla_decode_splitkv(const mla_shape_t *shape, const void *q, const void *k_cache,
                       const int32_t *block_table, const int32_t *cache_seqlens,
                       const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                       float softmax_scale, int causal, void *out, float *softmax_lse,
                       void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * The second launch of mla_decode_fwd: merges the partials of every split
 * sequence by log-sum-exp weighting (lse = ln sum_s exp(lse_s),
 * out = sum_s exp(lse_s - lse) * out_s) and writes out / softmax_lse for
 * them, and out = 0, softmax_lse = -inf for empty sequences.
 * Same arguments as mla_decode_fwd (q, k_cache and block_table unused).
 */
int mla_decode_combine(const mla_shape_t *shape, const void *q, const void *k_cache,
                       const int32_t *block_table, const int32_t *cache_seqlens,
                       const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                       float softmax_scale, int causal, void *out, float *softmax_lse,
                       void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * Size of the scratch built into the library for mla_decode_fwd_noalloc:
 * 64 MiB of device memory on every GPU that loads the library, held until
 * the process exits.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * mla_decode_fwd without a workspace argument, for callers that cannot
 * allocate device memory themselves: code whose device memory is owned by
 * another allocator (an inference server's pool, say) or a latency-critical
 * loop that cannot afford the device-wide synchronisation cudaMalloc or
 * cudaFree may cause.  The split partials go to a scratch array built into
 * the library (MLA_NOALLOC_SCRATCH_BYTES); this call allocates nothing.
 * The pages this library follows have no counterpart of this call.
 *
 * Arguments, results and errors as mla_decode_fwd, plus MLA_ERR_UNSUPPORTED
 * (with a message giving both sizes) when mla_workspace_size(shape) exceeds
 * MLA_NOALLOC_SCRATCH_BYTES.  The first call on a device looks up the
 * scratch's device address with that device current; make it before any
 * stream capture (and again after mla_shutdown, which forgets it).  All calls share the one scratch array: calls whose
 * kernels may overlap on the GPU (unordered streams) race on it and must not
 * be issued.  Nothing in the scratch needs clearing between calls.
 */
int mla_decode_fwd_noalloc(const mla_shape_t *shape, const void *q, const void *k_cache,
                           const int32_t *block_table, const int32_t *cache_seqlens,
                           const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                           float softmax_scale, int causal, void *out, float *softmax_lse,
                           mla_stream_t stream);

/*
 * Strides (elements) of the RoPE tensors of mla_decode_fwd_split.
 */
typedef struct {
    int64_t q_rope_stride[3];   /* q_rope (batch, s_q, h_q, 64): {batch, token, head}            */
    int64_t krope_stride[3];    /* krope (num_blocks, 64, h_k, 64): {block, row, kv-head}          */
} mla_rope_strides_t;

/*
 * mla_decode_fwd on split inputs: the latent and RoPE parts of the query and
 * of the cache in separate tensors, the layout of the Ascend ATB MLA page
 * (parameter table: qNope, qRope, ctKV, kRope; cacheMode 1, separate
 * caches).  The result is that of mla_decode_fwd on the concatenations
 * q = [q_nope | q_rope] and k_cache = [ctkv | krope] along the last
 * dimension; V is ctkv.
 *   q_nope  (batch, s_q, h_q, 512) bf16   strides shape->q_stride
 *   q_rope  (batch, s_q, h_q, 64) bf16    strides rope->q_rope_stride
 *   ctkv    (num_blocks, 64, h_k, 512) bf16  strides shape->k_stride
 *   krope   (num_blocks, 64, h_k, 64) bf16   strides rope->krope_stride
 * shape->head_dim stays 576 (the logical q . k length).  Every pointer
 * 16-byte aligned, every stride a positive multiple of 8 elements, head
 * strides at least the head's dims.  Everything else (schedule, workspace,
 * errors, the two launches) as mla_decode_fwd.  Both calls read the same
 * bytes from HBM for the same problem.
 */
int mla_decode_fwd_split(const mla_shape_t *shape, const mla_rope_strides_t *rope,
                         const void *q_nope, const void *q_rope, const void *ctkv, const void *krope,
                         const int32_t *block_table, const int32_t *cache_seqlens,
                         const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                         float softmax_scale, int causal, void *out, float *softmax_lse,
                         void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_decode_fwd over an e4m3 (FP8, 1 sign, 4 exponent, 3 mantissa bits)
 * query and latent cache, with the two fused product scales of the FlashInfer
 * page (trtllm_batch_decode_with_kv_cache_mla, the note on bmm1_scale and
 * bmm2_scale):
 *   s_t = bmm1_scale * sum_{d < 576} q[d] * k[t][d]
 *   out = bmm2_scale * sum_t softmax(s)_t * k[t][0:512]      (bf16)
 *   softmax_lse = ln sum_t exp(s_t)                           (fp32)
 * with q and k the e4m3 values as stored.  bmm1_scale folds the query and key
 * dequantisation scales into the softmax scale; bmm2_scale is the value
 * dequantisation scale.
 *   q        (batch, s_q, h_q, 576) e4m3 bytes      strides shape->q_stride (elements = bytes)
 *   k_cache  (num_blocks, 64, h_k, 576) e4m3 bytes  strides shape->k_stride
 *   out      (batch, s_q, h_q, 512) bf16, softmax_lse (batch, h_q, s_q) fp32, as mla_decode_fwd
 * Masking, schedule (mla_get_metadata), workspace (NULL = internal) and the
 * two launches are those of mla_decode_fwd.
 *
 * Accuracy.  The probabilities are rounded to e4m3 for the PV product (the
 * denominator sums them unrounded): each weight errs by up to 2^-4 of itself.
 * With more than 32 query rows per KV head the two halves of each logit,
 * s_0 and s_1 (latent dims 0-255 + RoPE dims 512-543, and the rest), are
 * rounded to bf16 before they are added, which moves a logit by at most
 * bmm1_scale * 2^-8 * (|s_0| + |s_1|) and softmax_lse by at most the
 * probability-weighted mean of those moves.
 *
 * Errors: as mla_decode_fwd, and MLA_ERR_ARG when bmm1_scale is not positive
 * and finite, bmm2_scale not finite, or a q / k_cache stride is not a
 * multiple of 16 bytes.
 */
int mla_decode_fwd_fp8(const mla_shape_t *shape, const void *q, const void *k_cache,
                       const int32_t *block_table, const int32_t *cache_seqlens,
                       const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                       float bmm1_scale, float bmm2_scale, int causal, void *out, float *softmax_lse,
                       void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * The first of the two launches of mla_decode_fwd_fp8 (the e4m3 split-KV
 * decode), with its arguments; the second is mla_decode_combine on the same
 * workspace, which merges split sequences exactly as for bf16 inputs (the
 * partials already carry bmm2_scale).  A NULL workspace selects the same
 * internal one for both calls on one stream.
 */
int mla_decode_splitkv_fp8(const mla_shape_t *shape, const void *q, const void *k_cache,
                           const int32_t *block_table, const int32_t *cache_seqlens,
                           const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                           float bmm1_scale, float bmm2_scale, int causal, void *out, float *softmax_lse,
                           void *workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * One whole decode step from host buffers: copies q, block_table and
 * cache_seqlens to the device, computes the schedule (mla_get_metadata with
 * shape->num_sm_parts parts), decodes (mla_decode_fwd) and returns out and
 * softmax_lse to host memory, all enqueued on `stream` -- the sequence of the
 * FlashMLA-PyTorch page's usage (get_mla_metadata from cache_seqlens, then
 * flash_mla_with_kvcache) with the host transfers around it.  The results are in
 * the host buffers once `stream` has completed; the inputs must stay
 * unchanged until then.
 *   q_host              host, bf16, laid out by shape->q_stride
 *   block_table_host    host, int32, row stride shape->bt_stride
 *   cache_seqlens_host  host, int32, batch entries
 *   k_cache             DEVICE (the cache stays resident), as mla_decode_fwd
 *   out_host            host, bf16 (batch, s_q, h_q, 512), contiguous:
 *                       shape->out_stride must be {s_q*h_q*512, h_q*512, 512}
 *   softmax_lse_host    host, fp32 (batch, h_q, s_q), contiguous
 * Host buffers should be page-locked (cudaHostAlloc, cudaHostRegister) for
 * the copies to be asynchronous; pageable memory works, with copies that
 * block the host.  When out_host / softmax_lse_host are page-locked and
 * mapped into the device's address space, the kernels store the results
 * there directly and no device-to-host copy is made; otherwise they are
 * staged in device memory and copied back.  The schedule runs on a second,
 * library-owned stream while q is copied, and `stream` waits for it before
 * the decode, so work enqueued on `stream` afterwards is ordered after the
 * whole step.
 * Device staging (inputs, schedule, workspace, output staging) is one
 * buffer per (device, stream), allocated and grown with cudaMallocAsync on
 * `stream`, and released, with the second stream, by mla_shutdown.
 * batch == 0 enqueues nothing (the pointers may then be NULL).
 * Errors: as mla_decode_fwd and mla_get_metadata (MLA_ERR_UNSUPPORTED for
 * batch > 16384 or num_sm_parts > 1024), plus MLA_ERR_ARG for a
 * non-contiguous out.  A CUDA failure after the first copy was enqueued
 * returns MLA_ERR_CUDA with part of the step enqueued.
 */
int mla_decode_fwd_host(const mla_shape_t *shape, const void *q_host, const void *k_cache,
                        const int32_t *block_table_host, const int32_t *cache_seqlens_host,
                        float softmax_scale, int causal, void *out_host, float *softmax_lse_host,
                        mla_stream_t stream);

/*
 * Releases the internal workspaces that calls without a workspace allocated
 * and the staging buffers and streams of mla_decode_fwd_host (synchronizing
 * each device that holds one first).  Later such calls
 * allocate again.  It also forgets what the library set up per device
 * (kernel attributes, the device addresses of its error word and of the
 * built-in scratch of mla_decode_fwd_noalloc, cache tensor maps), which the
 * next call on each device sets up again: call it before resetting a device
 * (cudaDeviceReset), since the reset may reload the library's module at
 * other addresses.  Not to be called while another thread uses the library.
 * Errors: MLA_ERR_CUDA.
 */
int mla_shutdown(void);

/*
 * Synchronizes the current device, then stores in *bits the OR of the
 * MLA_DEVERR_* bits kernels of this library raised on it since the last
 * clear, and clears them when `clear` is non-zero.  Returns MLA_OK, or
 * MLA_ERR_CUDA when synchronization itself failed.
 */
int mla_check_device_error(int *bits, int clear);

/* Static description of a status code. */
const char *mla_status_string(int status);

/* Detail message of the last failing call on the calling thread ("" if none). */
const char *mla_last_error(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBMLA_H */
