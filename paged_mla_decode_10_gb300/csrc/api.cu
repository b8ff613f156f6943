// api.cu -- the C ABI of libmla (declared in include/libmla.h): argument
// validation, TMA descriptor encoding, and the kernel launches.
#include <cuda_runtime.h>
#include <cuda.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "libmla.h"
#include "decode_common.cuh"

namespace mla {
__global__ void mla_splitkv_kernel(const __grid_constant__ CUtensorMap km128, const __grid_constant__ CUtensorMap km64,
                                   const __grid_constant__ CUtensorMap kq, const __grid_constant__ CUtensorMap kqr,
                                   const __grid_constant__ DecodeParams p);
__global__ void mla_splitkv_kernel_f8(const __grid_constant__ CUtensorMap km128,
                                      const __grid_constant__ CUtensorMap km64, const __grid_constant__ CUtensorMap kq,
                                      const __grid_constant__ CUtensorMap kqr, const __grid_constant__ DecodeParams p);
__global__ void mla_combine_kernel(const __grid_constant__ DecodeParams p);
__global__ void mla_metadata_kernel(const int32_t *seqlens, int batch, int parts, int cost, int32_t *md,
                                    int32_t *num_splits);
size_t metadata_smem_bytes(int batch, int parts);
uint32_t splitkv_smem_bytes();
uint32_t splitkv_f8_smem_bytes();
uint32_t splitkv_threads();
uint32_t combine_threads();
uint32_t combine_rows_per_block();
void noalloc_forget_devices();
}  // namespace mla

// Error bits raised by the kernels on this device (MLA_DEVERR_*).
__device__ int g_mla_device_error = 0;

namespace {

using namespace mla;

constexpr int kMaxDevices = 64;
constexpr int kMaxBatchMetadata = 16384;
constexpr int kMaxPartsMetadata = 1024;
constexpr int kMaxRowsPerHead = 1024;

thread_local std::string t_last_error;

int fail(int status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceState {
    bool ready = false;
    int status = MLA_OK;
    int sm_count = 0;
    int max_clusters = 0;
    int *err_word = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Per-device one-time setup (with that device current): architecture check,
// kernel attributes, occupancy of the cluster kernel, device error word.
int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3) {
            st.ready = true;
            st.status = MLA_ERR_ARCH;
        } else {
            const int smem = (int)splitkv_smem_bytes();
            if ((e = cudaFuncSetAttribute(mla_splitkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
                cudaSuccess)
                return cuda_fail(e, "cudaFuncSetAttribute(splitkv)");
            if ((e = cudaFuncSetAttribute(mla_splitkv_kernel_f8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)splitkv_f8_smem_bytes())) != cudaSuccess)
                return cuda_fail(e, "cudaFuncSetAttribute(splitkv e4m3)");
            if ((e = cudaFuncSetAttribute(mla_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)metadata_smem_bytes(kMaxBatchMetadata, kMaxPartsMetadata))) != cudaSuccess)
                return cuda_fail(e, "cudaFuncSetAttribute(metadata)");
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * 64, 1, 1);
            cfg.blockDim = dim3(splitkv_threads(), 1, 1);
            cfg.dynamicSmemBytes = smem;
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, (void *)mla_splitkv_kernel, &cfg);
            if (e != cudaSuccess || clusters <= 0) {
                (void)cudaGetLastError();
                clusters = st.sm_count / 2;
            }
            st.max_clusters = clusters;
            void *addr = nullptr;
            if ((e = cudaGetSymbolAddress(&addr, g_mla_device_error)) != cudaSuccess)
                return cuda_fail(e, "cudaGetSymbolAddress(error word)");
            st.err_word = static_cast<int *>(addr);
            st.ready = true;
            st.status = MLA_OK;
        }
    }
    if (st.status != MLA_OK)
        return fail(st.status, "device %d is not compute capability 10.3 (sm_103)", dev);
    *out = &st;
    return MLA_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors over k_cache, cached per (pointer, geometry)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Where the cache rows come from: the latent dims (TMA boxes of 128-byte rows:
// 64 bf16 or 128 e4m3 dims) and the RoPE dims (a box of 32), either one
// tensor of 576-dim rows or two tensors (512 and 64 dims).  Strides in
// elements: {block, row, kv-head}.
struct KvSource {
    int elem = 2;              // bytes per element: 2 (bf16) or 1 (e4m3)
    const void *latent;
    int64_t lat_stride[3];
    int lat_dims;              // extent of the latent tensor's last dimension (576 or 512)
    const void *rope;          // base of the RoPE tensor (the cache itself when rows are concatenated)
    int64_t rope_stride[3];
    int rope_dims;             // extent of the RoPE tensor's last dimension (576 or 64)
};

// A cache of 576-dim rows: both maps span the whole row; the RoPE boxes start
// at dim 512 (DecodeParams::rope_x0).
KvSource concat_source(const mla_shape_t *sh, const void *k_cache) {
    KvSource k;
    k.latent = k.rope = k_cache;
    for (int i = 0; i < 3; ++i) k.lat_stride[i] = k.rope_stride[i] = sh->k_stride[i];
    k.lat_dims = k.rope_dims = sh->head_dim;
    return k;
}

struct MapEntry {
    KvSource src;
    int device = -1, num_blocks = 0, h_k = 0;
    CUtensorMap m128, m64;
    bool valid = false;
};
constexpr int kMapCache = 16;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

int get_encoder(EncodeTiledFn *fn) {
    static EncodeTiledFn cached = nullptr;
    if (!cached) {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
            return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        cached = reinterpret_cast<EncodeTiledFn>(f);
    }
    *fn = cached;
    return MLA_OK;
}

bool same_source(const KvSource &a, const KvSource &b) {
    return a.elem == b.elem && a.latent == b.latent && a.rope == b.rope && a.lat_dims == b.lat_dims && a.rope_dims == b.rope_dims &&
           !memcmp(a.lat_stride, b.lat_stride, sizeof a.lat_stride) &&
           !memcmp(a.rope_stride, b.rope_stride, sizeof a.rope_stride);
}

// Tensor maps {dims, h_k, 64 rows, num_blocks} over the latent and the RoPE
// dims of the cache, cached per (device, source, geometry).
int kcache_maps(const mla_shape_t *sh, const KvSource &src, CUtensorMap *m128, CUtensorMap *m64) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto &e : g_maps) {
        if (e.valid && e.device == dev && e.num_blocks == sh->num_blocks && e.h_k == sh->h_k && same_source(e.src, src)) {
            *m128 = e.m128;
            *m64 = e.m64;
            return MLA_OK;
        }
    }
    EncodeTiledFn enc;
    int st = get_encoder(&enc);
    if (st != MLA_OK) return st;
    const cuuint64_t gdim_l[4] = {(cuuint64_t)src.lat_dims, (cuuint64_t)sh->h_k, (cuuint64_t)sh->page_block_size,
                                  (cuuint64_t)sh->num_blocks};
    const cuuint64_t gdim_r[4] = {(cuuint64_t)src.rope_dims, (cuuint64_t)sh->h_k, (cuuint64_t)sh->page_block_size,
                                  (cuuint64_t)sh->num_blocks};
    const cuuint64_t eb = (cuuint64_t)src.elem;
    const cuuint64_t gstr_l[3] = {(cuuint64_t)src.lat_stride[2] * eb, (cuuint64_t)src.lat_stride[1] * eb,
                                  (cuuint64_t)src.lat_stride[0] * eb};
    const cuuint64_t gstr_r[3] = {(cuuint64_t)src.rope_stride[2] * eb, (cuuint64_t)src.rope_stride[1] * eb,
                                  (cuuint64_t)src.rope_stride[0] * eb};
    // latent boxes of 128-byte rows (SW128); RoPE boxes of 32 dims: 64-byte rows (SW64) in bf16,
    // 32-byte rows (SW32) in e4m3
    const cuuint32_t box128[4] = {(cuuint32_t)(128 / src.elem), 1, 64, 1}, box64[4] = {32, 1, 64, 1},
                     es[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = src.elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle rsw = src.elem == 1 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
    MapEntry &e = g_maps[g_map_next];
    CUresult r1 = enc(&e.m128, dt, 4, const_cast<void *>(src.latent), gdim_l, gstr_l, box128, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = enc(&e.m64, dt, 4, const_cast<void *>(src.rope), gdim_r, gstr_r, box64, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, rsw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) {
        e.valid = false;
        return fail(MLA_ERR_ARG, "cache tensor map rejected by the driver (codes %d, %d): check alignment/strides",
                    (int)r1, (int)r2);
    }
    e.src = src;
    e.device = dev;
    e.num_blocks = sh->num_blocks;
    e.h_k = sh->h_k;
    e.valid = true;
    g_map_next = (g_map_next + 1) % kMapCache;
    *m128 = e.m128;
    *m64 = e.m64;
    return MLA_OK;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const mla_shape_t *sh) {
    if (!sh) return fail(MLA_ERR_ARG, "shape is NULL");
    if (sh->batch < 0) return fail(MLA_ERR_ARG, "batch %d < 0", sh->batch);
    if (sh->s_q < 1 || sh->h_q < 1 || sh->h_k < 1)
        return fail(MLA_ERR_ARG, "s_q, h_q, h_k must be >= 1 (got %d, %d, %d)", sh->s_q, sh->h_q, sh->h_k);
    if (sh->h_q % sh->h_k != 0) return fail(MLA_ERR_ARG, "h_q %d not divisible by h_k %d", sh->h_q, sh->h_k);
    if (sh->head_dim != MLA_HEAD_DIM) return fail(MLA_ERR_ARG, "head_dim must be 576 (got %d)", sh->head_dim);
    if (sh->head_dim_v != MLA_HEAD_DIM_V)
        return fail(MLA_ERR_ARG, "head_dim_v must be 512 (got %d)", sh->head_dim_v);
    if (sh->page_block_size != MLA_PAGE_BLOCK_SIZE)
        return fail(MLA_ERR_ARG, "page_block_size must be 64 (got %d)", sh->page_block_size);
    if (sh->num_blocks < 1 || sh->max_blocks_per_seq < 1)
        return fail(MLA_ERR_ARG, "num_blocks and max_blocks_per_seq must be >= 1");
    if (sh->num_sm_parts < 1) return fail(MLA_ERR_ARG, "num_sm_parts must be >= 1");
    const long long rows = (long long)sh->s_q * sh->h_q / sh->h_k;
    if (sh->batch > 65535) return fail(MLA_ERR_UNSUPPORTED, "batch %d exceeds 65535", sh->batch);
    if (rows > kMaxRowsPerHead)
        return fail(MLA_ERR_UNSUPPORTED, "s_q*h_q/h_k = %lld query rows per KV head exceeds %d", rows, kMaxRowsPerHead);
    for (int i = 0; i < 3; ++i) {
        if (sh->q_stride[i] <= 0 || sh->q_stride[i] % 8 || sh->k_stride[i] <= 0 || sh->k_stride[i] % 8 ||
            sh->out_stride[i] <= 0 || sh->out_stride[i] % 8)
            return fail(MLA_ERR_ARG, "strides must be positive multiples of 8 elements");
    }
    if (sh->bt_stride < sh->max_blocks_per_seq) return fail(MLA_ERR_ARG, "bt_stride < max_blocks_per_seq");
    return MLA_OK;
}

size_t workspace_bytes_for(const mla_shape_t *sh, size_t *lse_off) {
    const size_t slots = (size_t)sh->batch + (size_t)sh->num_sm_parts;
    const size_t rows = (size_t)sh->s_q * sh->h_q;        // h_k * R
    const size_t o_bytes = slots * rows * MLA_HEAD_DIM_V * sizeof(float);
    const size_t off = (o_bytes + 255) & ~(size_t)255;
    if (lse_off) *lse_off = off;
    return off + ((slots * rows * sizeof(float) + 255) & ~(size_t)255);
}

// Workspace for calls that pass none: one buffer per (device, stream),
// allocated with cudaMallocAsync on that stream and grown the same way (the
// smaller one released with cudaFreeAsync on the stream, after the work
// already queued there).  Calls on one stream run in order, so they can share
// the buffer; calls on different streams get different buffers.
struct WsEntry {
    int device = -1;
    cudaStream_t stream = nullptr;
    void *ptr = nullptr;
    size_t bytes = 0;
};
constexpr int kWsEntries = 32;
std::mutex g_ws_mu;
WsEntry g_ws[kWsEntries];

int internal_workspace(const mla_shape_t *sh, cudaStream_t stream, void **ws, size_t *ws_bytes) {
    int st = check_shape(sh);
    if (st != MLA_OK) return st;
    const size_t need = workspace_bytes_for(sh, nullptr);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_ws_mu);
    WsEntry *slot = nullptr;
    for (auto &w : g_ws) {
        if (w.ptr && w.device == dev && w.stream == stream) { slot = &w; break; }
        if (!w.ptr && !slot) slot = &w;
    }
    if (!slot) return fail(MLA_ERR_UNSUPPORTED, "more than %d (device, stream) pairs use the internal workspace", kWsEntries);
    if (slot->bytes < need) {
        if (slot->ptr && (e = cudaFreeAsync(slot->ptr, stream)) != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(workspace)");
        slot->ptr = nullptr;
        slot->bytes = 0;
        void *ptr = nullptr;
        if ((e = cudaMallocAsync(&ptr, need, stream)) != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
        slot->ptr = ptr;
        slot->bytes = need;
        slot->device = dev;
        slot->stream = stream;
    }
    *ws = slot->ptr;
    *ws_bytes = slot->bytes;
    return MLA_OK;
}

struct Prepared {
    DecodeParams p;
    dim3 grid;
};

// Argument checks that need no CUDA call.
int check_args(const mla_shape_t *sh, const void *q, const void *k_cache, const int32_t *block_table,
               const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, const void *out,
               const float *lse, bool need_kv) {
    int st = check_shape(sh);
    if (st != MLA_OK) return st;
    if (!cache_seqlens || !md || !num_splits || !out || !lse)
        return fail(MLA_ERR_ARG, "NULL tensor pointer");
    if (need_kv && (!q || !k_cache || !block_table)) return fail(MLA_ERR_ARG, "NULL tensor pointer");
    if ((need_kv && (!aligned16(q) || !aligned16(k_cache))) || !aligned16(out))
        return fail(MLA_ERR_ARG, "q, k_cache and out must be 16-byte aligned");
    return MLA_OK;
}

int prepare(const mla_shape_t *sh, const void *q, const void *k_cache, const int32_t *block_table,
            const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float scale, int causal,
            void *out, float *lse, void *ws, size_t ws_bytes, bool need_kv, Prepared *pr, DeviceState **dst) {
    int st = check_args(sh, q, k_cache, block_table, cache_seqlens, md, num_splits, out, lse, need_kv);
    if (st != MLA_OK) return st;
    size_t lse_off = 0;
    const size_t need = workspace_bytes_for(sh, &lse_off);
    if (!ws) return fail(MLA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(MLA_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (ws_bytes < need) return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
    st = device_state(dst);
    if (st != MLA_OK) return st;

    if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt((float)sh->head_dim);
    DecodeParams &p = pr->p;
    memset(&p, 0, sizeof p);
    p.q = static_cast<const uint16_t *>(q);
    p.q_s0 = sh->q_stride[0]; p.q_s1 = sh->q_stride[1]; p.q_s2 = sh->q_stride[2];
    p.q_rope = q ? p.q + MLA_HEAD_DIM_V : nullptr;   // concatenated q; the split call overrides it
    p.qr_s0 = p.q_s0; p.qr_s1 = p.q_s1; p.qr_s2 = p.q_s2;
    p.q_concat = 1;
    p.rope_x0 = MLA_HEAD_DIM_V;                      // concatenated cache; the split call sets 0
    p.block_table = block_table;
    p.bt_stride = sh->bt_stride;
    p.seqlens = cache_seqlens;
    p.md = md;
    p.num_splits = num_splits;
    p.out = static_cast<uint16_t *>(out);
    p.o_s0 = sh->out_stride[0]; p.o_s1 = sh->out_stride[1]; p.o_s2 = sh->out_stride[2];
    p.lse = lse;
    p.ws_o = static_cast<float *>(ws);
    p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(ws) + lse_off);
    p.err = (*dst)->err_word;
    p.batch = sh->batch; p.s_q = sh->s_q; p.h_q = sh->h_q; p.h_k = sh->h_k;
    p.hpk = sh->h_q / sh->h_k;
    p.rows = sh->s_q * p.hpk;
    p.num_blocks = sh->num_blocks;
    p.max_blocks = sh->max_blocks_per_seq;
    p.num_parts = sh->num_sm_parts;
    p.max_slots = sh->batch + sh->num_sm_parts;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    const int row_blocks = (p.rows + kRowsPerBlock - 1) / kRowsPerBlock;
    pr->grid = dim3(2 * sh->num_sm_parts, row_blocks, sh->h_k);
    return MLA_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors over the query, so that the decode kernel can bring a
// segment's Q through its page ring: {dims, h_q, s_q, batch} maps of the
// latent and of the RoPE dims.  A latent box covers one 128-row block of a KV
// head (q_hb heads x q_tb tokens), a RoPE box 64 rows.  This needs the blocks
// to align with heads and tokens (heads per KV head a multiple or a divisor
// of 128); otherwise, or when the driver rejects a map, the kernel loads Q
// itself (q_tma = 0).  Cached per (device, query geometry).
// ---------------------------------------------------------------------------
struct QMapKey {
    int device = -1, elem = 0, h_q = 0, s_q = 0, batch = 0, hpk = 0, lat_dims = 0, rope_dims = 0;
    const void *lat = nullptr, *rope = nullptr;
    int64_t lat_stride[3] = {0, 0, 0}, rope_stride[3] = {0, 0, 0};
    bool operator==(const QMapKey &o) const {
        return device == o.device && elem == o.elem && h_q == o.h_q && s_q == o.s_q && batch == o.batch &&
               hpk == o.hpk && lat_dims == o.lat_dims && rope_dims == o.rope_dims && lat == o.lat && rope == o.rope &&
               !memcmp(lat_stride, o.lat_stride, sizeof lat_stride) && !memcmp(rope_stride, o.rope_stride, sizeof rope_stride);
    }
};
struct QMapEntry {
    QMapKey key;
    CUtensorMap lat, rope;
    bool ok = false, valid = false;
};
QMapEntry g_qmaps[kMapCache];
int g_qmap_next = 0;

// Fills the query maps and the q_* fields of p; false (p.q_tma = 0) when Q cannot come by TMA.
bool query_maps(const mla_shape_t *sh, int elem, DecodeParams &p, CUtensorMap *lat, CUtensorMap *rope) {
    p.q_tma = 0;
    const int hpk = p.hpk;
    if (!(hpk % kRowsPerBlock == 0 || kRowsPerBlock % hpk == 0) || sh->batch < 1) return false;
    QMapKey k;
    cudaGetDevice(&k.device);
    k.elem = elem;
    k.h_q = sh->h_q; k.s_q = sh->s_q; k.batch = sh->batch; k.hpk = hpk;
    const bool concat = elem == 1 || p.q_concat;
    k.lat = elem == 1 ? static_cast<const void *>(p.q8) : static_cast<const void *>(p.q);
    // a concatenated query has one map base for both: the RoPE boxes start at dim qr_x0 = 512
    k.rope = concat ? k.lat : static_cast<const void *>(p.q_rope);
    k.lat_dims = concat ? MLA_HEAD_DIM : MLA_HEAD_DIM_V;
    k.rope_dims = concat ? MLA_HEAD_DIM : MLA_HEAD_DIM - MLA_HEAD_DIM_V;
    const int64_t ls[3] = {p.q_s2, p.q_s1, p.q_s0}, rs[3] = {p.qr_s2, p.qr_s1, p.qr_s0};
    for (int i = 0; i < 3; ++i) {
        k.lat_stride[i] = ls[i];
        k.rope_stride[i] = concat ? ls[i] : rs[i];
    }
    const int hb = hpk >= kRowsPerBlock ? kRowsPerBlock : hpk, tb = kRowsPerBlock / hb;
    const int hbr = hpk >= 64 ? 64 : hpk, tbr = 64 / hbr;
    p.q_hb = hb;
    p.q_tb = tb;
    p.qr_x0 = concat ? MLA_HEAD_DIM_V : 0;
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto &e : g_qmaps) {
        if (e.valid && e.key == k) {
            *lat = e.lat;
            *rope = e.rope;
            p.q_tma = e.ok ? 1 : 0;
            return e.ok;
        }
    }
    EncodeTiledFn enc;
    if (get_encoder(&enc) != MLA_OK) return false;
    const cuuint64_t eb = (cuuint64_t)elem;
    const cuuint64_t gdim_l[4] = {(cuuint64_t)k.lat_dims, (cuuint64_t)sh->h_q, (cuuint64_t)sh->s_q, (cuuint64_t)sh->batch};
    const cuuint64_t gdim_r[4] = {(cuuint64_t)k.rope_dims, (cuuint64_t)sh->h_q, (cuuint64_t)sh->s_q, (cuuint64_t)sh->batch};
    const cuuint64_t gstr_l[3] = {(cuuint64_t)k.lat_stride[0] * eb, (cuuint64_t)k.lat_stride[1] * eb,
                                  (cuuint64_t)k.lat_stride[2] * eb};
    const cuuint64_t gstr_r[3] = {(cuuint64_t)k.rope_stride[0] * eb, (cuuint64_t)k.rope_stride[1] * eb,
                                  (cuuint64_t)k.rope_stride[2] * eb};
    // latent boxes of 128-byte rows (SW128); RoPE boxes of 32 dims: 64-byte rows (SW64) in bf16,
    // 32-byte rows (SW32) in e4m3 -- the layouts of the Q RoPE tile the kernel keeps
    const cuuint32_t box_l[4] = {(cuuint32_t)(128 / elem), (cuuint32_t)hb, (cuuint32_t)tb, 1},
                     box_r[4] = {32, (cuuint32_t)hbr, (cuuint32_t)tbr, 1}, es[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle rsw = elem == 1 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
    QMapEntry &e = g_qmaps[g_qmap_next];
    g_qmap_next = (g_qmap_next + 1) % kMapCache;
    e.key = k;
    CUresult r1 = enc(&e.lat, dt, 4, const_cast<void *>(k.lat), gdim_l, gstr_l, box_l, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = enc(&e.rope, dt, 4, const_cast<void *>(k.rope), gdim_r, gstr_r, box_r, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, rsw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    e.ok = r1 == CUDA_SUCCESS && r2 == CUDA_SUCCESS;
    e.valid = true;
    *lat = e.lat;
    *rope = e.rope;
    p.q_tma = e.ok ? 1 : 0;
    return e.ok;
}

int launch_splitkv(const mla_shape_t *sh, const KvSource &src, const Prepared &pr, cudaStream_t stream) {
    CUtensorMap m128, m64, mq, mqr;
    int st = kcache_maps(sh, src, &m128, &m64);
    if (st != MLA_OK) return st;
    DecodeParams p = pr.p;
    if (!query_maps(sh, src.elem, p, &mq, &mqr)) {
        memset(&mq, 0, sizeof mq);
        memset(&mqr, 0, sizeof mqr);
    }
    if (src.elem == 1)
        mla_splitkv_kernel_f8<<<pr.grid, splitkv_threads(), splitkv_f8_smem_bytes(), stream>>>(m128, m64, mq, mqr, p);
    else
        mla_splitkv_kernel<<<pr.grid, splitkv_threads(), splitkv_smem_bytes(), stream>>>(m128, m64, mq, mqr, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "split-KV decode launch");
    return MLA_OK;
}

// The combine is a programmatic dependent launch: its blocks may be scheduled
// while the split-KV kernel drains and wait (griddepcontrol.wait) for its
// results, which hides most of the launch gap between the two kernels.
int launch_combine(const mla_shape_t *sh, const Prepared &pr, cudaStream_t stream) {
    const uint32_t rpb = combine_rows_per_block();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((pr.p.rows + rpb - 1) / rpb, sh->batch, sh->h_k);
    cfg.blockDim = dim3(combine_threads(), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, mla_combine_kernel, pr.p);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return MLA_OK;
}

int launch_metadata(const int32_t *seqlens, int batch, int parts, int cost, int32_t *md, int32_t *num_splits,
                    cudaStream_t stream) {
    mla_metadata_kernel<<<1, 256, metadata_smem_bytes(batch, parts), stream>>>(seqlens, batch, parts, cost, md,
                                                                              num_splits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "metadata launch");
    return MLA_OK;
}

// ---------------------------------------------------------------------------
// the host-buffer path (mla_decode_fwd_host)
// ---------------------------------------------------------------------------
// Device staging for one (device, stream): the workspace, the inputs copied
// from the host, the schedule, and output staging for host buffers the
// kernels cannot write directly.  Grown with cudaMallocAsync / cudaFreeAsync
// on the stream.  `side` is a second stream on which the schedule is
// computed while q is copied; `fork` / `join` order it against `stream`.
struct HostEntry {
    int device = -1;
    cudaStream_t stream = nullptr;
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    void *ptr = nullptr;
    size_t bytes = 0;
};
constexpr int kHostEntries = 16;
HostEntry g_host[kHostEntries];   // guarded by g_ws_mu

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Staging areas, in order: workspace, q, block_table, cache_seqlens,
// metadata, num_splits, out, lse (each 256-byte aligned).
enum { kStWs, kStQ, kStBt, kStLen, kStMd, kStNs, kStOut, kStLse, kStCount };
struct HostLayout {
    size_t off[kStCount], size[kStCount], total;
};

HostLayout host_layout(const mla_shape_t *sh) {
    const int64_t B = sh->batch;
    HostLayout l;
    l.size[kStWs] = workspace_bytes_for(sh, nullptr);
    l.size[kStQ] = B > 0 ? (size_t)((B - 1) * sh->q_stride[0] + (sh->s_q - 1) * sh->q_stride[1] +
                                    (sh->h_q - 1) * sh->q_stride[2] + sh->head_dim) * 2
                         : 0;
    l.size[kStBt] = B > 0 ? (size_t)((B - 1) * sh->bt_stride + sh->max_blocks_per_seq) * 4 : 0;
    l.size[kStLen] = (size_t)B * 4;
    l.size[kStMd] = (size_t)sh->num_sm_parts * MLA_METADATA_SIZE * 4;
    l.size[kStNs] = (size_t)(B + 1) * 4;
    l.size[kStOut] = (size_t)B * sh->s_q * sh->h_q * MLA_HEAD_DIM_V * 2;
    l.size[kStLse] = (size_t)B * sh->h_q * sh->s_q * 4;
    size_t o = 0;
    for (int i = 0; i < kStCount; ++i) {
        l.off[i] = o;
        o += align256(l.size[i]);
    }
    l.total = o;
    return l;
}

int host_entry(cudaStream_t stream, size_t need, HostEntry **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_ws_mu);
    HostEntry *slot = nullptr;
    for (auto &h : g_host) {
        if (h.side && h.device == dev && h.stream == stream) { slot = &h; break; }
        if (!h.side && !slot) slot = &h;
    }
    if (!slot) return fail(MLA_ERR_UNSUPPORTED, "more than %d (device, stream) pairs use the host-buffer path", kHostEntries);
    if (!slot->side) {
        if ((e = cudaStreamCreateWithFlags(&slot->side, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamCreateWithFlags");
        if ((e = cudaEventCreateWithFlags(&slot->fork, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&slot->join, cudaEventDisableTiming)) != cudaSuccess) {
            if (slot->fork) cudaEventDestroy(slot->fork);
            cudaStreamDestroy(slot->side);
            *slot = HostEntry();
            return cuda_fail(e, "cudaEventCreateWithFlags");
        }
        slot->device = dev;
        slot->stream = stream;
    }
    if (slot->bytes < need) {
        if (slot->ptr && (e = cudaFreeAsync(slot->ptr, stream)) != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(staging)");
        slot->ptr = nullptr;
        slot->bytes = 0;
        void *ptr = nullptr;
        if ((e = cudaMallocAsync(&ptr, need, stream)) != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(staging)");
        slot->ptr = ptr;
        slot->bytes = need;
    }
    *out = slot;
    return MLA_OK;
}

// The device address the kernels may write for host buffer `h`: its mapped
// alias when `h` is page-locked memory mapped into the device's address
// space, else NULL (the result is staged and copied back).
void *mapped_alias(void *h) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

namespace mla {
// Records `msg` as the calling thread's last error (mla_last_error) and
// returns `status`; for entry points defined in other files.
int report_error(int status, const char *msg) { return fail(status, "%s", msg); }
}  // namespace mla

extern "C" {

int mla_version(void) { return 100; }

const char *mla_status_string(int status) {
    switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_ARCH: return "device is not sm_103 (GB300)";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_DEVICE: return "device-side error reported by a kernel";
    default: return "unknown status";
    }
}

const char *mla_last_error(void) { return t_last_error.c_str(); }

int mla_get_num_sm_parts(int device, int num_heads_per_head_k, int num_heads_k, int *num_sm_parts) {
    if (!num_sm_parts || num_heads_per_head_k < 1 || num_heads_k < 1)
        return fail(MLA_ERR_ARG, "mla_get_num_sm_parts: bad argument");
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (device != prev && (e = cudaSetDevice(device)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    DeviceState *ds = nullptr;
    int st = device_state(&ds);
    if (device != prev) cudaSetDevice(prev);
    if (st != MLA_OK) return st;
    const int row_blocks = (num_heads_per_head_k + kRowsPerBlock - 1) / kRowsPerBlock;
    int parts = ds->max_clusters / (row_blocks * num_heads_k);
    *num_sm_parts = parts < 1 ? 1 : parts;
    return MLA_OK;
}

int mla_get_metadata(const int32_t *cache_seqlens, int batch, int num_heads_per_head_k, int num_heads_k,
                     int num_sm_parts, int32_t *tile_scheduler_metadata, int32_t *num_splits, mla_stream_t stream) {
    return mla_get_metadata_ex(cache_seqlens, batch, num_heads_per_head_k, num_heads_k, 2, num_sm_parts,
                               tile_scheduler_metadata, num_splits, stream);
}

int mla_get_metadata_ex(const int32_t *cache_seqlens, int batch, int num_heads_per_head_k, int num_heads_k,
                        int kv_bytes, int num_sm_parts, int32_t *tile_scheduler_metadata, int32_t *num_splits,
                        mla_stream_t stream) {
    if (!tile_scheduler_metadata || !num_splits || (batch > 0 && !cache_seqlens))
        return fail(MLA_ERR_ARG, "mla_get_metadata: NULL pointer");
    if (batch < 0 || num_sm_parts < 1 || num_heads_per_head_k < 1 || num_heads_k < 1)
        return fail(MLA_ERR_ARG, "mla_get_metadata: bad argument");
    if (kv_bytes != 1 && kv_bytes != 2) return fail(MLA_ERR_ARG, "mla_get_metadata_ex: kv_bytes must be 1 or 2");
    if (batch > kMaxBatchMetadata) return fail(MLA_ERR_UNSUPPORTED, "batch %d > %d", batch, kMaxBatchMetadata);
    if (num_sm_parts > kMaxPartsMetadata)
        return fail(MLA_ERR_UNSUPPORTED, "num_sm_parts %d > %d", num_sm_parts, kMaxPartsMetadata);
    DeviceState *ds = nullptr;
    int st = device_state(&ds);
    if (st != MLA_OK) return st;
    return launch_metadata(cache_seqlens, batch, num_sm_parts, segment_cost(num_heads_per_head_k, kv_bytes),
                           tile_scheduler_metadata, num_splits, reinterpret_cast<cudaStream_t>(stream));
}

int mla_workspace_size(const mla_shape_t *shape, size_t *bytes) {
    if (!bytes) return fail(MLA_ERR_ARG, "bytes is NULL");
    int st = check_shape(shape);
    if (st != MLA_OK) return st;
    *bytes = workspace_bytes_for(shape, nullptr);
    return MLA_OK;
}

int mla_decode_splitkv(const mla_shape_t *shape, const void *q, const void *k_cache, const int32_t *block_table,
                       const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float scale,
                       int causal, void *out, float *lse, void *ws, size_t ws_bytes, mla_stream_t stream) {
    if (!ws && ws_bytes == 0) {
        int wst = check_args(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, out, lse, true);
        if (wst == MLA_OK) wst = internal_workspace(shape, reinterpret_cast<cudaStream_t>(stream), &ws, &ws_bytes);
        if (wst != MLA_OK) return wst;
    }
    Prepared pr;
    DeviceState *ds = nullptr;
    int st = prepare(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, scale, causal, out, lse, ws,
                     ws_bytes, true, &pr, &ds);
    if (st != MLA_OK) return st;
    if (shape->batch == 0) return MLA_OK;
    return launch_splitkv(shape, concat_source(shape, k_cache), pr, reinterpret_cast<cudaStream_t>(stream));
}

int mla_decode_combine(const mla_shape_t *shape, const void *q, const void *k_cache, const int32_t *block_table,
                       const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float scale,
                       int causal, void *out, float *lse, void *ws, size_t ws_bytes, mla_stream_t stream) {
    if (!ws && ws_bytes == 0) {
        int wst = check_args(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, out, lse, false);
        if (wst == MLA_OK) wst = internal_workspace(shape, reinterpret_cast<cudaStream_t>(stream), &ws, &ws_bytes);
        if (wst != MLA_OK) return wst;
    }
    Prepared pr;
    DeviceState *ds = nullptr;
    int st = prepare(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, scale, causal, out, lse, ws,
                     ws_bytes, false, &pr, &ds);
    if (st != MLA_OK) return st;
    if (shape->batch == 0) return MLA_OK;
    return launch_combine(shape, pr, reinterpret_cast<cudaStream_t>(stream));
}

int mla_decode_fwd(const mla_shape_t *shape, const void *q, const void *k_cache, const int32_t *block_table,
                   const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float scale,
                   int causal, void *out, float *lse, void *ws, size_t ws_bytes, mla_stream_t stream) {
    if (!ws && ws_bytes == 0) {
        int wst = check_args(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, out, lse, true);
        if (wst == MLA_OK) wst = internal_workspace(shape, reinterpret_cast<cudaStream_t>(stream), &ws, &ws_bytes);
        if (wst != MLA_OK) return wst;
    }
    Prepared pr;
    DeviceState *ds = nullptr;
    int st = prepare(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, scale, causal, out, lse, ws,
                     ws_bytes, true, &pr, &ds);
    if (st != MLA_OK) return st;
    if (shape->batch == 0) return MLA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = launch_splitkv(shape, concat_source(shape, k_cache), pr, s);
    if (st != MLA_OK) return st;
    return launch_combine(shape, pr, s);
}

}  // extern "C"

namespace {
// Validation and launches of the e4m3 decode; `combine` selects both launches
// (mla_decode_fwd_fp8) or the split-KV one alone (mla_decode_splitkv_fp8).
int decode_fp8(const mla_shape_t *shape, const void *q, const void *k_cache, const int32_t *block_table,
               const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float bmm1_scale,
               float bmm2_scale, int causal, void *out, float *lse, void *ws, size_t ws_bytes, mla_stream_t stream,
               bool combine) {
    int st = check_args(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, out, lse, true);
    if (st != MLA_OK) return st;
    if (!(bmm1_scale > 0.f) || !std::isfinite(bmm1_scale) || !std::isfinite(bmm2_scale))
        return fail(MLA_ERR_ARG, "bmm1_scale must be positive and finite, bmm2_scale finite");
    for (int i = 0; i < 3; ++i)
        if (shape->q_stride[i] % 16 || shape->k_stride[i] % 16)
            return fail(MLA_ERR_ARG, "e4m3 q and k_cache strides must be multiples of 16 elements");
    if (!ws && ws_bytes == 0) {
        st = internal_workspace(shape, reinterpret_cast<cudaStream_t>(stream), &ws, &ws_bytes);
        if (st != MLA_OK) return st;
    }
    Prepared pr;
    DeviceState *ds = nullptr;
    st = prepare(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, bmm1_scale, causal, out, lse, ws,
                 ws_bytes, true, &pr, &ds);
    if (st != MLA_OK) return st;
    pr.p.q = nullptr;
    pr.p.q_rope = nullptr;
    pr.p.q8 = static_cast<const uint8_t *>(q);
    pr.p.out_scale = bmm2_scale;
    if (shape->batch == 0) return MLA_OK;
    KvSource src = concat_source(shape, k_cache);
    src.elem = 1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = launch_splitkv(shape, src, pr, s)) != MLA_OK) return st;
    return combine ? launch_combine(shape, pr, s) : MLA_OK;
}
}  // namespace

extern "C" {

int mla_decode_fwd_fp8(const mla_shape_t *shape, const void *q, const void *k_cache, const int32_t *block_table,
                       const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float bmm1_scale,
                       float bmm2_scale, int causal, void *out, float *lse, void *ws, size_t ws_bytes,
                       mla_stream_t stream) {
    return decode_fp8(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, bmm1_scale, bmm2_scale, causal,
                      out, lse, ws, ws_bytes, stream, true);
}

int mla_decode_splitkv_fp8(const mla_shape_t *shape, const void *q, const void *k_cache,
                           const int32_t *block_table, const int32_t *cache_seqlens, const int32_t *md,
                           const int32_t *num_splits, float bmm1_scale, float bmm2_scale, int causal, void *out,
                           float *lse, void *ws, size_t ws_bytes, mla_stream_t stream) {
    return decode_fp8(shape, q, k_cache, block_table, cache_seqlens, md, num_splits, bmm1_scale, bmm2_scale, causal,
                      out, lse, ws, ws_bytes, stream, false);
}

int mla_decode_fwd_split(const mla_shape_t *shape, const mla_rope_strides_t *rope, const void *q_nope,
                         const void *q_rope, const void *ctkv, const void *krope, const int32_t *block_table,
                         const int32_t *cache_seqlens, const int32_t *md, const int32_t *num_splits, float scale,
                         int causal, void *out, float *lse, void *ws, size_t ws_bytes, mla_stream_t stream) {
    if (!rope) return fail(MLA_ERR_ARG, "rope strides are NULL");
    int st = check_args(shape, q_nope, ctkv, block_table, cache_seqlens, md, num_splits, out, lse, true);
    if (st != MLA_OK) return st;
    if (!q_rope || !krope) return fail(MLA_ERR_ARG, "NULL tensor pointer");
    if (!aligned16(q_rope) || !aligned16(krope)) return fail(MLA_ERR_ARG, "q_rope and krope must be 16-byte aligned");
    for (int i = 0; i < 3; ++i) {
        if (rope->q_rope_stride[i] <= 0 || rope->q_rope_stride[i] % 8 || rope->krope_stride[i] <= 0 ||
            rope->krope_stride[i] % 8)
            return fail(MLA_ERR_ARG, "rope strides must be positive multiples of 8 elements");
    }
    if (shape->q_stride[2] < MLA_HEAD_DIM_V || shape->k_stride[2] < MLA_HEAD_DIM_V ||
        rope->q_rope_stride[2] < MLA_HEAD_DIM - MLA_HEAD_DIM_V || rope->krope_stride[2] < MLA_HEAD_DIM - MLA_HEAD_DIM_V)
        return fail(MLA_ERR_ARG, "head strides smaller than the head's dims");
    if (!ws && ws_bytes == 0) {
        if ((st = internal_workspace(shape, reinterpret_cast<cudaStream_t>(stream), &ws, &ws_bytes)) != MLA_OK) return st;
    }
    Prepared pr;
    DeviceState *ds = nullptr;
    if ((st = prepare(shape, q_nope, ctkv, block_table, cache_seqlens, md, num_splits, scale, causal, out, lse, ws,
                      ws_bytes, true, &pr, &ds)) != MLA_OK)
        return st;
    pr.p.q_rope = static_cast<const uint16_t *>(q_rope);
    pr.p.qr_s0 = rope->q_rope_stride[0]; pr.p.qr_s1 = rope->q_rope_stride[1]; pr.p.qr_s2 = rope->q_rope_stride[2];
    pr.p.rope_x0 = 0;
    pr.p.q_concat = pr.p.q_rope == pr.p.q + MLA_HEAD_DIM_V && pr.p.qr_s0 == pr.p.q_s0 && pr.p.qr_s1 == pr.p.q_s1 &&
                    pr.p.qr_s2 == pr.p.q_s2;
    if (shape->batch == 0) return MLA_OK;
    KvSource src;
    src.latent = ctkv;
    src.rope = krope;
    for (int i = 0; i < 3; ++i) {
        src.lat_stride[i] = shape->k_stride[i];
        src.rope_stride[i] = rope->krope_stride[i];
    }
    src.lat_dims = MLA_HEAD_DIM_V;
    src.rope_dims = MLA_HEAD_DIM - MLA_HEAD_DIM_V;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = launch_splitkv(shape, src, pr, s)) != MLA_OK) return st;
    return launch_combine(shape, pr, s);
}

int mla_decode_fwd_host(const mla_shape_t *shape, const void *q_host, const void *k_cache,
                        const int32_t *block_table_host, const int32_t *cache_seqlens_host, float scale, int causal,
                        void *out_host, float *lse_host, mla_stream_t stream) {
    int st = check_shape(shape);
    if (st != MLA_OK) return st;
    const mla_shape_t &sh = *shape;
    if (sh.batch == 0) return MLA_OK;   // nothing to compute; the pointers of empty tensors may be NULL
    if (!q_host || !k_cache || !block_table_host || !cache_seqlens_host || !out_host || !lse_host)
        return fail(MLA_ERR_ARG, "NULL pointer");
    if (!aligned16(q_host) || !aligned16(k_cache) || !aligned16(out_host))
        return fail(MLA_ERR_ARG, "q, k_cache and out must be 16-byte aligned");
    const int64_t o2 = MLA_HEAD_DIM_V, o1 = (int64_t)sh.h_q * o2, o0 = (int64_t)sh.s_q * o1;
    if (sh.out_stride[0] != o0 || sh.out_stride[1] != o1 || sh.out_stride[2] != o2)
        return fail(MLA_ERR_ARG, "out must be contiguous for the host-buffer call");
    if (sh.batch > kMaxBatchMetadata) return fail(MLA_ERR_UNSUPPORTED, "batch %d > %d", sh.batch, kMaxBatchMetadata);
    if (sh.num_sm_parts > kMaxPartsMetadata)
        return fail(MLA_ERR_UNSUPPORTED, "num_sm_parts %d > %d", sh.num_sm_parts, kMaxPartsMetadata);
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MLA_OK) return st;

    const HostLayout lay = host_layout(&sh);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    HostEntry *h = nullptr;
    if ((st = host_entry(s, lay.total, &h)) != MLA_OK) return st;
    char *base = static_cast<char *>(h->ptr);
    void *ws = base + lay.off[kStWs];
    void *q_d = base + lay.off[kStQ];
    int32_t *bt_d = reinterpret_cast<int32_t *>(base + lay.off[kStBt]);
    int32_t *L_d = reinterpret_cast<int32_t *>(base + lay.off[kStLen]);
    int32_t *md_d = reinterpret_cast<int32_t *>(base + lay.off[kStMd]);
    int32_t *ns_d = reinterpret_cast<int32_t *>(base + lay.off[kStNs]);
    void *out_direct = mapped_alias(out_host);
    void *lse_direct = mapped_alias(lse_host);
    void *out_d = out_direct ? out_direct : base + lay.off[kStOut];
    float *lse_d = static_cast<float *>(lse_direct ? lse_direct : base + lay.off[kStLse]);

    Prepared pr;
    if ((st = prepare(&sh, q_d, k_cache, bt_d, L_d, md_d, ns_d, scale, causal, out_d, lse_d, ws, lay.size[kStWs], true,
                      &pr, &ds)) != MLA_OK)
        return st;
    cudaError_t e;
    // schedule stream: cache_seqlens and block_table in, then the schedule
    if ((e = cudaEventRecord(h->fork, s)) != cudaSuccess || (e = cudaStreamWaitEvent(h->side, h->fork, 0)) != cudaSuccess)
        return cuda_fail(e, "fork to the schedule stream");
    if ((e = cudaMemcpyAsync(L_d, cache_seqlens_host, lay.size[kStLen], cudaMemcpyHostToDevice, h->side)) != cudaSuccess ||
        (e = cudaMemcpyAsync(bt_d, block_table_host, lay.size[kStBt], cudaMemcpyHostToDevice, h->side)) != cudaSuccess)
        return cuda_fail(e, "copy of cache_seqlens / block_table");
    const int rows = (int)((long long)sh.s_q * sh.h_q / sh.h_k);
    if ((st = launch_metadata(L_d, sh.batch, sh.num_sm_parts, segment_cost(rows, 2), md_d, ns_d, h->side)) != MLA_OK)
        return st;
    if ((e = cudaEventRecord(h->join, h->side)) != cudaSuccess) return cuda_fail(e, "join event");
    // this stream: q in, wait for the schedule, decode, results out
    if ((e = cudaMemcpyAsync(q_d, q_host, lay.size[kStQ], cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "copy of q");
    if ((e = cudaStreamWaitEvent(s, h->join, 0)) != cudaSuccess) return cuda_fail(e, "join of the schedule stream");
    if ((st = launch_splitkv(&sh, concat_source(&sh, k_cache), pr, s)) != MLA_OK) return st;
    if ((st = launch_combine(&sh, pr, s)) != MLA_OK) return st;
    if (!out_direct && (e = cudaMemcpyAsync(out_host, out_d, lay.size[kStOut], cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "copy of out");
    if (!lse_direct && (e = cudaMemcpyAsync(lse_host, lse_d, lay.size[kStLse], cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "copy of softmax_lse");
    return MLA_OK;
}

int mla_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int status = MLA_OK;
    for (auto &w : g_ws) {
        if (!w.ptr) continue;
        if ((e = cudaSetDevice(w.device)) == cudaSuccess && (e = cudaDeviceSynchronize()) == cudaSuccess)
            e = cudaFree(w.ptr);
        if (e != cudaSuccess && status == MLA_OK) status = cuda_fail(e, "mla_shutdown: freeing the internal workspace");
        w = WsEntry();
    }
    for (auto &h : g_host) {
        if (!h.side) continue;
        if ((e = cudaSetDevice(h.device)) == cudaSuccess && (e = cudaDeviceSynchronize()) == cudaSuccess) {
            if (h.ptr) e = cudaFree(h.ptr);
            cudaEventDestroy(h.fork);
            cudaEventDestroy(h.join);
            cudaStreamDestroy(h.side);
        }
        if (e != cudaSuccess && status == MLA_OK) status = cuda_fail(e, "mla_shutdown: releasing the host-path staging");
        h = HostEntry();
    }
    cudaSetDevice(prev);
    {
        // what was looked up per device (kernel attributes, symbol addresses,
        // tensor maps) is set up again by the next call: after a context reset
        // the module may be loaded at other addresses
        std::lock_guard<std::mutex> dlock(g_mu);
        for (auto &d : g_dev) d = DeviceState();
        for (auto &m : g_maps) m.valid = false;
        for (auto &m : g_qmaps) m.valid = false;
    }
    mla::noalloc_forget_devices();
    return status;
}

int mla_check_device_error(int *bits, int clear) {
    if (!bits) return fail(MLA_ERR_ARG, "bits is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_mla_device_error, sizeof v)) != cudaSuccess)
        return cuda_fail(e, "read device error word");
    *bits = v;
    if (clear && v) {
        const int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_mla_device_error, &zero, sizeof zero)) != cudaSuccess)
            return cuda_fail(e, "clear device error word");
    }
    return MLA_OK;
}

}  // extern "C"
