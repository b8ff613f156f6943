// noalloc.cu -- mla_decode_fwd_noalloc: the decode with built-in scratch.
//
// mla_decode_fwd needs a caller-provided workspace for the partial results of
// the sequences the schedule splits.  Some callers cannot hand one over:
// code whose device memory is entirely owned by another allocator (an
// inference server's memory pool, for instance), or a latency-critical loop
// that cannot risk the device-wide synchronisation cudaMalloc / cudaFree may
// trigger.  This entry point serves them: its scratch is a fixed array in the
// library's own device memory, so the call allocates nothing.
//
// Costs and rules of that choice:
//   * every GPU that loads the library holds MLA_NOALLOC_SCRATCH_BYTES for
//     it until the process exits;
//   * all calls share the one array, so two calls whose kernels overlap on
//     the GPU (different streams, no ordering between them) race on it;
//   * nothing in it has to start at zero: every partial slot the combine
//     reads is written earlier in the same call, so the leftovers of the
//     previous call are never read;
//   * the first call on a device looks up the array's device address (with
//     that device current); make that first call before any stream capture.
//     mla_shutdown forgets the address, so that a call after a context reset
//     (cudaDeviceReset, which may reload the module elsewhere) looks it up
//     again.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "libmla.h"

namespace mla {
int report_error(int status, const char *msg);
void noalloc_forget_devices();
}

// The scratch itself: file-scope device memory, MLA_NOALLOC_SCRATCH_BYTES per GPU.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device (set up once).
// In host code the array's name is only a stand-in, not a device pointer.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return mla::report_error(MLA_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return mla::report_error(MLA_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(built-in scratch): %s", cudaGetErrorString(e));
            return mla::report_error(MLA_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

}  // namespace

// Called by mla_shutdown: the next call on each device looks the address up again.
void mla::noalloc_forget_devices() {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto &p : g_scratch_ptr) p = nullptr;
}

extern "C" int mla_decode_fwd_noalloc(const mla_shape_t *shape, const void *q, const void *k_cache,
                                      const int32_t *block_table, const int32_t *cache_seqlens,
                                      const int32_t *tile_scheduler_metadata, const int32_t *num_splits,
                                      float softmax_scale, int causal, void *out, float *softmax_lse,
                                      mla_stream_t stream) {
    size_t need = 0;
    int st = mla_workspace_size(shape, &need);
    if (st != MLA_OK) return st;
    if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "mla_decode_fwd_noalloc: this problem needs %zu bytes of scratch, the built-in scratch holds %zu; "
                 "use mla_decode_fwd with a caller-provided workspace",
                 need, (size_t)MLA_NOALLOC_SCRATCH_BYTES);
        return mla::report_error(MLA_ERR_UNSUPPORTED, msg);
    }
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != MLA_OK) return st;
    return mla_decode_fwd(shape, q, k_cache, block_table, cache_seqlens, tile_scheduler_metadata, num_splits,
                          softmax_scale, causal, out, softmax_lse, scratch, MLA_NOALLOC_SCRATCH_BYTES, stream);
}
