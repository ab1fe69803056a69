// ga_noalloc.cu -- a global-family decode entry point whose split-KV scratch
// lives in a fixed device array built into the library, so the caller never
// has to allocate a workspace.
//
// Who needs it: callers that cannot allocate device memory when they decode.
// A plain-C serving loop without a caching allocator would otherwise call
// cudaMalloc, which synchronises the whole device in the middle of a decode
// step; a host that has handed all free device memory to its fixed KV pools
// has nothing left to allocate from.  Such callers still pass their own
// inputs and outputs; only the scratch (split-KV partials and their
// log-sum-exp values) comes from here.
//
// The array is GA_NOALLOC_SCRATCH_BYTES (64 MiB) per GPU, held by every GPU
// that loads the library until the process exits.  All calls share it: two
// calls whose kernels overlap on the GPU (different streams, or different
// threads without ordering) race on it and give wrong results.  The array
// keeps whatever the last call left; nothing in it has to start at zero,
// because the decode kernel writes every partial that the merge step reads.
#include <cuda_runtime.h>

#include <mutex>

#include "ga_internal.h"

namespace ga {
namespace {

constexpr size_t kScratchBytes = GA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  The name
// g_noalloc_scratch is only a host-side stand-in; its device address is looked
// up once per device (with that device current) and cached.
int scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return GA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GA_OK;
}

}  // namespace
}  // namespace ga

extern "C" int ga_decode_global_hd512_noalloc(
    const void* q, const void* k_pool, const void* v_pool, int32_t kv_dtype,
    const float* k_scale, const float* v_scale, const int32_t* page_table, int64_t pt_stride,
    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t page_size, int64_t num_pages, float scale, const ga_plan* plan, void* out,
    int32_t* err_word, ga_stream_t stream) {
    if (plan == nullptr) return GA_ERR_INVALID_ARG;
    if (plan->workspace_bytes < 0 ||
        (uint64_t)plan->workspace_bytes > (uint64_t)ga::kScratchBytes)
        return GA_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    if (plan->workspace_bytes > 0) {
        const int rc = ga::scratch_on_current_device(&scratch);
        if (rc != GA_OK) return rc;
    }
    return ga_decode_global_hd512(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table,
                                  pt_stride, seq_lens, batch, num_q_heads, num_kv_heads,
                                  page_size, num_pages, scale, plan, scratch,
                                  scratch ? ga::kScratchBytes : 0, out, err_word, stream);
}
