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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ga_internal.h"

namespace ga {
namespace {

constexpr size_t kScratchBytes = GA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CachedScratch {
    unsigned long long ctx_id;   // context the address belongs to
    void* ptr;
};

std::mutex g_scratch_mu;
CachedScratch g_scratch[kMaxDevices] = {};

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

DriverFns lookup_driver_fns() {
    DriverFns f;
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess && a && b) {
        f.get_current = reinterpret_cast<CtxGetCurrentFn>(a);
        f.get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
    return f;
}

// Unique id of the calling thread's current context (0: none current).  Ids
// are never reused within a process, so a device reset or another context
// made current shows up as a new id.
int current_context_id(unsigned long long* id) {
    static const DriverFns fns = lookup_driver_fns();   // thread-safe one-time init
    if (!fns.get_current || !fns.get_id) return GA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (fns.get_current(&ctx) != CUDA_SUCCESS) return GA_ERR_CUDA;
    *id = 0;
    if (ctx && fns.get_id(ctx, id) != CUDA_SUCCESS) return GA_ERR_CUDA;
    return GA_OK;
}

// Device address of the array in the current device's current context.  The
// name g_noalloc_scratch is only a host-side stand-in; its device address is
// looked up with the device current and cached per device together with the
// context it belongs to, and looked up again when that context changes.
int scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GA_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    int rc = current_context_id(&id);
    if (rc != GA_OK) return rc;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (id != 0 && g_scratch[dev].ptr != nullptr && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].ptr;
        return GA_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return GA_ERR_CUDA;
    // the lookup makes the device's primary context current if none was
    rc = current_context_id(&id);
    if (rc != GA_OK) return rc;
    g_scratch[dev] = CachedScratch{id, p};
    *out = p;
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
    // the touch log would land in the built-in array, where the caller cannot
    // read it
    if (plan->flags & GA_PLAN_TOUCH_LOG) return GA_ERR_INVALID_ARG;
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
