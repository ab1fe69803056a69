// ga_stream.cu -- a read-only HBM stream: the practical read ceiling the
// decode kernels are measured against.  Nothing of the attention method; a
// measurement helper exported as ga_read_stream.
#include <cuda_runtime.h>

#include "ga_device.cuh"
#include "ga_internal.h"

namespace ga {

namespace {

constexpr int kStreamThreads = 256;
constexpr int kStreamCtasPerSm = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Grid-stride loop, four independent 16-byte loads in flight per thread; the
// loaded words are XOR-folded and the fold decides a (practically never taken)
// store, so no load can be dropped.
__global__ void __launch_bounds__(kStreamThreads) read_stream_kernel(const uint4* __restrict__ src,
                                                                    int64_t n16,
                                                                    unsigned long long* sink) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = ld_stream(src + i), b = ld_stream(src + i + stride),
                    c = ld_stream(src + i + 2 * stride), d = ld_stream(src + i + 3 * stride);
        acc ^= (a.x ^ a.y ^ a.z ^ a.w) ^ (b.x ^ b.y ^ b.z ^ b.w) ^ (c.x ^ c.y ^ c.z ^ c.w) ^
               (d.x ^ d.y ^ d.z ^ d.w);
    }
    for (; i < n16; i += stride) {
        const uint4 a = ld_stream(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (acc == 0x9E3779B9u) atomicAdd(sink, 1ull);
}

}  // namespace

}  // namespace ga

extern "C" int ga_read_stream(const void* src, int64_t bytes, void* sink, ga_stream_t stream) {
    if (src == nullptr || sink == nullptr || bytes <= 0 || bytes % 16 != 0 || !ga::aligned16(src))
        return GA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GA_ERR_CUDA;
    const int grid = sms * ga::kStreamCtasPerSm;
    ga::read_stream_kernel<<<grid, ga::kStreamThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(src), bytes / 16, static_cast<unsigned long long*>(sink));
    return cudaGetLastError() == cudaSuccess ? GA_OK : GA_ERR_CUDA;
}
