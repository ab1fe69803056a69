// ga_combine.cu -- log-sum-exp merge of split-KV partials.
//
// For row b, query head h and the row's chunks s = 0 .. S_b-1:
//     M = max_s lse_s,  w_s = e^{lse_s - M},  out = sum_s w_s o_s / sum_s w_s
// ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is mandatory here":
// flash-decode with split factor 8).  o_s is normalised within its chunk and
// lse_s is the chunk's natural-log log-sum-exp; empty chunks carry -inf.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "ga_device.cuh"
#include "ga_internal.h"

namespace ga {

struct CombineParams {
    const float* po;        // [rc, Hq, D]
    const float* plse;      // [rc, Hq]
    const int32_t* seq_lens;
    __nv_bfloat16* out;     // [B, Hq, D]
    int32_t* err_word;
    int64_t pt_stride;
    int64_t rc_capacity;
    int32_t B, Hq, D, window, mode, splits, chunk_pages;
};

// One CTA per (query head, row); blockDim.x = D / 4 threads, 4 dims each.
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
    const int h = blockIdx.x, b = blockIdx.y;
    __shared__ int32_t s_red[32];
    // row-chunk offset of row b: chunks of all rows before it
    int32_t part = 0;
    for (int r = threadIdx.x; r < b; r += blockDim.x)
        part += row_geometry(__ldg(p.seq_lens + r), p.window, p.pt_stride, p.mode, p.splits,
                             p.chunk_pages).chunks;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = part;
    __syncthreads();
    int64_t rc0 = 0;
    for (int wv = 0; wv < (int)(blockDim.x + 31) / 32; ++wv) rc0 += s_red[wv];
    const RowGeom g = row_geometry(__ldg(p.seq_lens + b), p.window, p.pt_stride, p.mode,
                                   p.splits, p.chunk_pages);
    const int S = g.chunks;
    if (S <= 1) return;                       // written by the decode kernel
    if (rc0 + S > p.rc_capacity) {
        if (threadIdx.x == 0) report(p.err_word, kErrCapacity);
        return;
    }
    const float* lse = p.plse + rc0 * p.Hq + h;
    float M = -CUDART_INF_F;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldg(lse + (int64_t)s * p.Hq));
    const int d = threadIdx.x * 4;
    const float Ms = (M == -CUDART_INF_F) ? 0.f : M;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    for (int s = 0; s < S; ++s) {
        const float ls = __ldg(lse + (int64_t)s * p.Hq);
        if (ls == -CUDART_INF_F) continue;                 // empty chunk (NaN is kept)
        const float wgt = expf(ls - Ms);
        den += wgt;
        const float4 v = __ldg(reinterpret_cast<const float4*>(
            p.po + ((rc0 + s) * p.Hq + h) * (int64_t)p.D + d));
        acc.x += wgt * v.x;
        acc.y += wgt * v.y;
        acc.z += wgt * v.z;
        acc.w += wgt * v.w;
    }
    const float inv = (den == 0.f) ? 0.f : 1.0f / den;
    uint2 o;
    o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + ((int64_t)b * p.Hq + h) * p.D + d) = o;
}

int launch_combine(const float* partial_o, const float* partial_lse, const ga_plan* plan,
                   const int32_t* seq_lens, void* out, int32_t* err_word, int64_t pt_stride,
                   cudaStream_t stream) {
    CombineParams p;
    p.po = partial_o;
    p.plse = partial_lse;
    p.seq_lens = seq_lens;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.err_word = err_word;
    p.pt_stride = pt_stride;
    p.rc_capacity = plan->row_chunks;
    p.B = plan->batch;
    // an S-query plan has S (query, head) columns per query head, laid out
    // [B, Hq, S, D]: the combine sees them as Hq * S heads
    p.Hq = plan->num_q_heads * plan->q_len;
    p.D = plan->head_dim;
    p.window = effective_window(plan->window, plan->q_len);
    p.mode = plan->mode;
    p.splits = plan->splits;
    p.chunk_pages = plan->chunk_pages;
    if (p.B == 0) return GA_OK;
    dim3 grid(p.Hq, p.B);
    combine_kernel<<<grid, p.D / 4, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GA_OK : GA_ERR_CUDA;
}

}  // namespace ga
