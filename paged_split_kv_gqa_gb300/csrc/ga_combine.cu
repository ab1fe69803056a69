// ga_combine.cu -- the log-sum-exp merge of split-KV partials
// (ga_splitkv_combine; the decode calls launch it after a split decode).
// For row b, column h and the row's chunks s:
//     M = max_s lse_s,  out = sum_s e^{lse_s - M} o_s / sum_s e^{lse_s - M}
// ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is mandatory here":
// flash-decode with split factor 8); the arithmetic is in ga_combine.cuh.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "ga_combine.cuh"
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
    int32_t rows_per_cta;   // consecutive rows of one CTA
};

// One CTA of 4 warps per (4 merge tasks, block of rows_per_cta consecutive
// rows); a task is one column's 128-dim block, taken by one warp
// (merge_warp128).  A CTA finds its first row's first row-chunk from the
// lengths of the rows before it (a strided sum over its 128 threads) and
// steps through its other rows from there.  The host makes row blocks of
// ceil(B / 128) rows, so at most 128 row blocks sum their prefixes: O(B) per
// CTA, O(B * tasks / 4 * 128) in all, at any batch.  Small batches keep one
// row per CTA: wider CTAs (8 warps, 16 tasks) serialised the merges there
// (the ragged 60-layer step at B = 1 took 1.108 ms with them against 0.834 ms
// with these).
constexpr int kCombineWarps = 4;
constexpr int kTasksPerCta = 4;
constexpr int kCombineRowBlocks = 128;

__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(const CombineParams p) {
    const int b0 = blockIdx.y * p.rows_per_cta;
    const int b1 = min(p.B, b0 + p.rows_per_cta);
    __shared__ int32_t s_red[kCombineWarps];
    // row-chunk offset of row b0: chunks of all rows before it
    int32_t part = 0;
    for (int r = threadIdx.x; r < b0; r += blockDim.x)
        part += row_geometry(__ldg(p.seq_lens + r), p.window, p.pt_stride, p.mode, p.splits,
                             p.chunk_pages).chunks;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = part;
    __syncthreads();
    int64_t rc0 = 0;
    for (int wv = 0; wv < kCombineWarps; ++wv) rc0 += s_red[wv];
    const int nb = p.D / 128;
    for (int b = b0; b < b1; ++b) {
        const RowGeom g = row_geometry(__ldg(p.seq_lens + b), p.window, p.pt_stride, p.mode,
                                       p.splits, p.chunk_pages);
        const int S = g.chunks;
        if (S > 1) {                          // (one chunk: written by the decode kernel)
            if (rc0 + S > p.rc_capacity) {
                if (threadIdx.x == 0 && blockIdx.x == 0) report(p.err_word, kErrCapacity);
                return;
            }
            for (int t = blockIdx.x * kTasksPerCta + (threadIdx.x >> 5);
                 t < min(p.Hq * nb, (int)(blockIdx.x + 1) * kTasksPerCta); t += kCombineWarps) {
                const int h = t / nb, d0 = (t % nb) * 128;
                const uint2 o = merge_warp128(p.po, p.plse, rc0, S, p.Hq, p.D, h, d0);
                *reinterpret_cast<uint2*>(p.out + ((int64_t)b * p.Hq + h) * p.D + d0 +
                                          4 * (threadIdx.x & 31)) = o;
            }
        }
        rc0 += S;
    }
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
    p.rows_per_cta = (p.B + kCombineRowBlocks - 1) / kCombineRowBlocks;
    const int tasks = p.Hq * (p.D / 128);
    dim3 grid((tasks + kTasksPerCta - 1) / kTasksPerCta,
              (p.B + p.rows_per_cta - 1) / p.rows_per_cta);
    combine_kernel<<<grid, 32 * kCombineWarps, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GA_OK : GA_ERR_CUDA;
}

}  // namespace ga
