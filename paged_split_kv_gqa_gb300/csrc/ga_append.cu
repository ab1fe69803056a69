// ga_append.cu -- write this step's new token into its KV page slot.
//
// Row b's token goes to page page_table[b][pos_b / P], slot pos_b % P, for
// every kv head ("[Model] Gemma 4 M1 12B", Description: paged prefill and
// decode).  The E4M3 pool of the sliding family stores
// E4M3FN(RNE, saturate-to-finite)(fp32(x) / scale[c]) ("[Model] Gemma 4 M2
// 26B-A4B", Proposed Plan: opt-in FP8 KV pool for the sliding family).  The
// page offset comes from the shared checked helper.
#include <cuda_runtime.h>

#include "ga_device.cuh"
#include "ga_internal.h"

namespace ga {

struct AppendParams {
    const uint4* k_new;      // [B, Hkv, D] bf16, 8 elements per uint4
    const uint4* v_new;
    void* k_pool;
    void* v_pool;
    const float* k_scale;
    const float* v_scale;
    const int32_t* page_table;
    const int32_t* positions;   // or null: the position is seq_lens[b] - 1
    const int32_t* seq_lens;
    int32_t* err_word;
    int64_t pt_stride;
    int64_t num_pages;
    int32_t B, Hkv, D, kv_dtype;
};

// One thread per 8 consecutive elements of one (row, kv head).
__global__ void __launch_bounds__(128) append_kernel(const AppendParams p) {
    const int per_head = p.D / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)p.B * p.Hkv * per_head) return;
    const int d8 = (int)(idx % per_head);
    const int c = (int)((idx / per_head) % p.Hkv);
    const int b = (int)(idx / ((int64_t)per_head * p.Hkv));
    int32_t pos;
    if (p.positions != nullptr) {
        pos = __ldg(p.positions + b);
    } else {
        // one-query decode step: the token at L - 1; an empty row appends
        // nothing, and a length the table cannot hold is the decode's to report
        const int32_t L = __ldg(p.seq_lens + b);
        if ((int64_t)L > p.pt_stride * kPageSize) return;
        pos = L - 1;
    }
    if (pos < 0) return;
    const int64_t lp = pos / kPageSize;
    if (lp >= p.pt_stride) {
        if (c == 0 && d8 == 0) report(p.err_word, kErrPosition);
        return;
    }
    const int32_t page = __ldg(p.page_table + (int64_t)b * p.pt_stride + lp);
    if (!page_ok(page, p.num_pages)) {
        if (c == 0 && d8 == 0) report(p.err_word, kErrPosition);
        return;
    }
    const int64_t elem = page_block_elem(page, c, p.Hkv, p.D) +
                         (int64_t)(pos % kPageSize) * p.D + (int64_t)d8 * 8;
    const uint4 kx = __ldg(p.k_new + idx);
    const uint4 vx = __ldg(p.v_new + idx);
    if (p.kv_dtype == GA_KV_BF16) {
        reinterpret_cast<uint4*>(p.k_pool)[elem / 8] = kx;
        reinterpret_cast<uint4*>(p.v_pool)[elem / 8] = vx;
    } else {
        reinterpret_cast<uint2*>(p.k_pool)[elem / 8] = quantize8(kx, __ldg(p.k_scale + c));
        reinterpret_cast<uint2*>(p.v_pool)[elem / 8] = quantize8(vx, __ldg(p.v_scale + c));
    }
}

int launch_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                  int32_t kv_dtype, const float* k_scale, const float* v_scale,
                  const int32_t* page_table, int64_t pt_stride, const int32_t* positions,
                  int32_t batch, int32_t num_kv_heads, int32_t head_dim, int64_t num_pages,
                  int32_t* err_word, cudaStream_t stream, const int32_t* seq_lens) {
    AppendParams p;
    p.seq_lens = seq_lens;
    p.k_new = static_cast<const uint4*>(k_new);
    p.v_new = static_cast<const uint4*>(v_new);
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.page_table = page_table;
    p.positions = positions;
    p.err_word = err_word;
    p.pt_stride = pt_stride;
    p.num_pages = num_pages;
    p.B = batch;
    p.Hkv = num_kv_heads;
    p.D = head_dim;
    p.kv_dtype = kv_dtype;
    const int64_t n = (int64_t)batch * num_kv_heads * (head_dim / 8);
    if (n == 0) return GA_OK;
    append_kernel<<<(unsigned)((n + 127) / 128), 128, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? GA_OK : GA_ERR_CUDA;
}

}  // namespace ga
