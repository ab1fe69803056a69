// ga_combine.cuh -- the log-sum-exp merge of split-KV partials: the
// arithmetic, written once with every rounding step spelled out, in a
// latency-friendly warp form and a plain per-thread form that give the same
// bits.
//
// For row b, (query, head) column h and the row's chunks s = 0 .. S-1:
//     M = max_s lse_s,  w_s = e^{lse_s - M},  out = sum_s w_s o_s / sum_s w_s
// ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is mandatory here":
// flash-decode with split factor 8).  o_s is normalised within its chunk and
// lse_s is the chunk's natural-log log-sum-exp; empty chunks carry -inf and
// weigh nothing; a NaN partial reaches the output.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>

#include "ga_device.cuh"

namespace ga {

__device__ __forceinline__ float ld_part(const float* a) { return __ldg(a); }
__device__ __forceinline__ float4 ld_part4(const float* a) {
    return __ldg(reinterpret_cast<const float4*>(a));
}

// Dims d .. d+3 of column h: partial o at po[(rc0 + s) * Hq + h][D], lse at
// plse[(rc0 + s) * Hq + h].  Returns the four outputs packed as bf16.  Every
// rounding step is spelled out so that merge_warp128 computes the same bits.
__device__ __forceinline__ uint2 merge_chunks4(const float* po, const float* plse, int64_t rc0,
                                               int S, int64_t Hq, int D, int64_t h, int d) {
    const float* lse = plse + rc0 * Hq + h;
    float M = -CUDART_INF_F;
    for (int s = 0; s < S; ++s) M = fmaxf(M, ld_part(lse + (int64_t)s * Hq));
    const float Ms = (M == -CUDART_INF_F) ? 0.f : M;
    float ax = 0.f, ay = 0.f, az = 0.f, aw = 0.f, den = 0.f;
    for (int s = 0; s < S; ++s) {
        const float ls = ld_part(lse + (int64_t)s * Hq);
        if (ls == -CUDART_INF_F) continue;                 // empty chunk (NaN is kept)
        const float wgt = expf(__fsub_rn(ls, Ms));
        den = __fadd_rn(den, wgt);
        const float4 v = ld_part4(po + ((rc0 + s) * Hq + h) * (int64_t)D + d);
        ax = __fmaf_rn(wgt, v.x, ax);
        ay = __fmaf_rn(wgt, v.y, ay);
        az = __fmaf_rn(wgt, v.z, az);
        aw = __fmaf_rn(wgt, v.w, aw);
    }
    const float inv = (den == 0.f) ? 0.f : __fdiv_rn(1.0f, den);
    uint2 o;
    o.x = pack_bf16x2(__fmul_rn(ax, inv), __fmul_rn(ay, inv));
    o.y = pack_bf16x2(__fmul_rn(az, inv), __fmul_rn(aw, inv));
    return o;
}

// Weights of the fast path held by one lane: chunks s = lane and s = lane + 32.
constexpr int kMergeWarpMaxChunks = 64;
// Marks a chunk whose lse is -inf (empty): it is skipped, as in merge_chunks4
// (no weight produced by expf is negative).
constexpr float kSkipChunk = -1.0f;

// One warp merges the 128 dims [d0, d0 + 128) of column h; lane l returns dims
// d0 + 4l .. d0 + 4l + 3 packed as bf16.  The arithmetic is merge_chunks4's,
// step for step (the same maximum, weights, sums in chunk order and
// rounding), so both give the same bits; what changes is latency: the
// chunks' log-sum-exps are read once per warp (one per lane), their weights
// are shared by shuffles, and the partials are read 8 chunks at a time with
// independent loads.  Rows with more than kMergeWarpMaxChunks chunks take
// merge_chunks4 itself.
__device__ __forceinline__ uint2 merge_warp128(const float* po, const float* plse, int64_t rc0,
                                               int S, int64_t Hq, int D, int64_t h, int d0) {
    const int lane = threadIdx.x & 31;
    if (S > kMergeWarpMaxChunks)
        return merge_chunks4(po, plse, rc0, S, Hq, D, h, d0 + 4 * lane);
    const float* lse = plse + rc0 * Hq + h;
    const float l0 = lane < S ? ld_part(lse + (int64_t)lane * Hq) : -CUDART_INF_F;
    const float l1 =
        lane + 32 < S ? ld_part(lse + (int64_t)(lane + 32) * Hq) : -CUDART_INF_F;
    // the maximum ignores NaN (fmaxf), like merge_chunks4's running maximum
    float M = fmaxf(fmaxf(-CUDART_INF_F, l0), l1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Ms = (M == -CUDART_INF_F) ? 0.f : M;
    const float w0 = (l0 == -CUDART_INF_F) ? kSkipChunk : expf(__fsub_rn(l0, Ms));
    const float w1 = (l1 == -CUDART_INF_F) ? kSkipChunk : expf(__fsub_rn(l1, Ms));
    auto weight = [&](int s) {            // s is warp-uniform
        return __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
    };
    float den = 0.f;
    for (int s = 0; s < S; ++s) {
        const float ws = weight(s);
        if (ws != kSkipChunk) den = __fadd_rn(den, ws);
    }
    const float inv = (den == 0.f) ? 0.f : __fdiv_rn(1.0f, den);
    const float* base = po + (rc0 * Hq + h) * (int64_t)D + d0 + 4 * lane;
    const int64_t step = Hq * (int64_t)D;
    float ax = 0.f, ay = 0.f, az = 0.f, aw = 0.f;
    for (int s0 = 0; s0 < S; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (s0 + j < S) v[j] = ld_part4(base + (int64_t)(s0 + j) * step);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j < S) {
                const float ws = weight(s0 + j);
                if (ws != kSkipChunk) {
                    ax = __fmaf_rn(ws, v[j].x, ax);
                    ay = __fmaf_rn(ws, v[j].y, ay);
                    az = __fmaf_rn(ws, v[j].z, az);
                    aw = __fmaf_rn(ws, v[j].w, aw);
                }
            }
        }
    }
    uint2 o;
    o.x = pack_bf16x2(__fmul_rn(ax, inv), __fmul_rn(ay, inv));
    o.y = pack_bf16x2(__fmul_rn(az, inv), __fmul_rn(aw, inv));
    return o;
}

}  // namespace ga
