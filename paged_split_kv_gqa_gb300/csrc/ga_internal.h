// ga_internal.h -- host-side declarations shared by the library's translation
// units (argument checks, tensor-map encoding, kernel launchers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ga.h"
#include "ga_geometry.h"

namespace ga {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Everything one decode launch needs, already validated on the host.
struct DecodeArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    int32_t kv_dtype;
    const float* k_scale;
    const float* v_scale;
    const int32_t* page_table;
    int64_t pt_stride;
    const int32_t* seq_lens;
    int32_t batch, num_q_heads, num_kv_heads, head_dim, window;
    int64_t num_pages;
    float scale;
    const ga_plan* plan;
    void* workspace;
    void* out;
    int32_t* err_word;
    cudaStream_t stream;
    // this step's token [B, Hkv, D] bf16, written by the decode kernel itself
    // at position seq_lens[b] - 1 before it reads that page, or null
    const void* k_new = nullptr;
    const void* v_new = nullptr;
};

// Builds a 3-D tensor map over a row-major [rows, D] array (a KV pool as
// [num_pages * Hkv * P, D], or q as [B * Hq, D]) whose box is box_rows rows:
// D * elem / 128 tiles of [box_rows][128 bytes], 128-byte swizzled (box_cols
// > 0: only that many 128-byte columns per box).
int encode_rows_map(CUtensorMap* map, const void* base, int32_t kv_dtype, int64_t rows,
                    int32_t head_dim, int32_t box_rows, int32_t box_cols = 0);

// Builds the 5-D tensor map of one 128-byte region of an E4M3 pool whose box
// is one page of hp consecutive kv heads ([key / 8][head][key % 8] rows).
int encode_heads_map(CUtensorMap* map, const void* pool, int32_t region, int32_t num_kv_heads,
                     int64_t num_pages, int32_t head_dim, int32_t hp);

// Builds the 5-D tensor map of a pool whose box is box_regions consecutive
// 128-byte regions of one page-head block, landing as [key / 8][region]
// [key % 8] rows of 128 bytes.
int encode_region_map(CUtensorMap* map, const void* pool, int32_t kv_dtype, int64_t num_blocks,
                      int32_t head_dim, int32_t box_regions);

int launch_decode(const DecodeArgs& a);

// Decode over an E4M3 pool (hd256 sliding window, hd512 global with two
// pools) on tcgen05 tensor cores.
int launch_decode_tc(const DecodeArgs& a);

// Multi-query decode over two bf16 pools (64 (query, head) columns per unit)
// on tcgen05 tensor cores.
int launch_mq_tc(const DecodeArgs& a);

int launch_combine(const float* partial_o, const float* partial_lse, const ga_plan* plan,
                   const int32_t* seq_lens, void* out, int32_t* err_word, int64_t pt_stride,
                   cudaStream_t stream);

// Sets the dynamic shared-memory limit of `func` once per device (slot < 32
// identifies the kernel).
int ensure_smem_attr(const void* func, int bytes, int slot);

}  // namespace ga
