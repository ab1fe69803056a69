// ga_api.cu -- the exported C ABI: argument checks (fail closed before any
// launch), the split-KV planner and the launch of the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <vector>

#include "ga_internal.h"

namespace ga {

// positions null: each row's token goes to seq_lens[b] - 1 (rows of length 0,
// or longer than the table holds, append nothing)
int launch_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                  int32_t kv_dtype, const float* k_scale, const float* v_scale,
                  const int32_t* page_table, int64_t pt_stride, const int32_t* positions,
                  int32_t batch, int32_t num_kv_heads, int32_t head_dim, int64_t num_pages,
                  int32_t* err_word, cudaStream_t stream, const int32_t* seq_lens = nullptr);

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> cached{nullptr};
    EncodeTiledFn f = cached.load();
    if (f) return f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    cached.store(f);
    return f;
}

// The pool viewed as a 3-D tensor (e = elements in one 128-byte row chunk,
// key row, chunk column): strides D*esize bytes per key row and 128 bytes per
// chunk column.  One box {e, 16, D*esize/128} is a whole page-head block and
// lands in shared memory as [chunk column][key row][128 bytes] with the
// 128-byte swizzle, i.e. one 2 KB tile per 128-byte column; box_cols > 0
// narrows the box to that many chunk columns.
int encode_rows_map(CUtensorMap* map, const void* base, int32_t kv_dtype, int64_t rows,
                    int32_t head_dim, int32_t box_rows, int32_t box_cols) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return GA_ERR_CUDA;
    const int esz = kv_dtype == GA_KV_BF16 ? 2 : 1;
    const cuuint32_t e = (cuuint32_t)(128 / esz);
    const cuuint32_t cols = (cuuint32_t)(head_dim * esz / 128);
    const cuuint64_t dims[3] = {(cuuint64_t)e, (cuuint64_t)rows, (cuuint64_t)cols};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * esz, 128};
    const cuuint32_t box[3] = {e, (cuuint32_t)box_rows,
                               box_cols > 0 ? (cuuint32_t)box_cols : cols};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map,
                           kv_dtype == GA_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                           3, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GA_OK : GA_ERR_CUDA;
}

// An E4M3 pool [num_pages, Hkv, 16, D] seen, for one 128-byte region of the
// head dim (bytes 128 * region .. + 127 of every key row), as the 5-D tensor
// (byte e < 128, key % 8, kv head, key / 8, page) with byte strides
// (1, D, 16 D, 8 D, Hkv 16 D).  One box {128, 8, hp, 2, 1} holds that region
// of hp consecutive kv heads of one page and lands as [key / 8][head][key % 8]
// rows of 128 bytes (128-byte swizzle): each head's keys in groups of 8 rows,
// the groups of one head 8 * hp rows apart.
int encode_heads_map(CUtensorMap* map, const void* pool, int32_t region, int32_t num_kv_heads,
                     int64_t num_pages, int32_t head_dim, int32_t hp) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return GA_ERR_CUDA;
    const cuuint64_t D = (cuuint64_t)head_dim;
    const cuuint64_t dims[5] = {128, 8, (cuuint64_t)num_kv_heads, 2, (cuuint64_t)num_pages};
    const cuuint64_t strides[4] = {D, 16 * D, 8 * D, (cuuint64_t)num_kv_heads * 16 * D};
    const cuuint32_t box[5] = {128, 8, (cuuint32_t)hp, 2, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                           const_cast<uint8_t*>(static_cast<const uint8_t*>(pool)) + 128 * region,
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GA_OK : GA_ERR_CUDA;
}

// A pool [num_pages, Hkv, 16, D] (bf16 or E4M3 codes) seen as the 5-D tensor
// (element e of a 128-byte row chunk, key % 8, 128-byte region of the head
// dim, key / 8, page-head block) with byte strides (esize, D esize, 128,
// 8 D esize, 16 D esize).  One box {128 / esize, 8, box_regions, 2, 1} covers
// box_regions consecutive regions of one page-head block and lands as
// [key / 8][region][key % 8] rows of 128 bytes (128-byte swizzle): each
// region's keys in groups of 8 rows, 8 box_regions rows apart.
int encode_region_map(CUtensorMap* map, const void* pool, int32_t kv_dtype, int64_t num_blocks,
                      int32_t head_dim, int32_t box_regions) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return GA_ERR_CUDA;
    const cuuint64_t esz = kv_dtype == GA_KV_BF16 ? 2 : 1;
    const cuuint64_t row = (cuuint64_t)head_dim * esz;        // bytes per key row
    const cuuint64_t dims[5] = {128 / esz, 8, row / 128, 2, (cuuint64_t)num_blocks};
    const cuuint64_t strides[4] = {row, 128, 8 * row, 16 * row};
    const cuuint32_t box[5] = {(cuuint32_t)(128 / esz), 8, (cuuint32_t)box_regions, 2, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(map,
                           kv_dtype == GA_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                           5, const_cast<void*>(pool), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GA_OK : GA_ERR_CUDA;
}

int ensure_smem_attr(const void* func, int bytes, int slot) {
    static std::atomic<uint64_t> done[32];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GA_ERR_CUDA;
    const uint64_t bit = 1ull << (dev & 63);
    if (done[slot].load() & bit) return GA_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return GA_ERR_CUDA;
    done[slot].fetch_or(bit);
    return GA_OK;
}

// ------------------------------------------------------------------ planner

namespace {

struct PlanInput {
    const int32_t* lens;
    int32_t B, Hq, Hkv, D, W, num_sms, S;    // W: the window of the union of S queries
    int32_t TW;                              // columns per work unit
    int32_t HP;                              // kv heads per work unit
    double page_weight;                      // a page-head's bytes relative to bf16
    double unit_ovh;                         // fixed cost of a work unit, in bf16 page-heads
};

// Row-chunk count and per-unit page counts of a candidate chunking.
struct Candidate {
    int32_t mode, splits, chunk_pages;
    int64_t row_chunks = 0, units = 0;
    int32_t max_cp = 0;
    int32_t schedule = kScheduleRoundRobin;
    double cost = 0;
};

void evaluate(const PlanInput& in, Candidate& cand) {
    const int32_t HG = ceil_div(in.Hq / in.Hkv * in.S, in.TW);
    const int64_t per_rc = (int64_t)(in.Hkv / in.HP) * HG;
    std::vector<int32_t> rc_pages;
    rc_pages.reserve(in.B * 4);
    // chunked plans, the rows-by-size deal's order of row-chunks: the full
    // chunks in row order, then the shorter last chunks, longest first
    std::vector<int64_t> full_rc, last_rc;
    int64_t split_rows_rc = 0;
    for (int32_t b = 0; b < in.B; ++b) {
        const RowGeom g = row_geometry(in.lens[b], in.W, INT64_MAX / 64, cand.mode, cand.splits,
                                       cand.chunk_pages);
        cand.max_cp = std::max(cand.max_cp, std::min(g.cp, std::max(g.npages, 1)));
        const int32_t nfull = full_chunks(g);
        for (int32_t j = 0; j < g.chunks; ++j) {
            int32_t p0, np;
            chunk_pages_of(g, j, &p0, &np);
            (j < nfull ? full_rc : last_rc).push_back((int64_t)rc_pages.size());
            rc_pages.push_back(np);
        }
        if (g.chunks > 1) split_rows_rc += g.chunks;
    }
    cand.row_chunks = (int64_t)rc_pages.size();
    cand.units = cand.row_chunks * per_rc;
    // Static round-robin schedule of the persistent grid: unit u -> CTA u % G.
    // Cost in "page loads per SM" (bf16 page-head blocks): each unit costs its
    // pages (times its kv heads, weighted by the KV element size) plus a fixed
    // overhead (in.unit_ovh); a split adds the partial round trip spread over
    // all SMs plus one extra launch.  (With 2 pages of overhead the ragged
    // 256-row global family got 32-page chunks, 6411 GB/s; 64-page chunks
    // measure 6559 GB/s.)
    const int64_t G = std::max<int64_t>(1, std::min<int64_t>(cand.units, in.num_sms));
    const double unit_ovh = in.unit_ovh;
    std::vector<double> load((size_t)G, 0.0);
    for (int64_t u = 0; u < cand.units; ++u) {
        const int64_t rc = u / per_rc;
        load[(size_t)(u % G)] += rc_pages[(size_t)rc] * in.HP * in.page_weight + unit_ovh;
    }
    double makespan = 0;
    for (double v : load) makespan = std::max(makespan, v);
    // The rows-by-size deal (longest first, every other pass over the CTAs
    // reversed) when it evens the CTA loads out by more than 3 %: one chunk
    // per row (the ragged 256-row sliding family: 213 against 238
    // superstages on the busiest CTA), or fixed-size chunks with the rows'
    // shorter last chunks sorted after the full ones (the 31B global family
    // on E4M3 pools, 256-page chunks: 2123 against 2304 pages).  Simulated
    // here exactly as the kernels deal it.
    cand.schedule = kScheduleRoundRobin;
    const bool sortable = cand.mode == kSplitNone ? sorted_schedule_fits(in.B)
                          : cand.mode == kSplitChunk && sorted_chunk_schedule_fits(in.B);
    if (sortable && in.S == 1 && cand.units > G) {
        std::vector<int64_t> order;           // row-chunks in the deal's order
        if (cand.mode == kSplitNone) {
            for (int32_t b = 0; b < in.B; ++b) order.push_back(b);
        } else {
            order = full_rc;
            order.insert(order.end(), last_rc.begin(), last_rc.end());
        }
        std::stable_sort(order.begin() + (cand.mode == kSplitNone ? 0 : (int64_t)full_rc.size()),
                         order.end(), [&](int64_t a, int64_t b) {
                             return row_sort_key(rc_pages[(size_t)a]) <
                                    row_sort_key(rc_pages[(size_t)b]);
                         });
        std::vector<double> sorted_load((size_t)G, 0.0);
        for (int64_t u = 0; u < cand.units; ++u) {
            const uint32_t pos = snake_position((uint32_t)u, (uint32_t)G, (uint32_t)cand.units);
            const int64_t rc = order[(size_t)(pos / per_rc)];
            sorted_load[(size_t)(u % G)] += rc_pages[(size_t)rc] * in.HP * in.page_weight + unit_ovh;
        }
        double sorted_span = 0;
        for (double v : sorted_load) sorted_span = std::max(sorted_span, v);
        if (sorted_span < 0.97 * makespan) {
            makespan = sorted_span;
            cand.schedule = kScheduleSorted;
        }
    }
    double combine = 0;
    if (split_rows_rc > 0) {
        const double page_bytes = 2.0 * kPageSize * in.D * 2.0;   // K + V page-head, bf16
        const double partial_bytes = 2.0 * (double)split_rows_rc * in.Hq * in.S * in.D * 4.0;
        combine = partial_bytes / page_bytes / in.num_sms + 4.0;
    }
    cand.cost = makespan + combine;
}

}  // namespace

}  // namespace ga

using namespace ga;

extern "C" {

int32_t ga_version(void) { return 0x000400; }

const char* ga_strerror(int status) {
    switch (status) {
        case GA_OK: return "GA_OK";
        case GA_ERR_INVALID_ARG: return "GA_ERR_INVALID_ARG: invalid argument";
        case GA_ERR_UNSUPPORTED: return "GA_ERR_UNSUPPORTED: unsupported configuration";
        case GA_ERR_WORKSPACE_TOO_SMALL: return "GA_ERR_WORKSPACE_TOO_SMALL: workspace too small";
        case GA_ERR_CUDA: return "GA_ERR_CUDA: CUDA call or kernel launch failed";
        case GA_ERR_DEVICE_CHECK: return "GA_ERR_DEVICE_CHECK: a kernel reported invalid device data";
        default: return "unknown ga status";
    }
}

int ga_check_error_word(int32_t word) { return word == 0 ? GA_OK : GA_ERR_DEVICE_CHECK; }

int ga_plan_splits(const int32_t* seq_lens_host, int32_t batch, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, int32_t window, int32_t page_size,
                   int32_t num_sms, int32_t requested_splits, int32_t fixed_chunk_tokens,
                   int32_t flags, ga_plan* plan_out) {
    return ga_plan_splits_mq(seq_lens_host, batch, num_q_heads, num_kv_heads, head_dim, window,
                             page_size, 1, num_sms, requested_splits, fixed_chunk_tokens, flags,
                             plan_out);
}

int ga_plan_splits_mq(const int32_t* seq_lens_host, int32_t batch, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t window, int32_t page_size,
                      int32_t q_len, int32_t num_sms, int32_t requested_splits,
                      int32_t fixed_chunk_tokens, int32_t flags, ga_plan* plan_out) {
    if (plan_out == nullptr || batch < 0 || (batch > 0 && seq_lens_host == nullptr))
        return GA_ERR_INVALID_ARG;
    if (q_len < 1) return GA_ERR_INVALID_ARG;
    if (q_len > kMaxQLen) return GA_ERR_UNSUPPORTED;
    static_assert(GA_PLAN_KV_E4M3 == kPlanKvE4m3, "plan flag");
    const int32_t known_flags = GA_PLAN_TOUCH_LOG | GA_PLAN_EXTERNAL_COMBINE |
                                GA_PLAN_TEST_WAIT_TIMEOUT | GA_PLAN_TENSOR_CORE_UNITS |
                                GA_PLAN_COLUMN_PARALLEL_UNITS | GA_PLAN_KV_E4M3;
    if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || window < 0 ||
        num_sms < 1 || requested_splits < 0 || fixed_chunk_tokens < 0 ||
        (requested_splits > 0 && fixed_chunk_tokens > 0) || (flags & ~known_flags) ||
        ((flags & GA_PLAN_TENSOR_CORE_UNITS) && (flags & GA_PLAN_COLUMN_PARALLEL_UNITS)))
        return GA_ERR_INVALID_ARG;
    if (batch > kMaxBatch) return GA_ERR_UNSUPPORTED;
    if (head_dim != 256 && head_dim != 512) return GA_ERR_UNSUPPORTED;
    if (page_size != kPageSize) return GA_ERR_UNSUPPORTED;
    if (fixed_chunk_tokens % page_size != 0) return GA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b)
        if (seq_lens_host[b] < 0) return GA_ERR_INVALID_ARG;

    const int32_t weff = effective_window(window, q_len);
    // more than 8 (query, head) columns per kv head: units of 64 columns for
    // the tensor-core kernel, or column-parallel units of 4 tiles of 8 (every
    // page read once for all of them)
    const int32_t cols = num_q_heads / num_kv_heads * q_len;
    const bool tc = (flags & GA_PLAN_TENSOR_CORE_UNITS) ||
                    (!(flags & GA_PLAN_COLUMN_PARALLEL_UNITS) && cols >= tc_min_cols(head_dim));
    // (E4M3 pools run the tcgen05 E4M3 kernel, whose units hold 8 columns,
    // or 16 for a kv head with more than 8: a plan made for them is costed
    // with those units, and asks the kernel for 16-column ones)
    const int32_t tw = (flags & GA_PLAN_KV_E4M3) ? (cols > kHeadTile ? 2 * kHeadTile : kHeadTile)
                       : cols <= kHeadTile       ? kHeadTile
                       : tc                      ? kTcColTile
                                                 : 4 * kHeadTile;
    // A unit's fixed cost: the page-parallel kernels' merge and pipeline
    // refill (~3.5K cycles, about 4 pages of stream time); the tcgen05 E4M3
    // kernels' unit start and drain (q preparation, the first superstage's
    // products, the epilogue from tensor memory: one-page rows measure ~6 us
    // a unit, about 18 bf16 pages; with 4 the ragged batch's first 4 rows got
    // 16-page chunks, 19.2 us a layer with the combine, against 15.6 unsplit).
    const bool e4m3 = (flags & GA_PLAN_KV_E4M3) != 0;
    PlanInput in{seq_lens_host, batch, num_q_heads, num_kv_heads, head_dim, weff, num_sms, q_len,
                 tw, 1, e4m3 ? 0.5 : 1.0, e4m3 ? 18.0 : 4.0};
    Candidate best;
    if (requested_splits == 1) {
        best = Candidate{kSplitNone, 0, 0};
        evaluate(in, best);
    } else if (requested_splits > 1) {
        best = Candidate{kSplitCount, requested_splits, 0};
        evaluate(in, best);
    } else if (fixed_chunk_tokens > 0) {
        best = Candidate{kSplitChunk, 0, fixed_chunk_tokens / page_size};
        evaluate(in, best);
    } else {
        best = Candidate{kSplitNone, 0, 0};
        evaluate(in, best);
        int32_t max_np = 0;
        for (int32_t b = 0; b < batch; ++b)
            max_np = std::max(max_np,
                              row_geometry(seq_lens_host[b], weff, INT64_MAX / 64, kSplitNone,
                                           0, 0).npages);
        for (int32_t cp = 4; cp < max_np; cp *= 2) {
            Candidate c{kSplitChunk, 0, cp};
            evaluate(in, c);
            if (c.cost < best.cost * 0.98) best = c;
        }
    }
    // E4M3 sliding family: units of several kv heads when the one-head plan
    // needs no split and the wider units alone fill at least four rounds of
    // the SMs (measured on the ragged 256-row batch: 4-head units 5884 vs 5580
    // GB/s; on 128 rows, 31B or 12B batches, or whenever they forced a split,
    // they were slower)
    int32_t hp = 1;
    const int32_t hp_rule = tc_heads_per_unit(flags, head_dim, q_len,
                                              num_q_heads / num_kv_heads, num_kv_heads);
    if (hp_rule > 1 && best.mode == kSplitNone &&
        best.row_chunks * (num_kv_heads / hp_rule) >= 4 * (int64_t)num_sms) {
        hp = hp_rule;
        in.HP = hp;
        in.TW = kHeadTile;
        evaluate(in, best);
    }
    ga_plan p{};
    p.kv_heads_per_unit = hp;
    static_assert(GA_SCHEDULE_ROWS_BY_SIZE == kScheduleSorted &&
                      GA_SCHEDULE_ROUND_ROBIN == kScheduleRoundRobin, "schedule ids");
    p.schedule = best.schedule;
    p.mode = best.mode;
    p.splits = best.splits;
    p.chunk_pages = best.chunk_pages;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.window = window;
    p.page_size = page_size;
    p.flags = flags;
    p.q_len = q_len;
    p.col_tile = tw;
    p.row_chunks = best.row_chunks;
    p.units = best.units;
    p.grid = (int32_t)std::max<int64_t>(1, std::min<int64_t>(best.units, num_sms));
    int64_t off = 0;
    auto take = [&off](int64_t bytes) {
        const int64_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    if (p.mode != kSplitNone) {
        p.partial_o_offset = take(p.row_chunks * num_q_heads * (int64_t)q_len * head_dim * 4);
        p.partial_lse_offset = take(p.row_chunks * num_q_heads * (int64_t)q_len * 4);
    }
    if (flags & GA_PLAN_TOUCH_LOG) {
        p.touch_stride = std::max(best.max_cp, 1);
        p.touch_log_offset = take(p.row_chunks * (int64_t)p.touch_stride * 4);
    }
    p.workspace_bytes = off;
    *plan_out = p;
    return GA_OK;
}

int ga_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                 int32_t kv_dtype, const float* k_scale, const float* v_scale,
                 const int32_t* page_table, int64_t pt_stride, const int32_t* positions,
                 int32_t batch, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                 int64_t num_pages, int32_t* err_word, ga_stream_t stream) {
    if (batch < 0 || num_kv_heads < 1 || pt_stride < 1 || num_pages < 1) return GA_ERR_INVALID_ARG;
    if (kv_dtype != GA_KV_BF16 && kv_dtype != GA_KV_E4M3) return GA_ERR_UNSUPPORTED;
    if (head_dim != 256 && head_dim != 512) return GA_ERR_UNSUPPORTED;
    if (page_size != kPageSize) return GA_ERR_UNSUPPORTED;
    if (batch == 0) return GA_OK;
    if (!k_new || !v_new || !k_pool || !v_pool || !page_table || !positions)
        return GA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return GA_ERR_INVALID_ARG;
    if (kv_dtype == GA_KV_E4M3 && (!k_scale || !v_scale)) return GA_ERR_INVALID_ARG;
    return launch_append(k_new, v_new, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table,
                         pt_stride, positions, batch, num_kv_heads, head_dim, num_pages,
                         err_word, reinterpret_cast<cudaStream_t>(stream));
}

static int decode_entry(const void* q, const void* k_pool, const void* v_pool, int32_t kv_dtype,
                        const float* k_scale, const float* v_scale, const int32_t* page_table,
                        int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t window, int32_t page_size, int64_t num_pages, float scale,
                        const ga_plan* plan, void* workspace, size_t workspace_bytes, void* out,
                        int32_t* err_word, ga_stream_t stream, const void* k_new = nullptr,
                        const void* v_new = nullptr) {
    if (plan == nullptr || batch < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || pt_stride < 1 || num_pages < 1 ||
        !std::isfinite(scale))
        return GA_ERR_INVALID_ARG;
    if (kv_dtype != GA_KV_BF16 && kv_dtype != GA_KV_E4M3) return GA_ERR_UNSUPPORTED;
    if (page_size != kPageSize) return GA_ERR_UNSUPPORTED;
    if (batch > kMaxBatch) return GA_ERR_UNSUPPORTED;
    if (num_pages * num_kv_heads * (int64_t)kPageSize >= (int64_t(1) << 31))
        return GA_ERR_UNSUPPORTED;
    if (plan->batch != batch || plan->num_q_heads != num_q_heads ||
        plan->num_kv_heads != num_kv_heads || plan->head_dim != head_dim ||
        plan->window != window || plan->page_size != page_size || plan->q_len < 1 ||
        plan->q_len > kMaxQLen ||
        (plan->col_tile != kHeadTile && plan->col_tile != 4 * kHeadTile &&
         plan->col_tile != kTcColTile &&
         (plan->col_tile != 2 * kHeadTile || kv_dtype != GA_KV_E4M3)))
        return GA_ERR_INVALID_ARG;
    if (batch == 0) return GA_OK;
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out) return GA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return GA_ERR_INVALID_ARG;
    if (kv_dtype == GA_KV_E4M3 && (!k_scale || !v_scale)) return GA_ERR_INVALID_ARG;
    if (plan->workspace_bytes > 0) {
        if (!workspace || !aligned16(workspace)) return GA_ERR_INVALID_ARG;
        if ((int64_t)workspace_bytes < plan->workspace_bytes) return GA_ERR_WORKSPACE_TOO_SMALL;
    }
    // kv heads per unit: 0 or 1, or the wider units the geometry allows
    if (plan->kv_heads_per_unit > 1 &&
        plan->kv_heads_per_unit != tc_heads_per_unit(plan->flags, head_dim, plan->q_len,
                                                     num_q_heads / num_kv_heads, num_kv_heads))
        return GA_ERR_INVALID_ARG;
    if (plan->kv_heads_per_unit < 0) return GA_ERR_INVALID_ARG;
    const bool append = k_new != nullptr || v_new != nullptr;
    if (append && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new) ||
                   plan->q_len != 1))
        return GA_ERR_INVALID_ARG;
    DecodeArgs a{q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride, seq_lens,
                 batch, num_q_heads, num_kv_heads, head_dim, window, num_pages, scale, plan,
                 workspace, out, err_word, reinterpret_cast<cudaStream_t>(stream)};
    if (append) {
        // (the E4M3 kernel's 16-column units hold a kv head of up to 16 query heads)
        const int32_t unit_cols =
            kv_dtype == GA_KV_E4M3 && plan->col_tile == 2 * kHeadTile ? 2 * kHeadTile : kHeadTile;
        if (num_q_heads / num_kv_heads <= unit_cols && plan->col_tile != kTcColTile) {
            // every kv head of a row chunk is one unit of a kernel that
            // appends: the decode appends
            a.k_new = k_new;
            a.v_new = v_new;
        } else {
            // a kv head spans several units: append first, then decode
            const int rc = launch_append(k_new, v_new, const_cast<void*>(k_pool),
                                         const_cast<void*>(v_pool), kv_dtype, k_scale, v_scale,
                                         page_table, pt_stride, nullptr, batch, num_kv_heads,
                                         head_dim, num_pages, err_word, a.stream, seq_lens);
            if (rc != GA_OK) return rc;
        }
    }
    return launch_decode(a);
}

int ga_decode_local_hd256(const void* q, const void* k_pool, const void* v_pool,
                          int32_t kv_dtype, const float* k_scale, const float* v_scale,
                          const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t window, int32_t page_size, int64_t num_pages, float scale,
                          const ga_plan* plan, void* workspace, size_t workspace_bytes,
                          void* out, int32_t* err_word, ga_stream_t stream) {
    if (window < 1) return GA_ERR_INVALID_ARG;
    return decode_entry(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride,
                        seq_lens, batch, num_q_heads, num_kv_heads, 256, window, page_size,
                        num_pages, scale, plan, workspace, workspace_bytes, out, err_word,
                        stream);
}

int ga_decode_global_hd512(const void* q, const void* k_pool, const void* v_pool,
                           int32_t kv_dtype, const float* k_scale, const float* v_scale,
                           const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                           int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t page_size, int64_t num_pages, float scale,
                           const ga_plan* plan, void* workspace, size_t workspace_bytes,
                           void* out, int32_t* err_word, ga_stream_t stream) {
    return decode_entry(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride,
                        seq_lens, batch, num_q_heads, num_kv_heads, 512, 0, page_size,
                        num_pages, scale, plan, workspace, workspace_bytes, out, err_word,
                        stream);
}

int ga_decode_local_hd256_append(const void* k_new, const void* v_new, const void* q,
                                 void* k_pool, void* v_pool, int32_t kv_dtype,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* page_table, int64_t pt_stride,
                                 const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t window, int32_t page_size,
                                 int64_t num_pages, float scale, const ga_plan* plan,
                                 void* workspace, size_t workspace_bytes, void* out,
                                 int32_t* err_word, ga_stream_t stream) {
    if (window < 1 || !k_new || !v_new) return GA_ERR_INVALID_ARG;
    return decode_entry(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride,
                        seq_lens, batch, num_q_heads, num_kv_heads, 256, window, page_size,
                        num_pages, scale, plan, workspace, workspace_bytes, out, err_word,
                        stream, k_new, v_new);
}

int ga_decode_global_hd512_append(const void* k_new, const void* v_new, const void* q,
                                  void* k_pool, void* v_pool, int32_t kv_dtype,
                                  const float* k_scale, const float* v_scale,
                                  const int32_t* page_table, int64_t pt_stride,
                                  const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t page_size, int64_t num_pages,
                                  float scale, const ga_plan* plan, void* workspace,
                                  size_t workspace_bytes, void* out, int32_t* err_word,
                                  ga_stream_t stream) {
    if (!k_new || !v_new) return GA_ERR_INVALID_ARG;
    return decode_entry(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride,
                        seq_lens, batch, num_q_heads, num_kv_heads, 512, 0, page_size,
                        num_pages, scale, plan, workspace, workspace_bytes, out, err_word,
                        stream, k_new, v_new);
}

int ga_splitkv_combine(const float* partial_o, const float* partial_lse, const ga_plan* plan,
                       const int32_t* seq_lens, int64_t pt_stride, void* out,
                       int32_t* err_word, ga_stream_t stream) {
    if (plan == nullptr || pt_stride < 1 || plan->q_len < 1 || plan->q_len > kMaxQLen)
        return GA_ERR_INVALID_ARG;
    if (plan->head_dim != 256 && plan->head_dim != 512) return GA_ERR_UNSUPPORTED;
    if (plan->batch == 0 || plan->mode == GA_SPLIT_NONE) return GA_OK;
    if (!partial_o || !partial_lse || !seq_lens || !out) return GA_ERR_INVALID_ARG;
    if (!aligned16(partial_o) || !aligned16(out)) return GA_ERR_INVALID_ARG;
    return launch_combine(partial_o, partial_lse, plan, seq_lens, out, err_word, pt_stride,
                          reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
