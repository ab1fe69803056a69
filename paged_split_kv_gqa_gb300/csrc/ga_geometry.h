// ga_geometry.h -- the one home of paged-KV index arithmetic, shared by the
// host planner and every kernel (append, decode, combine).
//
// Page offsets go through these checked helpers only, never re-derived by
// hand in a kernel ("[Model] Gemma 4 M2 26B-A4B", Proposed Plan: route the
// hand-derived page offsets through the checked helper; give the paged-KV
// launch bodies one home so the hd512 twin is not hand-copied).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define GA_HD __host__ __device__ __forceinline__
#else
#define GA_HD inline
#endif

namespace ga {

constexpr int kPageSize = 16;     // keys per page; one page = one 16-key MMA tile
constexpr int kHeadTile = 8;      // query heads per unit (MMA N)
constexpr int kMaxBatch = 2048;   // rows per call (decode keeps a row prefix in smem)
constexpr int kMaxQLen = 64;      // query tokens per row of a multi-query decode
constexpr int kTcColTile = 64;    // (query, head) columns per unit of the tensor-core
                                  // multi-query kernel (N of its products)

// Columns per kv head from which a plan uses tensor-core units by default
// (measured on the 31B-shaped batch: at hd512 32 columns already run faster
// on tcgen05, at hd256 the column-parallel kernel stays ahead up to 32).
GA_HD int32_t tc_min_cols(int32_t head_dim) { return head_dim == 512 ? 32 : 64; }

// Plan flag: the plan is for E4M3 pools (GA_PLAN_KV_E4M3).
constexpr int32_t kPlanKvE4m3 = 32;

// KV heads per work unit of the E4M3 tensor-core decode: 8 / group for the
// sliding family (head_dim 256, one query per row, GQA group 2 or 4, Hkv a
// multiple of it) when the plan was made for E4M3 pools; else 1.  The unit's
// 8 (query, head) columns are then the query heads of those kv heads.
GA_HD int32_t tc_heads_per_unit(int32_t plan_flags, int32_t head_dim, int32_t q_len,
                                int32_t group, int32_t num_kv_heads) {
    if (!(plan_flags & kPlanKvE4m3) || head_dim != 256 || q_len != 1) return 1;
    if (group != 2 && group != 4) return 1;
    const int32_t hp = 8 / group;
    return num_kv_heads % hp == 0 ? hp : 1;
}

enum { kSplitNone = 0, kSplitCount = 1, kSplitChunk = 2 };

// How a persistent grid of G CTAs walks the U work units.  CTA i takes slots
// i, i + G, i + 2G, ...  Round robin (kScheduleRoundRobin): slot = unit.
// Rows by size (kScheduleSorted, one-chunk plans of one-query decodes): the
// units are taken row by row in descending order of the row's attended
// pages (ties in row order), and every odd pass over the G CTAs runs
// backwards, so the CTA that took the largest unit of one pass takes the
// smallest of the next (a longest-first, snake-order deal of unequal units).
enum { kScheduleRoundRobin = 0, kScheduleSorted = 1 };
// The kernels' own id for the rows-by-size deal of a chunked plan (the plan
// says kScheduleSorted; the unit lookup and the chunk index then differ).
constexpr int kScheduleSortedChunks = 2;

GA_HD int32_t kernel_schedule(int32_t plan_schedule, int32_t mode) {
    return plan_schedule == kScheduleSorted && mode != kSplitNone ? kScheduleSortedChunks
                                                                  : plan_schedule;
}
constexpr int kSortKeys = 257;    // sort key = 256 - min(attended pages, 256)

GA_HD int32_t row_sort_key(int32_t npages) {
    return kSortKeys - 1 - (npages < kSortKeys - 1 ? npages : kSortKeys - 1);
}

// The sorted schedule keeps the row order and kSortKeys counters after the
// row prefix in shared memory: batches up to kMaxBatch - kSortKeys rows.
GA_HD bool sorted_schedule_fits(int32_t batch) { return batch + kSortKeys <= kMaxBatch; }

// Slot s of a grid of G CTAs over U units -> its position in the sorted
// order.  (Walking each CTA's passes from a different starting pass, so that
// long and short rows would mix at any moment, measured slower.)
GA_HD uint32_t snake_position(uint32_t s, uint32_t G, uint32_t U) {
    const uint32_t r = s / G, q = s - r * G;
    const uint32_t len = U - r * G < G ? U - r * G : G;      // CTAs in pass r
    return r * G + ((r & 1u) ? len - 1u - q : q);
}

// Geometry of one row for one call: which keys it attends, which logical
// pages hold them, and how those pages are cut into split-KV chunks.
struct RowGeom {
    int32_t len;         // L (0 if the given length was invalid)
    int32_t lo;          // first attended key: max(0, L - W) or 0
    int32_t first_page;  // logical page of key lo
    int32_t npages;      // logical pages holding keys [lo, L)
    int32_t cp;          // pages per chunk for this row
    int32_t chunks;      // chunks of this row (>= 1; an empty row has one empty chunk)
    bool bad_len;        // L < 0 or L > pt_stride * P
};

GA_HD int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }

GA_HD RowGeom row_geometry(int32_t L, int32_t window, int64_t pt_stride, int32_t mode,
                           int32_t splits, int32_t chunk_pages) {
    RowGeom g;
    g.bad_len = (L < 0) || ((int64_t)L > pt_stride * kPageSize);
    if (g.bad_len) L = 0;
    g.len = L;
    g.lo = (window > 0 && L > window) ? L - window : 0;
    g.first_page = g.lo / kPageSize;
    g.npages = L > 0 ? (L - 1) / kPageSize - g.first_page + 1 : 0;
    int32_t cp;
    if (mode == kSplitCount)
        cp = g.npages > 0 ? ceil_div(g.npages, splits > 0 ? splits : 1) : 1;
    else if (mode == kSplitChunk)
        cp = chunk_pages > 0 ? chunk_pages : 1;
    else
        cp = g.npages > 0 ? g.npages : 1;
    g.cp = cp;
    g.chunks = g.npages > 0 ? ceil_div(g.npages, cp) : 1;
    return g;
}

// Window of the keys any of a row's S queries attends (the last S positions,
// each with its own window): W + S - 1 for the sliding family, 0 (global)
// stays 0.  Saturates instead of overflowing.
GA_HD int32_t effective_window(int32_t window, int32_t S) {
    if (window <= 0) return 0;
    return window > 0x7fffffff - (S - 1) ? 0x7fffffff : window + (S - 1);
}

// Logical page range [*p0, *p0 + *np) of chunk j of a row.
GA_HD void chunk_pages_of(const RowGeom& g, int32_t j, int32_t* p0, int32_t* np) {
    int32_t a = j * g.cp;
    int32_t b = a + g.cp;
    if (b > g.npages) b = g.npages;
    if (a > b) a = b;
    *p0 = g.first_page + a;
    *np = b - a;
}

// A row of a chunked plan: its chunks of cp pages ("full"), then, unless its
// pages divide evenly, one shorter last chunk (an empty row: one empty last
// chunk and no full one).
GA_HD int32_t full_chunks(const RowGeom& g) {
    return (g.npages > 0 && g.npages % g.cp == 0) ? g.chunks : g.chunks - 1;
}

// The rows-by-size deal of a chunked plan (fixed chunk_pages) keeps three
// arrays after the row prefix in shared memory -- each row's full chunks
// before it (B + 1), the rows with a shorter last chunk in descending order
// of its pages (B), and kSortKeys counters: batches up to
// (kMaxBatch - kSortKeys - 1) / 3 rows.
GA_HD bool sorted_chunk_schedule_fits(int32_t batch) {
    return 3 * batch + kSortKeys + 1 <= kMaxBatch;
}

// Head groups of kHeadTile query heads per kv head.
GA_HD int32_t head_groups(int32_t group) { return ceil_div(group, kHeadTile); }

// Work unit u -> (row-chunk rc, kv head c, head group hg); units are ordered
// row-chunk major so that neighbouring CTAs share page-table lines.
GA_HD void unit_coords(int64_t u, int32_t Hkv, int32_t HG, int64_t* rc, int32_t* c,
                       int32_t* hg) {
    *hg = (int32_t)(u % HG);
    *c = (int32_t)((u / HG) % Hkv);
    *rc = u / ((int64_t)HG * Hkv);
}

// Checked page-id test: true iff page is a valid physical page.
GA_HD bool page_ok(int32_t page, int64_t num_pages) {
    return page >= 0 && (int64_t)page < num_pages;
}

// Index of the first element of page-head block (page, c) in a pool
// [num_pages, Hkv, P, D]; only call with page_ok(page).
GA_HD int64_t page_block_elem(int32_t page, int32_t c, int32_t Hkv, int32_t D) {
    return ((int64_t)page * Hkv + c) * (int64_t)kPageSize * D;
}

// Row of the 2-D [num_pages * Hkv * P, D] view a bulk tensor copy addresses.
GA_HD int32_t page_block_row(int32_t page, int32_t c, int32_t Hkv) {
    return (page * Hkv + c) * kPageSize;
}

}  // namespace ga
