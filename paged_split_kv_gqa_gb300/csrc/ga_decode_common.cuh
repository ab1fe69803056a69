// ga_decode_common.cuh -- what every decode kernel shares: the launch
// parameters, the work-unit geometry (row-chunk, kv head, head group) and the
// per-CTA prefix of row chunks that maps a unit index to its row.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "ga_device.cuh"
#include "ga_internal.h"

namespace ga {

struct DecodeParams {
    const __nv_bfloat16* q;       // [B, Hq, D]
    const int32_t* page_table;    // [B, pt_stride]
    const int32_t* seq_lens;      // [B]
    const float* k_scale;         // [Hkv] (E4M3)
    const float* v_scale;
    __nv_bfloat16* out;           // [B, Hq, D]
    float* partial_o;             // [rc_capacity, Hq, D]
    float* partial_lse;           // [rc_capacity, Hq]
    int32_t* touch_log;           // [rc_capacity, touch_stride] or null
    // this step's new token, [B, Hkv, D] bf16, appended by the decode itself
    // (one-query decode with the append fused), or null
    const uint4* k_new;
    const uint4* v_new;
    void* k_pool;                 // the pools, for that append
    void* v_pool;
    int32_t* err_word;
    int64_t pt_stride;
    int64_t num_pages;
    int64_t rc_capacity;
    // Hq and group count (query, head) columns: an S-query decode has
    // Hq * S columns, S adjacent per query head ([B, Hq, S, D]); window is
    // the union window of a row's S queries (page ranges), mask_window the
    // real one (per-column masks).
    int32_t B, Hq, Hkv, group, HG, window, mode, splits, chunk_pages, touch_stride;
    int32_t S, mask_window;
    int32_t TW;                   // columns per work unit (8, or 8 x warps column-parallel)
    int32_t schedule;             // kScheduleRoundRobin, kScheduleSorted (pre = row order) or
                                  // kScheduleSortedChunks (sorted arrays after the prefix)
    int32_t test_wait_timeout;    // test hook: CTA 0's producer issues nothing
    float scale_log2;             // softmax scale * log2(e)
    int64_t out_elems;            // B * Hq * D
    int64_t pool_rows;            // num_pages * Hkv * P
};

// GA_CHECKED builds test every shared- and global-memory access of the decode
// kernels against its buffer, record GA_DEVERR_SELF_CHECK and skip the access.
#ifdef GA_CHECKED
#define GA_CHK(cond) (cond)
#else
#define GA_CHK(cond) true
#endif

// Row owning row-chunk rc: largest b with pre[b] <= rc.
__device__ __forceinline__ int find_row(const int32_t* pre, int B, int64_t rc) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((int64_t)pre[mid] <= rc) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct UnitInfo {
    int64_t rc;
    int32_t b, c, hg, j, p0, np, h0, nvalid;
    RowGeom g;
};

// A unit's coordinates from shared memory only; its length load can be issued
// right after and consumed later (finish_unit), off the critical path.
struct UnitLoc {
    int64_t rc;
    int32_t b, c, hg;
};

// The rows-by-size deal of an unsplit plan: slot u -> position in the sorted
// order -> (row, kv head, head group); one chunk per row, so the row-chunk
// is the row, and pre[] holds the rows longest first.  Kept out of line: the
// decode kernels' hot loops are sensitive to the size of the code inlined
// into them (their instruction fetch).
static __device__ __noinline__ UnitLoc locate_sorted(const DecodeParams& p, const int32_t* pre,
                                                     int64_t u) {
    UnitLoc l;
    const uint32_t upr = (uint32_t)p.Hkv * (uint32_t)p.HG;
    const uint32_t pos = snake_position((uint32_t)u, gridDim.x, (uint32_t)p.B * upr);
    const uint32_t r = pos / upr, rem = pos - r * upr;
    const uint32_t hg = (p.HG == 1) ? 0u : rem % (uint32_t)p.HG;
    l.hg = (int32_t)hg;
    l.c = (int32_t)((rem - hg) / (uint32_t)p.HG);
    l.b = pre[r];
    l.rc = l.b;
    return l;
}

// The rows-by-size deal of a plan in fixed-size chunks: the full chunks
// first (row order), then the rows' shorter last chunks longest first.  pre[]
// keeps the row prefix; after it, fpre[0 .. B] (full chunks before each row)
// and the rows with a shorter last chunk in that order (build_chunk_order).
static __device__ __noinline__ UnitLoc locate_sorted_chunks(const DecodeParams& p,
                                                            const int32_t* pre, int64_t u) {
    UnitLoc l;
    const uint32_t upr = (uint32_t)p.Hkv * (uint32_t)p.HG;
    const uint32_t pos = snake_position((uint32_t)u, gridDim.x, (uint32_t)pre[p.B] * upr);
    const uint32_t r = pos / upr, rem = pos - r * upr;
    const uint32_t hg = (p.HG == 1) ? 0u : rem % (uint32_t)p.HG;
    l.hg = (int32_t)hg;
    l.c = (int32_t)((rem - hg) / (uint32_t)p.HG);
    const int32_t* fpre = pre + p.B + 1;           // full chunks before each row
    const int32_t* rrow = fpre + p.B + 1;          // rows with a shorter last chunk
    const int32_t F = fpre[p.B];
    if ((int32_t)r < F) {
        l.b = find_row(fpre, p.B, r);
        l.rc = pre[l.b] + ((int32_t)r - fpre[l.b]);
    } else {
        l.b = rrow[(int32_t)r - F];
        l.rc = pre[l.b + 1] - 1;
    }
    return l;
}

__device__ __forceinline__ UnitLoc locate_unit(const DecodeParams& p, const int32_t* pre,
                                               int64_t u) {
    if (p.schedule != kScheduleRoundRobin)
        return p.schedule == kScheduleSorted ? locate_sorted(p, pre, u)
                                             : locate_sorted_chunks(p, pre, u);
    UnitLoc l;
    if (u < (int64_t(1) << 31)) {      // unit_coords in 32 bits (64-bit division is slow)
        const uint32_t v = (uint32_t)u, hg = (uint32_t)p.HG, hkv = (uint32_t)p.Hkv;
        const uint32_t q1 = (hg == 1) ? v : v / hg;
        const uint32_t r = q1 / hkv;
        l.hg = (int32_t)(v - q1 * hg);
        l.c = (int32_t)(q1 - r * hkv);
        l.rc = r;
    } else {
        unit_coords(u, p.Hkv, p.HG, &l.rc, &l.c, &l.hg);
    }
    l.b = find_row(pre, p.B, l.rc);
    return l;
}

// First q row (in the [B * Hq, D] view) of a unit's head group.
__device__ __forceinline__ int32_t unit_q_row(const DecodeParams& p, const UnitLoc& l) {
    return l.b * p.Hq + l.c * p.group + l.hg * p.TW;
}

__device__ __forceinline__ UnitInfo finish_unit(const DecodeParams& p, const int32_t* pre,
                                                const UnitLoc& l, int32_t len) {
    UnitInfo x;
    x.rc = l.rc;
    x.b = l.b;
    x.c = l.c;
    x.hg = l.hg;
    x.j = p.schedule == kScheduleSorted ? 0 : (int32_t)(x.rc - pre[x.b]);
    x.g = row_geometry(len, p.window, p.pt_stride, p.mode, p.splits, p.chunk_pages);
    chunk_pages_of(x.g, x.j, &x.p0, &x.np);
    x.h0 = x.c * p.group + x.hg * p.TW;
    int nv = p.group - x.hg * p.TW;
    x.nvalid = nv < p.TW ? nv : p.TW;
    return x;
}

__device__ __forceinline__ UnitInfo unit_info(const DecodeParams& p, const int32_t* pre,
                                                     int64_t u) {
    const UnitLoc l = locate_unit(p, pre, u);
    return finish_unit(p, pre, l, __ldg(p.seq_lens + l.b));
}

__device__ __forceinline__ int32_t row_key(const DecodeParams& p, int32_t b) {
    return row_sort_key(row_geometry(__ldg(p.seq_lens + b), p.window, p.pt_stride, p.mode,
                                     p.splits, p.chunk_pages).npages);
}

// The rows-by-size schedule (one chunk per row, so pre[b] = b until now):
// pre[0 .. B) becomes the rows in descending order of attended pages, ties
// in row order -- the same order in every CTA (counts, then a stable scatter
// by one warp); the kSortKeys ints after pre[B] are its counters.
static __device__ __noinline__ void build_row_order(const DecodeParams& p, int32_t* pre,
                                                    int nthreads) {
    int32_t* cnt = pre + p.B + 1;
    for (int i = threadIdx.x; i < kSortKeys; i += nthreads) cnt[i] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += nthreads) atomicAdd(&cnt[row_key(p, b)], 1);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        constexpr int PER = (kSortKeys + 31) / 32;        // buckets per lane
        int v[PER], run = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int k = lane * PER + i;
            v[i] = k < kSortKeys ? cnt[k] : 0;
            run += v[i];
        }
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
        }
        int start = incl - run;                           // first slot of bucket lane * PER
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int k = lane * PER + i;
            if (k < kSortKeys) cnt[k] = start;
            start += v[i];
        }
        __syncwarp();
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            const bool live = b < p.B;
            const int key = live ? row_key(p, b) : kSortKeys + lane;   // dead lanes match none
            const uint32_t peers = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int pos = live ? cnt[key] + rank : 0;
            __syncwarp();
            if (live && rank == __popc(peers) - 1) cnt[key] += __popc(peers);
            __syncwarp();
            if (live) pre[pos] = b;
        }
    }
    __syncthreads();
}

// The same for a plan in fixed-size chunks (pre[] stays the row prefix):
// fpre[0 .. B] after it (full chunks before each row, a prefix by warp 0),
// then the rows that end in a shorter chunk in descending order of its
// pages (ties in row order), then the kSortKeys counters.
static __device__ __noinline__ void build_chunk_order(const DecodeParams& p, int32_t* pre,
                                                      int nthreads) {
    int32_t* fpre = pre + p.B + 1;
    int32_t* rrow = fpre + p.B + 1;
    int32_t* cnt = rrow + p.B;
    // a row's sort key (descending pages of its last chunk), or -1 if its
    // chunks are all full
    auto key_of = [&](int32_t b) -> int32_t {
        const RowGeom g = row_geometry(__ldg(p.seq_lens + b), p.window, p.pt_stride, p.mode,
                                       p.splits, p.chunk_pages);
        const int32_t full = full_chunks(g);
        return full < g.chunks ? row_sort_key(g.npages - full * g.cp) : -1;
    };
    for (int b = threadIdx.x; b < p.B; b += nthreads)
        fpre[b + 1] = full_chunks(row_geometry(__ldg(p.seq_lens + b), p.window, p.pt_stride,
                                               p.mode, p.splits, p.chunk_pages));
    for (int i = threadIdx.x; i < kSortKeys; i += nthreads) cnt[i] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += nthreads) {
        const int32_t key = key_of(b);
        if (key >= 0) atomicAdd(&cnt[key], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // fpre: inclusive prefix of the full-chunk counts
        {
            const int seg = (p.B + 31) / 32;
            const int lo = min(p.B, lane * seg), hi = min(p.B, lo + seg);
            int run = 0;
            for (int b = lo; b < hi; ++b) {
                run += fpre[b + 1];
                fpre[b + 1] = run;
            }
            int incl = run;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const int excl = incl - run;
            for (int b = lo; b < hi; ++b) fpre[b + 1] += excl;
            if (lane == 0) fpre[0] = 0;
        }
        // counting sort of the rows with a shorter last chunk into rrow
        constexpr int PER = (kSortKeys + 31) / 32;        // buckets per lane
        int v[PER], run = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int k = lane * PER + i;
            v[i] = k < kSortKeys ? cnt[k] : 0;
            run += v[i];
        }
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
        }
        int start = incl - run;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int k = lane * PER + i;
            if (k < kSortKeys) cnt[k] = start;
            start += v[i];
        }
        __syncwarp();
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            const int k0 = b < p.B ? key_of(b) : -1;
            const bool live = k0 >= 0;
            const int key = live ? k0 : kSortKeys + lane;   // dead lanes match none
            const uint32_t peers = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int pos = live ? cnt[key] + rank : 0;
            __syncwarp();
            if (live && rank == __popc(peers) - 1) cnt[key] += __popc(peers);
            __syncwarp();
            if (live) rrow[pos] = b;
        }
    }
    __syncthreads();
}

// Every thread of the block: chunk count of every row, then an inclusive
// prefix pre[b+1] = sum_{b' <= b} in shared memory.  Reports invalid lengths
// (block 0) and returns false (the whole block must then exit) when a split
// plan's row-chunk capacity is too small.
__device__ __forceinline__ bool build_row_prefix(const DecodeParams& p, int32_t* pre,
                                                 int nthreads, int64_t* total_rc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int bad = 0;
    for (int b = threadIdx.x; b < p.B; b += nthreads) {
        const RowGeom g = row_geometry(__ldg(p.seq_lens + b), p.window, p.pt_stride, p.mode,
                                       p.splits, p.chunk_pages);
        pre[b + 1] = g.chunks;
        bad |= g.bad_len ? 1 : 0;
    }
    bad = __syncthreads_or(bad);
    if (warp == 0) {
        const int seg = (p.B + 31) / 32;
        const int lo = min(p.B, lane * seg), hi = min(p.B, lo + seg);
        int run = 0;
        for (int b = lo; b < hi; ++b) {
            run += pre[b + 1];
            pre[b + 1] = run;
        }
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        const int excl = incl - run;
        for (int b = lo; b < hi; ++b) pre[b + 1] += excl;
        if (lane == 0) pre[0] = 0;
    }
    __syncthreads();
    if (bad && blockIdx.x == 0 && threadIdx.x == 0) report(p.err_word, kErrSeqLen);
    *total_rc = pre[p.B];
    if (p.schedule == kScheduleSorted) build_row_order(p, pre, nthreads);
    else if (p.schedule == kScheduleSortedChunks) build_chunk_order(p, pre, nthreads);
    if (p.mode != kSplitNone && *total_rc > p.rc_capacity) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(p.err_word, kErrCapacity);
        return false;
    }
    return true;
}

// ---- the KV page append fused into a one-query decode
//
// When the call carries this step's token (p.k_new), the unit that holds a
// row's last page (its last chunk; the token's position is L - 1) writes the
// token of its kv heads [x.c NH, x.c NH + NH) into that page's slot exactly
// as ga_kv_append does (bf16 bits, or the E4M3 quantisation), and orders those
// generic stores before the bulk tensor copy of that page.  Only this unit
// reads those page-head blocks of the row, so no other CTA waits for it.
template <int D, int KV, int NH>
struct TokenAppend {
    static constexpr int PER_HEAD = D / 8;                     // uint4 of bf16 per head
    static constexpr int PER_LANE = (NH * PER_HEAD + 31) / 32;
    static constexpr int LINES = NH * D * 2 / 128;             // 128-byte lines of k (or v)

    __device__ __forceinline__ static bool due(const DecodeParams& p, const UnitInfo& x) {
        return p.k_new != nullptr && x.hg == 0 && x.g.len > 0 && x.j == x.g.chunks - 1;
    }

    // The lanes of one warp write the token of row b, kv heads [c0, c0 + NH),
    // at position pos into `page` (reported, and nothing written, if the id
    // is not a page of the pool).  No fence.
    __device__ __forceinline__ static void write(const DecodeParams& p, int32_t b, int32_t c0,
                                                 int32_t pos, int32_t page) {
        const int lane = threadIdx.x & 31;
        if (!page_ok(page, p.num_pages)) {
            if (lane == 0) report(p.err_word, kErrPosition);
            return;
        }
        const int hkv = p.Hkv * NH;                            // kv heads of the pool
        const int64_t src0 = ((int64_t)b * hkv + c0) * PER_HEAD;
        const int64_t slot = (int64_t)(pos % kPageSize) * D;
        uint4 k[PER_LANE], v[PER_LANE];
        float ks[PER_LANE], vs[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            if (e < NH * PER_HEAD) {
                k[i] = __ldg(p.k_new + src0 + e);
                v[i] = __ldg(p.v_new + src0 + e);
                if constexpr (KV != GA_KV_BF16) {
                    ks[i] = __ldg(p.k_scale + c0 + e / PER_HEAD);
                    vs[i] = __ldg(p.v_scale + c0 + e / PER_HEAD);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            if (e < NH * PER_HEAD) {
                const int64_t elem = page_block_elem(page, c0 + e / PER_HEAD, hkv, D) + slot +
                                     (int64_t)(e % PER_HEAD) * 8;
                if constexpr (KV == GA_KV_BF16) {
                    reinterpret_cast<uint4*>(p.k_pool)[elem / 8] = k[i];
                    reinterpret_cast<uint4*>(p.v_pool)[elem / 8] = v[i];
                } else {
                    reinterpret_cast<uint2*>(p.k_pool)[elem / 8] = quantize8(k[i], ks[i]);
                    reinterpret_cast<uint2*>(p.v_pool)[elem / 8] = quantize8(v[i], vs[i]);
                }
            }
        }
    }

    __device__ __forceinline__ static const int32_t* page_entry(const DecodeParams& p,
                                                                int32_t b, int32_t pos) {
        return p.page_table + (int64_t)b * p.pt_stride + pos / kPageSize;
    }

    // The token's lines into L2 (lanes first, first + step, ...).
    __device__ __forceinline__ static void prefetch(const DecodeParams& p, int32_t b, int32_t c0,
                                                    int first, int step) {
        const int64_t src0 = ((int64_t)b * (p.Hkv * NH) + c0) * PER_HEAD;
        for (int l = first; l < LINES; l += step) {
            prefetch_l2(reinterpret_cast<const char*>(p.k_new + src0) + 128 * l);
            prefetch_l2(reinterpret_cast<const char*>(p.v_new + src0) + 128 * l);
        }
    }

    // Used by a producer warp that writes its own unit's token: start() at
    // the start of unit x, finish() right before it issues the copy of the
    // unit's last page, with that page's id (the lines have been on their
    // way to L2 since start()).
    int32_t b, c0, pos;
    bool pending;

    __device__ __forceinline__ void start(const DecodeParams& p, const UnitInfo& x) {
        pending = due(p, x);
        if (!pending) return;
        b = x.b;
        c0 = x.c * NH;
        pos = x.g.len - 1;
        prefetch(p, b, c0, threadIdx.x & 31, 32);
    }

    __device__ __forceinline__ void finish(const DecodeParams& p, int32_t page) {
        if (!pending) return;
        pending = false;
        write(p, b, c0, pos, page);
        fence_proxy_async_global();
        __syncwarp();
    }
};

// ---- pieces of the warp-specialised tcgen05 kernels

__device__ __forceinline__ uint32_t bar(uint32_t bars, int i) { return bars + 8u * (uint32_t)i; }

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t b, uint32_t parity,
                                              volatile int* abort_flag) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*abort_flag || clock64() - t0 > kWaitBudgetCycles) return false;
    }
    return true;
}

// Walks a CTA's units (blockIdx.x, + gridDim.x, ...) with the next unit's
// length load in flight while the current one is processed.
struct UnitCursor {
    int64_t u, U;
    UnitLoc nl;
    int32_t nlen;
    __device__ __forceinline__ UnitCursor(const DecodeParams& p, const int32_t* pre, int64_t U_)
        : u(blockIdx.x), U(U_), nl(), nlen(0) {
        if (u < U) fetch(p, pre);
    }
    __device__ __forceinline__ void fetch(const DecodeParams& p, const int32_t* pre) {
        nl = locate_unit(p, pre, u);
        nlen = __ldg(p.seq_lens + nl.b);
    }
    // The current unit's geometry; starts the next unit's length load.
    __device__ __forceinline__ UnitInfo take(const DecodeParams& p, const int32_t* pre) {
        const UnitInfo x = finish_unit(p, pre, nl, nlen);
        u += gridDim.x;
        if (u < U) fetch(p, pre);
        return x;
    }
    __device__ __forceinline__ bool more() const { return u < U; }
};

// Bounded wait of one issuing thread; on a timeout or an abort elsewhere it
// reports, raises the abort flag and returns false.
__device__ __forceinline__ bool issuer_wait(const DecodeParams& p, uint32_t b, uint32_t parity,
                                            volatile int* abort_flag) {
    if (!*abort_flag && wait_or_abort(b, parity, abort_flag)) return true;
    report(p.err_word, kErrTimeout);
    *abort_flag = 1;
    return false;
}

}  // namespace ga
