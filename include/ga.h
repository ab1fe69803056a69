/*
 * ga.h -- C ABI of the paged split-KV GQA decode-attention library (libga.so)
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation is one decode step of Gemma-4-shaped attention over two KV
 * families that keep their own head counts and cache shapes ("[Model] Gemma 4
 * M1 12B", Description): a local sliding-window family at head_dim 256 with a
 * 1024-token window and a global full-context family at head_dim 512 with
 * fewer KV heads ("[Model] Gemma 4 M3 31B", Description; "visible-cx/Gemma-4-
 * 31B-CoreAI", hybrid-pf64 numerics gate: 32 query heads over 4 global KV
 * heads).  Each family has its own paged KV pools and page table.
 *
 * For every row b and query head h (kv head c = h / (Hq / Hkv), block GQA):
 *     keys   j in [lo_b, L_b),  lo_b = max(0, L_b - window) (local) or 0 (global)
 *     s_j    = scale * <q[b,h,:], K[page_table[b][j/P], c, j%P, :]>
 *     out    = sum_j softmax(s)_j * V[page_table[b][j/P], c, j%P, :]
 * where L_b = seq_lens[b] counts the token appended this step.
 *
 * Conventions shared by every entry point:
 *   - Memory: the caller owns all buffers.  Pointer arguments named
 *     *_host are host memory; every other pointer is device memory of the
 *     current CUDA device.  The library never allocates, frees or
 *     synchronises.  Work is enqueued on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and returns before it runs.
 *   - Layouts are dense, row-major (C order):
 *       q, out      [B, Hq, D]            bf16  ([B, Hq, S, D] for S-query decode)
 *       k_new,v_new [B, Hkv, D]           bf16
 *       pools       [num_pages, Hkv, P, D] bf16 (GA_KV_BF16) or OCP E4M3FN
 *                   codes (GA_KV_E4M3), one page-head block of P*D elements
 *                   contiguous
 *       k_scale, v_scale [Hkv] fp32 (E4M3 pools only; value = code * scale)
 *       page_table  [B, pt_stride] int32 physical page ids
 *       seq_lens, positions [B] int32
 *     q, out, pools, k_new, v_new and workspace must be 16-byte aligned.
 *   - page_size must be 16.  Offsets are 64-bit; num_pages * Hkv * 16 must
 *     stay below 2^31.
 *   - Return value: GA_OK, or a GA_ERR_* code when the arguments are rejected
 *     before anything is launched (fail closed, nothing enqueued), or
 *     GA_ERR_CUDA when a launch fails.  ga_strerror() names a code.
 *   - Device-side checks: values only the device sees (page ids, seq_lens,
 *     positions) are checked by the kernels.  A violation is OR-ed into
 *     *err_word as GA_DEVERR_* bits and the offending access is skipped (an
 *     invalid page contributes no keys, an invalid length is treated as 0).
 *     err_word may be NULL (no reporting; accesses are still skipped).  Read
 *     it after the stream has completed; clear it to 0 yourself.
 */
#ifndef GA_H_
#define GA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* ga_stream_t;   /* same type as cudaStream_t */

/* ----------------------------------------------------------- status codes */
enum {
    GA_OK = 0,
    GA_ERR_INVALID_ARG = 1,         /* null / misaligned pointer, bad size or shape */
    GA_ERR_UNSUPPORTED = 2,         /* valid but not served: head_dim, page_size, dtype */
    GA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < plan->workspace_bytes */
    GA_ERR_CUDA = 4,                /* a CUDA runtime / driver call or launch failed */
    GA_ERR_DEVICE_CHECK = 5         /* returned by ga_check_error_word for a nonzero word */
};

/* KV element types. */
enum { GA_KV_BF16 = 0, GA_KV_E4M3 = 1 };

/* Bits a kernel ORs into *err_word. */
enum {
    GA_DEVERR_PAGE_ID = 1,       /* a page id outside [0, num_pages) was met */
    GA_DEVERR_SEQ_LEN = 2,       /* seq_len < 0 or > pt_stride * page_size */
    GA_DEVERR_CAPACITY = 4,      /* seq_lens need more split chunks than the plan holds */
    GA_DEVERR_Q_RANGE = 8,       /* E4M3 path: q holds an infinite value */
    GA_DEVERR_TIMEOUT = 16,      /* a bounded wait for a bulk copy ran out */
    GA_DEVERR_POSITION = 32,     /* append: position / page_table[pos / P] invalid */
    GA_DEVERR_SELF_CHECK = 64    /* GA_CHECKED builds: an access outside its buffer was skipped */
};

/* --------------------------------------------------------------- the plan */

/* Split modes. */
enum {
    GA_SPLIT_NONE = 0,    /* one chunk per (row, kv head); output written directly */
    GA_SPLIT_COUNT = 1,   /* each row's pages cut into `splits` near-equal chunks */
    GA_SPLIT_CHUNK = 2    /* chunks of `chunk_pages` pages; a row's chunking depends
                             only on its own length (batch-invariant) */
};

/* Plan flags. */
enum {
    GA_PLAN_TOUCH_LOG = 1,        /* decode records every physical page it reads (tests) */
    GA_PLAN_EXTERNAL_COMBINE = 2, /* a split decode call leaves the partials in the
                                     workspace; the caller runs ga_splitkv_combine */
    GA_PLAN_TEST_WAIT_TIMEOUT = 4, /* test hook: CTA 0 of the decode launch issues no page,
                                     so its consumers' bounded waits run out (~2 s) and the
                                     call reports GA_DEVERR_TIMEOUT; CTA 0's rows are then
                                     undefined.  Never set outside tests. */
    GA_PLAN_TENSOR_CORE_UNITS = 8, /* more than 8 (query, head) columns per kv head: always
                                      units of 64 columns (tensor-core kernel on bf16 pools) */
    GA_PLAN_COLUMN_PARALLEL_UNITS = 16, /* ... always column-parallel units of 32 columns.
                                      Neither flag: 64-column units from 32 columns per kv
                                      head at head_dim 512 and from 64 at head_dim 256
                                      (where each is the faster on GB300), else 32. */
    GA_PLAN_KV_E4M3 = 32          /* the plan is for E4M3 pools: the cost model weighs an
                                      E4M3 page at half a bf16 one, and on the sliding family
                                      (head_dim 256, one query per row, 2 or 4 query heads per
                                      kv head, Hkv a multiple of 8 / group) the planner may
                                      give a work unit 8 / group kv heads (kv_heads_per_unit),
                                      whose pages the decode then copies as one box per
                                      128-dim region for all of them: it does so when the
                                      one-head plan needs no split and the wider units alone
                                      fill at least four rounds of the SMs (fewer, larger units
                                      measured slower below that).  With more than 8 (query,
                                      head) columns per kv head it gives units of 16 columns
                                      (col_tile 16), each streaming a kv head's pages once
                                      for all 16; such a plan is for E4M3 pools only.  Results
                                      stay within the E4M3 tolerance either way; a plan made
                                      without it also serves E4M3 pools (8-column units), and
                                      bf16 pools ignore the flag otherwise. */
};

/*
 * Split-KV plan, filled by ga_plan_splits on the host and passed by pointer
 * to the decode and combine calls (read on the host at call time only).
 */
typedef struct ga_plan {
    int32_t mode;            /* GA_SPLIT_* */
    int32_t splits;          /* GA_SPLIT_COUNT: chunks per row */
    int32_t chunk_pages;     /* GA_SPLIT_CHUNK: pages per chunk */
    int32_t batch;           /* B the plan was made for */
    int32_t num_q_heads;     /* Hq */
    int32_t num_kv_heads;    /* Hkv */
    int32_t head_dim;        /* D */
    int32_t window;          /* W (0 = global family) */
    int32_t page_size;       /* P */
    int32_t grid;            /* CTAs the decode launch uses */
    int32_t flags;           /* GA_PLAN_* */
    int32_t touch_stride;    /* touch-log entries per row-chunk (flag set) */
    int32_t q_len;           /* query tokens per row S (1 = one-query decode) */
    int32_t col_tile;        /* (query, head) columns per work unit: 8; when a kv head has
                                more than 8, 32 (column-parallel mma.sync units) or 64
                                (tcgen05 units; bf16 pools with K and V apart, other
                                pools run 8-column units), or, in a plan made with
                                GA_PLAN_KV_E4M3, 16: units of 16 columns of the E4M3
                                decode (accepted with E4M3 pools only) */
    int64_t row_chunks;      /* (row, chunk) pairs the workspace holds */
    int64_t units;           /* work units (row-chunk x kv head x head group) planned */
    int64_t workspace_bytes; /* device workspace the decode call needs (0 if none) */
    int64_t partial_o_offset;    /* byte offsets inside the workspace */
    int64_t partial_lse_offset;
    int64_t touch_log_offset;
    int32_t kv_heads_per_unit;   /* kv heads per work unit of the E4M3 sliding-family decode:
                                    1, or 8 / group when the plan has GA_PLAN_KV_E4M3 and the
                                    planner found such units better (see that flag).  A caller
                                    may set it to 1 or to that value; other kernels ignore it. */
    int32_t schedule;            /* how the persistent CTAs deal out the units:
                                    GA_SCHEDULE_ROUND_ROBIN (unit i to CTA i mod grid), or
                                    GA_SCHEDULE_ROWS_BY_SIZE, for one-query plans: unsplit
                                    ones of at most 1791 rows (rows in descending order of
                                    attended pages) or ones in fixed-size chunks of at most
                                    596 rows (the full chunks in row order, then the rows'
                                    shorter last chunks longest first); every other pass
                                    over the CTAs reversed.  The planner picks the second
                                    when it evens out the CTA loads.  Results do not depend on it.  The decode
                                    calls refuse any other value, and the second on other
                                    plans, with GA_ERR_INVALID_ARG before any launch. */
} ga_plan;

enum {
    GA_SCHEDULE_ROUND_ROBIN = 0,
    GA_SCHEDULE_ROWS_BY_SIZE = 1
};

/*
 * ga_plan_splits -- choose how each row's attended pages are cut into split-KV
 * chunks so that the decode launch fills all SMs ("[Model] Gemma 4 M3 31B",
 * Proposed Plan: the split-KV chunk policy re-checked when the global
 * family's head count changes; "visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa
 * is mandatory here": flash-decode split factor 8).  Host only, no CUDA call.
 *
 *   seq_lens_host [batch] int32, host memory: the lengths (or upper bounds of
 *       the lengths) the decode calls will see; the workspace is sized for them.
 *   window: 0 for the global family, else the sliding window W.
 *   num_sms: SMs of the device the decode runs on (>= 1).
 *   requested_splits > 0: GA_SPLIT_COUNT with that many chunks per row
 *       (1 = GA_SPLIT_NONE).  fixed_chunk_tokens > 0 (a multiple of
 *       page_size): GA_SPLIT_CHUNK with that chunk size.  Both 0: automatic
 *       (a cost model over candidate chunk sizes of the static round-robin
 *       schedule; the result may depend on the whole batch).  Both > 0 is an
 *       error.
 *   flags: GA_PLAN_* bits.
 * Returns GA_OK and fills *plan_out, or GA_ERR_INVALID_ARG / GA_ERR_UNSUPPORTED.
 */
int ga_plan_splits(const int32_t* seq_lens_host, int32_t batch, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, int32_t window, int32_t page_size,
                   int32_t num_sms, int32_t requested_splits, int32_t fixed_chunk_tokens,
                   int32_t flags, ga_plan* plan_out);

/*
 * ga_plan_splits_mq -- ga_plan_splits for multi-query decode: q_len (S, 1 ..
 * GA_MAX_Q_LEN) query tokens per row, the row's last S positions
 * ("visible-cx/Gemma-4-31B-CoreAI", hybrid-pf64/ bundles: a query axis with
 * an intra-chunk causal mask, and chunked walks that must agree with
 * token-by-token ones; "Gemma 4 31B on vLLM -- operating-point reference",
 * LIGHT recipe: EAGLE3 verify of 3 speculative tokens, i.e. 4 queries per
 * row).  The plan covers the pages any of a row's S queries attends (the
 * window grows by S - 1 for the sliding family) and work units over the
 * S x (Hq / Hkv) (query, head) columns of each kv head.  q_len = 1 is
 * ga_plan_splits.  Other arguments and errors as for ga_plan_splits.
 */
#define GA_MAX_Q_LEN 64
int ga_plan_splits_mq(const int32_t* seq_lens_host, int32_t batch, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t window, int32_t page_size,
                      int32_t q_len, int32_t num_sms, int32_t requested_splits,
                      int32_t fixed_chunk_tokens, int32_t flags, ga_plan* plan_out);

/*
 * ga_kv_append -- write this step's new K and V token of every row into its
 * page slot: page page_table[b][positions[b] / P], slot positions[b] % P, for
 * every kv head ("[Model] Gemma 4 M1 12B", Description: paged prefill and
 * decode; "[Model] Gemma 4 M2 26B-A4B", Proposed Plan: opt-in FP8 KV pool for
 * the sliding family, and page offsets through one checked helper).
 *
 *   k_new, v_new [batch, num_kv_heads, head_dim] bf16.
 *   k_pool, v_pool written in place; kv_dtype GA_KV_BF16 copies the bits,
 *       GA_KV_E4M3 stores E4M3FN(round-to-nearest-even, saturate to +-448)
 *       of fp32(x) / scale[c] (IEEE division); k_scale, v_scale required for
 *       E4M3 and ignored for bf16.
 *   positions [batch] int32: slot index of the new token (= L_b - 1); rows
 *       with a negative position are skipped.
 *   head_dim 256 or 512.
 * Device errors: GA_DEVERR_POSITION (row skipped).
 */
int ga_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                 int32_t kv_dtype, const float* k_scale, const float* v_scale,
                 const int32_t* page_table, int64_t pt_stride, const int32_t* positions,
                 int32_t batch, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                 int64_t num_pages, int32_t* err_word, ga_stream_t stream);

/*
 * ga_decode_local_hd256 -- sliding-window paged decode, head_dim 256
 * ("[Model] Gemma 4 M3 31B", Acceptance Criteria: window boundaries at 1023,
 * 1024, 1025 with multiple-window continuation).  Only the pages holding keys
 * [L_b - window, L_b) are read ("Gemma 4 31B on vLLM -- operating-point
 * reference", Three load-bearing facts: sliding-window tile pruning).
 *
 *   q [batch, num_q_heads, 256] bf16; num_q_heads % num_kv_heads == 0.
 *   kv_dtype GA_KV_BF16 or GA_KV_E4M3 (with k_scale, v_scale [Hkv] fp32;
 *       with E4M3 the products run on E4M3 tensor cores: q is scaled per head
 *       and split into two E4M3 parts, P likewise, about bf16 precision; an
 *       E4M3 pool passed as both k_pool and v_pool is read once).
 *   seq_lens [batch] int32 device; window >= 1.
 *   scale: softmax scale (e.g. 1/sqrt(256), or 1.0 for the Gemma convention).
 *   plan: from ga_plan_splits with the same batch, heads, head_dim, window
 *       and page_size.  If plan->mode != GA_SPLIT_NONE the call needs
 *       workspace (>= plan->workspace_bytes, 16-byte aligned) and runs the
 *       decode kernel then ga_splitkv_combine's kernel on `stream` (the
 *       latter is left to the caller when the plan has
 *       GA_PLAN_EXTERNAL_COMBINE).
 *   out [batch, num_q_heads, 256] bf16.
 * Rows with L_b = 0 produce zeros.
 * Multi-query decode (plan from ga_plan_splits_mq with q_len = S > 1): q and
 *   out are [batch, num_q_heads, S, 256] (a head's S query tokens adjacent);
 *   query i of row b sits at position p = L_b - S + i and attends keys
 *   [max(0, p - window + 1), p] (causal inside the chunk, the window ending
 *   at its own position); a query with p < 0 produces zeros.
 */
int ga_decode_local_hd256(const void* q, const void* k_pool, const void* v_pool,
                          int32_t kv_dtype, const float* k_scale, const float* v_scale,
                          const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t window, int32_t page_size, int64_t num_pages, float scale,
                          const ga_plan* plan, void* workspace, size_t workspace_bytes,
                          void* out, int32_t* err_word, ga_stream_t stream);

/*
 * ga_decode_global_hd512 -- full-context paged decode, head_dim 512
 * ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is mandatory here" and
 * hybrid-pf64 numerics gate: S=1 decode over the whole cache, no causal mask,
 * 32 query heads x 512 over 4 KV heads).  Arguments as for the local call
 * without `window`; head_dim is 512.  Passing the same pool as k_pool and
 * v_pool (K == V, as with a shared K/V projection: "[Model] Gemma 4 M1 12B",
 * Description) reads each page-head block once and uses it for both products.
 * Multi-query decode as for the local call: q, out [batch, num_q_heads, S,
 * 512], query i at position L_b - S + i attends keys [0, L_b - S + i].
 */
int ga_decode_global_hd512(const void* q, const void* k_pool, const void* v_pool,
                           int32_t kv_dtype, const float* k_scale, const float* v_scale,
                           const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                           int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t page_size, int64_t num_pages, float scale,
                           const ga_plan* plan, void* workspace, size_t workspace_bytes,
                           void* out, int32_t* err_word, ga_stream_t stream);

/*
 * ga_decode_local_hd256_append, ga_decode_global_hd512_append -- one decode
 * step with the KV page append fused in: the same result as
 *     ga_kv_append(k_new, v_new, k_pool, v_pool, ..., positions = seq_lens - 1)
 * followed by ga_decode_local_hd256 / ga_decode_global_hd512 on the same
 * stream (pools bit-identical, outputs bit-identical), in one launch ("[Model]
 * Gemma 4 M1 12B", Description: paged prefill and decode; a decode step's
 * token is appended at position L - 1 and then attended).  The unit of the
 * decode that reads a row's last page writes the row's token into it first.
 *   k_new, v_new [batch, num_kv_heads, D] bf16, 16-byte aligned: this step's
 *       token of every row, written at seq_lens[b] - 1 (rows of length 0
 *       write nothing; E4M3 pools get the quantisation ga_kv_append uses).
 *   plan->q_len must be 1.  Other arguments as for the decode call, with the
 *       pools writable.
 * When a kv head's query heads span several units (more than 8 query heads
 * per kv head), or the plan is one for 64-column multi-query units, the call
 * launches the append kernel before the decode: the
 * same result in two launches.  Device errors: those of both calls
 * (GA_DEVERR_POSITION for an invalid page id at the token's slot).
 */
int ga_decode_local_hd256_append(const void* k_new, const void* v_new, const void* q,
                                 void* k_pool, void* v_pool, int32_t kv_dtype,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* page_table, int64_t pt_stride,
                                 const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t window, int32_t page_size,
                                 int64_t num_pages, float scale, const ga_plan* plan,
                                 void* workspace, size_t workspace_bytes, void* out,
                                 int32_t* err_word, ga_stream_t stream);
int ga_decode_global_hd512_append(const void* k_new, const void* v_new, const void* q,
                                  void* k_pool, void* v_pool, int32_t kv_dtype,
                                  const float* k_scale, const float* v_scale,
                                  const int32_t* page_table, int64_t pt_stride,
                                  const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t page_size, int64_t num_pages,
                                  float scale, const ga_plan* plan, void* workspace,
                                  size_t workspace_bytes, void* out, int32_t* err_word,
                                  ga_stream_t stream);

/*
 * ga_splitkv_combine -- merge split-KV partials by log-sum-exp
 * ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is mandatory here":
 * flash-decode with split factor 8):
 *     M = max_s lse_s,  out = sum_s e^{lse_s - M} o_s / sum_s e^{lse_s - M}
 * with o_s normalised within its chunk and lse_s = ln sum_{j in chunk s} e^{s_j}
 * (natural log; an empty chunk has lse_s = -inf and weighs nothing).
 *
 *   partial_o [plan->row_chunks, Hq * S, D] fp32 and partial_lse
 *       [plan->row_chunks, Hq * S] fp32 (S = plan->q_len; query i of head h
 *       is column h * S + i), device: row-chunk r of row b is
 *       rc_b + j, rc_b = sum over rows b' < b of that row's chunk count, in
 *       the chunking the plan defines for the device seq_lens.
 *   seq_lens [plan->batch] int32 device and pt_stride: the same values the
 *   decode call got (a length beyond pt_stride * page_size counts as 0).
 *   Rows whose chunk count is 1 are left untouched (the decode call wrote
 *   them).  out [plan->batch, Hq, S, D] bf16.
 * The decode calls invoke this themselves when split; it is exported for
 * testing and for callers that write their own partials.
 */
int ga_splitkv_combine(const float* partial_o, const float* partial_lse, const ga_plan* plan,
                       const int32_t* seq_lens, int64_t pt_stride, void* out,
                       int32_t* err_word, ga_stream_t stream);

/*
 * ga_decode_global_hd512_noalloc -- the same decode as ga_decode_global_hd512,
 * for callers that cannot allocate device memory when they decode (the pages
 * have no counterpart; this is a library convenience).  Examples: a plain-C
 * serving loop without a caching allocator, where cudaMalloc would
 * synchronise the whole device in the middle of a decode step, or a host that
 * has given all free device memory to its fixed KV pools.
 *
 * The split-KV scratch comes from a device array built into the library,
 * GA_NOALLOC_SCRATCH_BYTES per GPU, held by every GPU that loads the library
 * until the process exits.  The caller still passes q, the pools, the page
 * table, seq_lens and out exactly as for ga_decode_global_hd512.
 *   - plan->workspace_bytes > GA_NOALLOC_SCRATCH_BYTES is rejected with
 *     GA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it together with the current context;
 *     make that first call before any stream capture.  A call made in another
 *     context of the device (after cudaDeviceReset, or a driver-API context
 *     made current) looks the address up again: the first call there should
 *     also come before any capture.
 *   - A plan built with GA_PLAN_TOUCH_LOG is rejected (GA_ERR_INVALID_ARG):
 *     the log would land in the built-in array, out of the caller's reach.
 *   - Every call shares the one array: calls whose kernels overlap on the GPU
 *     (other streams, unordered threads) race on it and give wrong results.
 *     The array keeps the last call's contents; nothing in it needs to start
 *     at zero.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define GA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int ga_decode_global_hd512_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                   int32_t kv_dtype, const float* k_scale, const float* v_scale,
                                   const int32_t* page_table, int64_t pt_stride,
                                   const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t page_size, int64_t num_pages,
                                   float scale, const ga_plan* plan, void* out,
                                   int32_t* err_word, ga_stream_t stream);

/*
 * ga_read_stream -- measurement helper, not part of the decode path: reads
 * `bytes` of device memory at src once with 16-byte non-allocating loads
 * (every SM, a grid of 8 CTAs per SM) and folds them into one word, so that
 * a caller can time the practical HBM read ceiling the decode kernels stream
 * against ("Gemma 4 31B on vLLM -- operating-point reference", Three
 * load-bearing facts: decode throughput saturates on HBM bandwidth).
 *   src: device memory, 16-byte aligned; bytes a multiple of 16 (> 0).
 *   sink: one device uint64, written only if the fold hits a fixed value.
 * Errors: GA_ERR_INVALID_ARG for a null / unaligned pointer or bad size.
 */
int ga_read_stream(const void* src, int64_t bytes, void* sink, ga_stream_t stream);

/* Name of a GA_* status code (static string). */
const char* ga_strerror(int status);

/* GA_OK for a zero device error word, else GA_ERR_DEVICE_CHECK. */
int ga_check_error_word(int32_t word);

/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t ga_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* GA_H_ */
