// ga_mq_tc.cu -- multi-query paged decode over bf16 pools (S query tokens per
// row at its last S positions, causal inside the chunk) with both products on
// the fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The method is the paged softmax attention of both families ("[Model] Gemma 4
// M3 31B", Acceptance Criteria: sliding windows of 1024 with the 1023 / 1024 /
// 1025 boundaries, full-context hd512 layers), with the S queries of a row as
// extra (query, head) columns of each kv head: g query heads give g * S
// columns, each with its own causal and window mask ("Gemma 4 31B on vLLM --
// operating-point reference", Operating-point recipes, LIGHT: EAGLE3 verify of
// 3 speculative tokens; "visible-cx/Gemma-4-31B-CoreAI" model card,
// hybrid-pf64/ bundles: prefill chunks of 64 tokens with a query axis and an
// intra-chunk causal mask).
//
// Why a separate kernel.  From a few dozen columns per kv head on, the work
// is a dense contraction (4 D flops per key and column), and the mma.sync
// decode kernels, which give each warp 8 columns, run it at a few percent of
// the tensor rate.  Here one thread issues the products of a whole stage.
//
// One unit = (row chunk, kv head, tile of 64 columns).  Per stage of 128 keys
// (8 pages), N = 64 columns, K = 16 per instruction, fp32 accumulate:
//   S^T [128 keys x 64]  = K [keys x D] . q^T       A = K (K-major), B = q (K-major)
//   O^T [128 dims x 64] += V^T [dims x keys] . P^T  A = V^T (MN-major), B = P^T (K-major)
//   l   [128 x 64]      += 1 [128 x keys] . P^T     every row: the column sums of P
// S^T sits in TMEM lanes = keys, so softmax thread t owns key t of every stage
// and dim t of every 128-dim block of O^T.  TMEM holds two S buffers, O^T
// (D / 128 blocks) and the sums, 64 columns each: 448 of 512 at hd512.
// Columns as M would need O = 128 x 512 fp32, all of TMEM, at hd512.
//
// Shared memory.  K: a ring of 64 KB in slots of one (or two) 64-dim regions
// of a stage, filled by one bulk tensor copy per page that lands as
// [key / 8][region][key % 8] rows: each region's 8-key groups sit at a uniform
// stride in key order over the stage's 8 pages, as the QK product's operand
// needs.  V: a ring of 64 KB in slots of whole page-head blocks
// ([page][D / 64 regions][16 keys][128 B]), one copy per page: the PV product
// takes one page per instruction, so a block's layout serves it as it lands.
// q of the unit as [D / 64][64 rows][128 B] (one copy per region; two
// buffers at hd256), P^T as two [64 columns][128 B] regions, and a constant
// all-ones tile for the sums.  Operand tiles carry the 128-byte swizzle.
//
// Softmax in base 2 with a lazily raised running max: a column's max moves
// only when a score exceeds it by more than SLACK (so P <= 2^16), then O^T and
// the sums are rescaled in TMEM.  P is rounded to bf16 once and feeds both the
// output and the sums, so numerator and denominator see the same weights.
//
// Roles (256 threads): warps 0-3 softmax and output; warp 4 streams K pages
// and the unit's q rows, warp 5 streams V pages; warp 6 allocates TMEM and its
// lane 0 issues QK; warp 7 zeroes V rows that no query attends (below the
// window, past the row's end, pages with an invalid id: P is 0 there but
// 0 x NaN is not 0) and its lane 0 issues PV and the sums.  Hand-offs are
// mbarriers; every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math_constants.h>

#include "ga_decode_common.cuh"

namespace ga {

namespace mq {

constexpr int NC = kTcColTile;                    // columns per unit: N of every product
constexpr int KEYS = 128;                         // keys per stage: M of the QK product
constexpr int SPG = KEYS / kPageSize;             // pages per stage
// K and V rings of 64 KB each, in slots of GA_MQ_SLOT_KB: 32 KB (2 slots: a K
// slot is a 128-dim block of a stage, a V slot two hd512 pages) or, as a
// build option, 16 KB (4 slots of one 64-dim region / one page: more of each
// ring in flight, but more barriers and commits per stage; measured slower,
// S = 64 global 10.95 vs 9.69 ms).
#ifndef GA_MQ_SLOT_KB
#define GA_MQ_SLOT_KB 32
#endif
constexpr int SLOT_BYTES = GA_MQ_SLOT_KB * 1024;    // a K or V slot
constexpr int K_REGIONS = SLOT_BYTES / (KEYS * 128); // 64-dim regions of a stage per K slot
static_assert(K_REGIONS == 1 || K_REGIONS == 2, "K slot: one or two 64-dim regions");
constexpr int QREG_BYTES = NC * 128;              // [64 columns][64 dims] bf16
constexpr int PREG_BYTES = NC * 128;              // [64 columns][64 keys] bf16
constexpr int P_BYTES = 2 * PREG_BYTES;           // P^T of a stage
constexpr int ONES_BYTES = 4096;                  // [16 keys][128 rows] bf16 ones
constexpr int NKS = 65536 / SLOT_BYTES, NVS = NKS; // K and V slots
constexpr int NSW = 4;                            // softmax warps
constexpr int KP_WARP = 4, VP_WARP = 5, QK_WARP = 6, PV_WARP = 7;
constexpr int NTHREADS = 256;
constexpr int TM_S = 0, TM_O = 2 * NC;            // two S buffers, then O^T, then the sums
constexpr float SLACK = 16.0f;
constexpr uint32_t FULL = 0xffffffffu;

// barriers: k_full / k_empty [NKS], v_full / v_empty [NVS], s_full / s_free
// [2], p_full, p_half (the products on keys 0..63 ran), pv_done, o_free,
// q_full / q_free [2], fin
constexpr int B_KFULL = 0, B_KEMPTY = B_KFULL + NKS, B_VFULL = B_KEMPTY + NKS,
              B_VEMPTY = B_VFULL + NVS, B_SFULL = B_VEMPTY + NVS, B_SFREE = B_SFULL + 2,
              B_PFULL = B_SFREE + 2, B_PHALF = B_PFULL + 1, B_PVDONE = B_PHALF + 1,
              B_OFREE = B_PVDONE + 1,
              B_QFULL = B_OFREE + 1, B_QFREE = B_QFULL + 2, B_FIN = B_QFREE + 2,
              NBARS = B_FIN + 1;

template <int D_>
struct Geo {
    static constexpr int D = D_;
    static constexpr int NDC = D / 128;            // 128-dim blocks: O^T blocks
    static constexpr int NR = D / 64;              // 64-dim regions (128 B of bf16)
    static constexpr int NQB = D == 256 ? 2 : 1;   // q buffers
    static constexpr int Q_BYTES = NR * QREG_BYTES;
    static constexpr int BLOCK_BYTES = kPageSize * D * 2;       // one page-head block
    static constexpr int KSPS = NR / K_REGIONS;                 // K slots per stage
    static constexpr int PPS = SLOT_BYTES / BLOCK_BYTES;        // pages per V slot
    static constexpr int VSPS = SPG / PPS;                      // V slots per stage
    static constexpr int TM_L = TM_O + NDC * NC;                // the column sums
    static constexpr int TMEM_COLS = TM_L + NC <= 256 ? 256 : 512;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NKS * SLOT_BYTES;
    static constexpr int OFF_Q = OFF_V + NVS * SLOT_BYTES;
    static constexpr int OFF_P = OFF_Q + NQB * Q_BYTES;
    static constexpr int OFF_ONES = OFF_P + P_BYTES;
    static constexpr int OFF_RED = OFF_ONES + ONES_BYTES;        // [NC][NSW] column maxima
    static constexpr int OFF_ALPHA = OFF_RED + NC * NSW * 4;     // [NC] rescale factors
    static constexpr int OFF_MAX = OFF_ALPHA + NC * 4;           // [NC] running maxima
    static constexpr int OFF_MSAFE = OFF_MAX + NC * 4;           // [NC] max, 0 for -inf
    static constexpr int OFF_MTH = OFF_MSAFE + NC * 4;           // [NC] max + SLACK
    static constexpr int OFF_COLQ = OFF_MTH + NC * 4;            // [NC] query index of a column
    static constexpr int OFF_PREFIX = OFF_COLQ + NC * 4;
    static constexpr int OFF_BARS = (OFF_PREFIX + (kMaxBatch + 1) * 4 + 7) / 8 * 8;
    static constexpr int SMEM_USED = OFF_BARS + NBARS * 8;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;          // slack for 1024-byte alignment
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(OFF_V % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_P % 1024 == 0 &&
                      OFF_ONES % 1024 == 0 && Q_BYTES % 1024 == 0 && BLOCK_BYTES % 1024 == 0,
                  "swizzle-128B operands need 1024-byte aligned tiles");
    static_assert(PPS * BLOCK_BYTES == SLOT_BYTES && VSPS * PPS == SPG, "V slots");
    static_assert(TM_L + NC <= TMEM_COLS, "tensor memory");
};

// Page ids of pages 32 j .. 32 j + 31 of a unit (one per lane), -1 past its end.
__device__ __forceinline__ int32_t page_ids32(const int32_t* tbl, int np, int j, int lane) {
    const int i = 32 * j + lane;
    return i < np ? __ldg(tbl + i) : -1;
}

// ------------------------------------------------------------------ producers

// Warps 4 (K, plus each unit's q rows) and 5 (V).  Lanes 0..7 hold the pages
// of a stage.  K: for each 128-dim block of each stage, wait until the ring
// slot is free, arm its "full" barrier with the bytes of the good pages, and
// copy each page's two 64-dim regions.  V: for each slot of PPS pages, the
// same with one copy of each whole page-head block.  Pages with an invalid id
// are reported by the K warp and copied by neither.
template <class G, bool IS_K>
__device__ void producer(const CUtensorMap* tm, const CUtensorMap* tmQ, const DecodeParams& p,
                         const int32_t* pre, int64_t U, uint32_t base, uint32_t bars,
                         volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    // Test hook: nothing is armed or copied for CTA 0, so the other roles'
    // bounded waits run out and report GA_DEVERR_TIMEOUT.
    if (p.test_wait_timeout && blockIdx.x == 0) return;
    constexpr int NS = IS_K ? NKS : NVS;
    constexpr int B_FULLB = IS_K ? B_KFULL : B_VFULL, B_EMPTYB = IS_K ? B_KEMPTY : B_VEMPTY;
    constexpr uint32_t OFF = IS_K ? G::OFF_K : G::OFF_V;
    constexpr int SLOTS_PER_STAGE = IS_K ? G::KSPS : G::VSPS;
    // Pages of K and V are read by every column tile of a kv head: keep them
    // in L2 at normal priority.
    const uint64_t pol = l2_evict_normal_policy();
    uint32_t seq = 0, k = 0;               // slots armed, units whose q was armed
    bool stop = false;
    auto fail = [&]() {
        if (lane == 0) {
            report(p.err_word, kErrTimeout);
            *abort_flag = 1;
        }
        stop = true;
    };
    UnitCursor cur(p, pre, U);
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        if (x.np == 0) continue;
        if (IS_K) {
            // q rows of the unit into buffer k % NQB once the QK products of
            // the unit that used it last have run
            const uint32_t qb = k % G::NQB;
            bool ok = true;
            if (lane == 0)
                ok = !*abort_flag &&
                     (k < (uint32_t)G::NQB ||
                      wait_or_abort(bar(bars, B_QFREE + (int)qb), (k / G::NQB - 1) & 1, abort_flag));
            if (__shfl_sync(FULL, ok ? 1 : 0, 0) == 0) {
                fail();
                break;
            }
            if (lane == 0) {
                const uint32_t qf = bar(bars, B_QFULL + (int)qb);
                mbar_arrive_expect_tx(qf, (uint32_t)G::Q_BYTES);
                const int32_t r0 = x.b * p.Hq + x.h0;             // first q row of the unit
#pragma unroll
                for (int r = 0; r < G::NR; ++r)
                    tma_load_3d(base + G::OFF_Q + qb * G::Q_BYTES + r * QREG_BYTES, tmQ, qf, 0, r0,
                                r, pol);
            }
            ++k;
        }
        const int32_t* tbl = p.page_table + (int64_t)x.b * p.pt_stride + x.p0;
        const bool log = IS_K && p.touch_log != nullptr && x.c == 0 && x.hg == 0;
        const int nst = (x.np + SPG - 1) / SPG;
        int32_t ids = page_ids32(tbl, x.np, 0, lane), ids_nxt = page_ids32(tbl, x.np, 1, lane);
        for (int s = 0; s < nst && !stop; ++s) {
            if (s > 0 && s % 4 == 0) {           // next 32 page ids, one batch ahead
                ids = ids_nxt;
                ids_nxt = page_ids32(tbl, x.np, s / 4 + 1, lane);
            }
            const int pl = lane & (SPG - 1);
            const int pi = SPG * s + pl;
            const int32_t pid = __shfl_sync(FULL, ids, (SPG * (s % 4) + pl) & 31);
            const bool present = lane < SPG && pi < x.np;
            const bool valid_id = present && page_ok(pid, p.num_pages);
            const int32_t y = valid_id ? page_block_row(pid, x.c, p.Hkv) : 0;
            const bool good = valid_id && GA_CHK(y >= 0 && (int64_t)y + kPageSize <= p.pool_rows);
            const uint32_t gm = __ballot_sync(FULL, good);
            if (IS_K) {
                if (present && !good) report(p.err_word, valid_id ? kErrSelfCheck : kErrPageId);
                if (log && present && pi < p.touch_stride && GA_CHK(x.rc < p.rc_capacity))
                    p.touch_log[x.rc * p.touch_stride + pi] = pid;
            }
#pragma unroll 1
            for (int j = 0; j < SLOTS_PER_STAGE; ++j) {
                const uint32_t slot = seq % NS;
                bool ok = true;
                if (lane == 0)
                    ok = !*abort_flag && wait_or_abort(bar(bars, B_EMPTYB + (int)slot),
                                                       ((seq / NS) & 1) ^ 1, abort_flag);
                if (__shfl_sync(FULL, ok ? 1 : 0, 0) == 0) {
                    fail();
                    break;
                }
                const uint32_t fb = bar(bars, B_FULLB + (int)slot);
                const uint32_t dst0 = base + OFF + slot * SLOT_BYTES;
                if (IS_K) {
                    // regions K_REGIONS j .. of every page as one box of 2 KB per
                    // region: page pl fills rows 16 K_REGIONS pl .. of the slot
                    if (lane == 0)
                        mbar_arrive_expect_tx(fb, (uint32_t)__popc(gm) * (uint32_t)K_REGIONS * 2048u);
                    __syncwarp();
                    if (good)
                        tma_load_5d(dst0 + (uint32_t)pl * (uint32_t)(K_REGIONS * 2048), tm, fb, 0, 0,
                                    K_REGIONS * j, 0, y / kPageSize, pol);
                } else {
                    // pages PPS j .. PPS j + PPS - 1, whole page-head blocks
                    const uint32_t sm = (gm >> (G::PPS * j)) & ((1u << G::PPS) - 1u);
                    if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)__popc(sm) * G::BLOCK_BYTES);
                    __syncwarp();
                    if (good && pl / G::PPS == j)
                        tma_load_3d(dst0 + (uint32_t)(pl % G::PPS) * G::BLOCK_BYTES, tm, fb, 0, y, 0,
                                    pol);
                }
                ++seq;
            }
        }
    }
    // Never leave with a copy in flight into this CTA's shared memory: wait
    // for the last round each slot (and q buffer) was armed for.
    if (lane < NS && (uint32_t)lane < seq) {
        const uint32_t last = (uint32_t)lane + ((seq - 1 - (uint32_t)lane) / NS) * NS;
        if (!mbar_wait(bar(bars, B_FULLB + lane), (last / NS) & 1)) {
            report(p.err_word, kErrTimeout);
            *abort_flag = 1;
        }
    }
    if (IS_K && lane < G::NQB && (uint32_t)lane < k) {
        const uint32_t last = (uint32_t)lane + ((k - 1 - (uint32_t)lane) / G::NQB) * G::NQB;
        if (!mbar_wait(bar(bars, B_QFULL + lane), (last / G::NQB) & 1)) {
            report(p.err_word, kErrTimeout);
            *abort_flag = 1;
        }
    }
}

// ------------------------------------------------------------------ MMA issuers

// Warp 6, lane 0: S^T(m) = K q^T for the CTA's stages in order, block by
// block as the K slots land, once the S buffer is free and the unit's q rows
// are in.  Each block's commit frees its K slot; the unit's last commit frees
// its q buffer.
template <class G>
__device__ void qk_issuer(const DecodeParams& p, const int32_t* pre, int64_t U, uint32_t base,
                          uint32_t bars, uint32_t tmem, volatile int* abort_flag) {
    constexpr uint32_t IQK = idesc_bf16(KEYS, NC, false, false);
    uint32_t m = 0, kseq = 0, k = 0;          // stages, K slots, active units so far
    bool stop = false;
    UnitCursor cur(p, pre, U);
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        if (x.np == 0) continue;
        const uint32_t qb = k % G::NQB;
        if (!issuer_wait(p, bar(bars, B_QFULL + (int)qb), (k / G::NQB) & 1, abort_flag)) break;
        const uint32_t qa = base + G::OFF_Q + qb * G::Q_BYTES;
        const int nst = (x.np + SPG - 1) / SPG;
        for (int s = 0; s < nst && !stop; ++s, ++m) {
            const uint32_t sb = m & 1;
            if (!issuer_wait(p, bar(bars, B_SFREE + (int)sb), ((m >> 1) & 1) ^ 1, abort_flag)) {
                stop = true;
                break;
            }
            for (int c = 0; c < G::KSPS; ++c, ++kseq) {
                const uint32_t slot = kseq % NKS;
                if (!issuer_wait(p, bar(bars, B_KFULL + (int)slot), (kseq / NKS) & 1, abort_flag)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                const uint32_t ka = base + G::OFF_K + slot * SLOT_BYTES;
                // region r of the slot: 8-key groups K_REGIONS KB apart, from r KB
#pragma unroll
                for (int r = 0; r < K_REGIONS; ++r)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(tmem + TM_S + NC * sb,
                                    smem_desc_sw128(ka + r * 1024 + 32 * kk, 16, K_REGIONS * 1024),
                                    smem_desc_sw128(qa + (K_REGIONS * c + r) * QREG_BYTES + 32 * kk,
                                                    16, 1024),
                                    IQK, (c | r | kk) != 0 ? 1u : 0u);
                tc_commit(bar(bars, B_KEMPTY + (int)slot));     // the K slot may be refilled
            }
            if (stop) break;
            tc_commit(bar(bars, B_SFULL + (int)sb));
        }
        if (stop) break;
        tc_commit(bar(bars, B_QFREE + (int)qb));                 // q buffer may be refilled
        ++k;
    }
}

// Warp 7: for each stage, once the softmax warps have written P(m), for each
// V slot as it lands: zero the slot's V rows that no query of the row attends
// (keys below the window or past the row's end in a copied page, every row of
// a page with an invalid id, never copied), then per page of the slot the
// column sums l += 1 . P^T and O^T += V^T P^T per 128-dim block.  Lane 0
// issues and commits: a slot's commit frees it; the commit after pages 0..3
// releases the first half of P^T (keys 0..63), the stage's last one the whole
// P buffer.  A unit's first products overwrite O^T and the sums (accumulate
// off) once the previous unit's epilogue has read them.
template <class G>
__device__ void pv_warp(const DecodeParams& p, const int32_t* pre, int64_t U, uint8_t* smem,
                        uint32_t base, uint32_t bars, uint32_t tmem, volatile int* abort_flag) {
    constexpr uint32_t IPV = idesc_bf16(128, NC, true, false);
    const int lane = threadIdx.x & 31;
    uint32_t m = 0, vseq = 0, k = 0;          // stages, V slots, active units so far
    bool stop = false;
    auto wait1 = [&](int b, uint32_t parity) -> bool {
        bool ok = true;
        if (lane == 0) ok = !*abort_flag && wait_or_abort(bar(bars, b), parity, abort_flag);
        ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
        if (!ok && lane == 0) {
            report(p.err_word, kErrTimeout);
            *abort_flag = 1;
        }
        return ok;
    };
    // P^T operand of the product for page kp of a stage (16 keys)
    auto pdesc = [&](int kp) {
        return smem_desc_sw128(base + G::OFF_P + (kp >> 2) * PREG_BYTES + 32 * (kp & 3), 16, 1024);
    };
    UnitCursor cur(p, pre, U);
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        if (x.np == 0) continue;
        const int32_t* tbl = p.page_table + (int64_t)x.b * p.pt_stride + x.p0;
        const int nst = (x.np + SPG - 1) / SPG;
        for (int s = 0; s < nst && !stop; ++s, ++m) {
            // rows of page (lane & 7) of this stage that must read as zero
            const int pi = SPG * s + (lane & (SPG - 1));
            uint32_t zmask = 0;
            if (lane < SPG && pi < x.np) {
                const int32_t pid = __ldg(tbl + pi);
                if (!page_ok(pid, p.num_pages)) {
                    zmask = 0xFFFFu;
                } else {
                    const int32_t k0 = (x.p0 + pi) * kPageSize;
                    const int lo_in = min(max(x.g.lo - k0, 0), kPageSize);
                    const int hi_in = min(max(x.g.len - k0, 0), kPageSize);
                    zmask = ((1u << lo_in) - 1u) | (0xFFFFu & ~((1u << hi_in) - 1u));
                }
            }
            const int npg = min(SPG, x.np - SPG * s);
            const bool any_zero = __any_sync(FULL, zmask != 0);
            if ((s == 0 && k > 0 && !wait1(B_OFREE, (k - 1) & 1)) || !wait1(B_PFULL, m & 1)) {
                stop = true;
                break;
            }
            for (int j = 0; j < G::VSPS; ++j, ++vseq) {
                const uint32_t slot = vseq % NVS;
                if (!wait1(B_VFULL + (int)slot, (vseq / NVS) & 1)) {
                    stop = true;
                    break;
                }
                uint8_t* vs = smem + G::OFF_V + slot * SLOT_BYTES;
                for (int i = 0; any_zero && i < G::PPS; ++i) {
                    const uint32_t zm = __shfl_sync(FULL, zmask, G::PPS * j + i);
                    if (zm == 0) continue;
                    // each zeroed row: 128 bytes in each of the NR regions
                    for (int e = lane; e < kPageSize * G::NR * 8; e += 32) {
                        const int row = e / (G::NR * 8), rest = e % (G::NR * 8);
                        if ((zm >> row) & 1u)
                            *reinterpret_cast<uint4*>(vs + i * G::BLOCK_BYTES + (rest >> 3) * 2048 +
                                                      row * 128 + (rest & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_shared();
                }
                __syncwarp();
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t va = base + G::OFF_V + slot * SLOT_BYTES;
                    const uint64_t ones = smem_desc_sw128(base + G::OFF_ONES, 2048, 1024);
                    for (int i = 0; i < G::PPS; ++i) {
                        const int kp = G::PPS * j + i;          // page of the stage
                        if (kp >= npg) break;
                        const uint32_t acc = (s == 0 && kp == 0) ? 0u : 1u;
                        tc_mma_bf16(tmem + G::TM_L, ones, pdesc(kp), IPV, acc);
#pragma unroll
                        for (int c = 0; c < G::NDC; ++c)
                            tc_mma_bf16(tmem + TM_O + NC * c,
                                        smem_desc_sw128(va + i * G::BLOCK_BYTES + 2 * c * 2048, 2048, 1024),
                                        pdesc(kp), IPV, acc);
                    }
                    tc_commit(bar(bars, B_VEMPTY + (int)slot));   // the V slot may be refilled
                    // P^T keys 0..63 (region 0) are read by the products so far
                    if (j == G::VSPS / 2 - 1) tc_commit(bar(bars, B_PHALF));
                }
                __syncwarp();
            }
            if (stop) break;
            if (lane == 0) tc_commit(bar(bars, B_PVDONE));        // P buffer free, O^T and l current
        }
        ++k;
    }
}

// ------------------------------------------------------------------ softmax warps

// Column maxima of v[64] over the warp's 32 lanes by recursive halving: after
// five exchange steps (62 shuffles) lane l holds the maxima of columns 2l and
// 2l + 1 in t[0], t[1].
__device__ __forceinline__ void warp_colmax64(const float (&v)[NC], int lane, float (&t)[32]) {
    const bool b4 = lane & 16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float keep = b4 ? v[i + 32] : v[i], send = b4 ? v[i] : v[i + 32];
        t[i] = fmaxf(keep, __shfl_xor_sync(FULL, send, 16));
    }
    // n values left: pairs (i, i + n / 2) across lanes l, l ^ (n / 4)
#pragma unroll
    for (int n = 32; n >= 4; n >>= 1) {
        const bool b = lane & (n / 4);
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = b ? t[i + n / 2] : t[i], send = b ? t[i] : t[i + n / 2];
            t[i] = fmaxf(keep, __shfl_xor_sync(FULL, send, n / 4));
        }
    }
}

// Warps 0-3.  Thread t owns key t of every stage (TMEM lane t of S^T) and dim
// t of each 128-dim block of O^T.  Per stage: read the 64 scores, mask each
// column (query i = column % S sits at position L - S + i and attends keys j
// with 0 <= (L - S + i) - j < window; keys inside every column's range skip
// the per-column test), raise a column's max only past SLACK (then O^T and the
// sums are rescaled once the previous stage's products have run), compute P
// in bf16 and write P^T once this warp's half of the buffer is free (keys
// 0..63 are released before 64..127).  At the end of a unit: O^T scaled by
// 1 / l to the output (or a split partial and its LSE).  The running maxima
// live in shared memory, one writer per column between barriers.
template <class G>
__device__ void softmax_warps(const DecodeParams& p, const int32_t* pre, int64_t U, uint8_t* smem,
                              uint32_t bars, uint32_t tmem, volatile int* abort_flag) {
    constexpr int D = G::D;
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const uint32_t tl = tmem + ((uint32_t)(32 * w) << 16);     // this warp's TMEM lanes
    float* red = reinterpret_cast<float*>(smem + G::OFF_RED);  // [NC][NSW] maxima
    float* alpha_sm = reinterpret_cast<float*>(smem + G::OFF_ALPHA);
    float* m_sm = reinterpret_cast<float*>(smem + G::OFF_MAX);
    float* msafe_sm = reinterpret_cast<float*>(smem + G::OFF_MSAFE);
    float* mth_sm = reinterpret_cast<float*>(smem + G::OFF_MTH);
    int32_t* colq = reinterpret_cast<int32_t*>(smem + G::OFF_COLQ);
    const float4* msafe4 = reinterpret_cast<const float4*>(msafe_sm);
    const float4* mth4 = reinterpret_cast<const float4*>(mth_sm);
    const int4* colq4 = reinterpret_cast<const int4*>(colq);
    const uint32_t wmask = p.mask_window > 0 ? (uint32_t)p.mask_window : 0x7fffffffu;
    bool stop = false;
    // a wait of one warp that failed, reported at the next 128-thread barrier
    // (every warp keeps the same sequence of named barriers)
    bool late_fail = false;

    auto poll = [&](int b, uint32_t parity) -> bool {
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(bar(bars, b), parity, abort_flag);
        return __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
    };
    auto settle = [&](bool ok) -> bool {
        const bool bad = !ok || late_fail;
        late_fail = false;
        if (named_barrier_or(1, 128, bad)) {
            if (tid == 0) {
                report(p.err_word, kErrTimeout);
                *abort_flag = 1;
            }
            stop = true;
            return false;
        }
        return true;
    };
    auto wait_all = [&](int b, uint32_t parity) -> bool { return settle(poll(b, parity)); };

    // A unit with no attended key: zero output (or a zero partial with an
    // empty LSE).
    auto write_empty = [&](const UnitInfo& x, bool single) {
        for (int f = 0; f < x.nvalid; ++f) {
            const int64_t h = x.h0 + f;
            if (single) {
                const int64_t r = (int64_t)x.b * p.Hq + h;
                if (!GA_CHK((r + 1) * D <= p.out_elems)) continue;
#pragma unroll
                for (int c = 0; c < G::NDC; ++c)
                    p.out[r * D + 128 * c + tid] = __float2bfloat16_rn(0.f);
            } else if (GA_CHK(x.rc < p.rc_capacity && p.partial_o != nullptr)) {
                float* po = p.partial_o + (x.rc * p.Hq + h) * (int64_t)D;
#pragma unroll
                for (int c = 0; c < G::NDC; ++c) po[128 * c + tid] = 0.f;
            }
        }
        if (!single && tid < x.nvalid && GA_CHK(x.rc < p.rc_capacity))
            p.partial_lse[x.rc * p.Hq + x.h0 + tid] = -CUDART_INF_F;
    };

    // This thread's P^T bytes: key tid is byte 2 (tid % 64) of the 128-byte
    // rows of region tid / 64; row f's 16-byte chunk is swizzled by f % 8.
    uint16_t* prow = reinterpret_cast<uint16_t*>(smem + G::OFF_P + (tid >> 6) * PREG_BYTES);
    const int pch = (tid & 63) >> 3, pin = tid & 7;
    int poff[8];                                // element offset of row f (f % 8 = i) in row 0
#pragma unroll
    for (int i = 0; i < 8; ++i) poff[i] = ((pch ^ i) << 3) | pin;

    uint32_t n = 0;                             // stages so far
    UnitCursor cur(p, pre, U);
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        const bool single = (x.g.chunks == 1);
        const int nst = (x.np + SPG - 1) / SPG;
        if (nst == 0) {
            write_empty(x, single);
            continue;
        }
        if (tid < NC) {
            m_sm[tid] = -CUDART_INF_F;
            msafe_sm[tid] = 0.f;
            mth_sm[tid] = -CUDART_INF_F;
            colq[tid] = (x.hg * NC + tid) % p.S;   // column tid is query i of its head
        }
        named_barrier(1, 128);                  // before anyone reads them
        const int32_t* tbl = p.page_table + (int64_t)x.b * p.pt_stride + x.p0;
        int32_t pid_next = (tid >> 4) < x.np ? __ldg(tbl + (tid >> 4)) : -1;
        for (int s = 0; s < nst; ++s) {
            const uint32_t ms = n + (uint32_t)s, sb = ms & 1;
            const int32_t pid = pid_next;       // page of this thread's key; next stage's on its way
            {
                const int pn = SPG * (s + 1) + (tid >> 4);
                pid_next = pn < x.np ? __ldg(tbl + pn) : -1;
            }
            if (!wait_all(B_SFULL + (int)sb, (ms >> 1) & 1)) break;
            tc_fence_after();
            uint32_t sr[NC];
#pragma unroll
            for (int q4 = 0; q4 < NC / 16; ++q4)
                tmem_ld16(tl + TM_S + NC * sb + 16 * q4,
                          *reinterpret_cast<uint32_t(*)[16]>(&sr[16 * q4]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars, B_SFREE + (int)sb));
            const int npg = min(SPG, x.np - SPG * s);
            const bool present = (tid >> 4) < npg && page_ok(pid, p.num_pages);
            const int32_t kj = (x.p0 + SPG * s) * kPageSize + tid;
            const int32_t dbase = x.g.len - p.S - kj;  // (position of query i) - kj = dbase + i
            // key inside every column's window: no per-column test
            const bool inside = present && x.nvalid == NC && dbase >= 0 &&
                                (uint32_t)(dbase + p.S - 1) < wmask;
            float sc[NC];
            if (inside) {
#pragma unroll
                for (int f = 0; f < NC; ++f) sc[f] = __uint_as_float(sr[f]) * p.scale_log2;
            } else {
#pragma unroll
                for (int f4 = 0; f4 < NC / 4; ++f4) {
                    const int4 qv = colq4[f4];
                    const int qf[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int f = 4 * f4 + e;
                        const bool valid = present && f < x.nvalid && (uint32_t)(dbase + qf[e]) < wmask;
                        sc[f] = valid ? __uint_as_float(sr[f]) * p.scale_log2 : -CUDART_INF_F;
                    }
                }
            }
            bool grow = false;
#pragma unroll
            for (int f4 = 0; f4 < NC / 4; ++f4) {
                const float4 t4 = mth4[f4];
                grow |= (sc[4 * f4] > t4.x) | (sc[4 * f4 + 1] > t4.y) | (sc[4 * f4 + 2] > t4.z) |
                        (sc[4 * f4 + 3] > t4.w);
            }
            bool rescale = false;
            if (named_barrier_or(1, 128, grow)) {
                // this stage's column maxima over the 128 keys
                {
                    float t[32];
                    warp_colmax64(sc, lane, t);
                    red[(2 * lane) * NSW + w] = t[0];
                    red[(2 * lane + 1) * NSW + w] = t[1];
                }
                named_barrier(1, 128);
                float a = 1.f;
                if (tid < NC) {
                    const float mo = m_sm[tid];
                    const float4 r4 = *reinterpret_cast<const float4*>(red + tid * NSW);
                    const float M = fmaxf(mo, fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w)));
                    // O^T and l hold this column's weights at the old max: scale them
                    a = (mo == -CUDART_INF_F || M == mo) ? 1.f : ex2_approx(mo - M);
                    alpha_sm[tid] = a;
                    m_sm[tid] = M;
                    msafe_sm[tid] = (M == -CUDART_INF_F) ? 0.f : M;
                    mth_sm[tid] = M + SLACK;
                }
                rescale = named_barrier_or(1, 128, a != 1.f);   // also publishes the maxima
            }
            // P^T row f, key tid: 2^(s - m) in bf16, two columns per conversion,
            // computed before the wait for the P buffer
            uint32_t pk[NC / 2];
#pragma unroll
            for (int f4 = 0; f4 < NC / 4; ++f4) {
                const float4 mv = msafe4[f4];
                pk[2 * f4] = pack_bf16x2(ex2_approx(sc[4 * f4] - mv.x), ex2_approx(sc[4 * f4 + 1] - mv.y));
                pk[2 * f4 + 1] =
                    pack_bf16x2(ex2_approx(sc[4 * f4 + 2] - mv.z), ex2_approx(sc[4 * f4 + 3] - mv.w));
            }
            // this warp's half of the P buffer (keys 0..63: warps 0-1, region 0)
            // is free once the previous stage's products on it have run
            if (ms > 0 && !poll(w < 2 ? B_PHALF : B_PVDONE, (ms - 1) & 1)) late_fail = true;
#pragma unroll
            for (int f = 0; f < NC; f += 2) {
                prow[f * 64 + poff[f & 7]] = (uint16_t)pk[f / 2];
                prow[(f + 1) * 64 + poff[(f + 1) & 7]] = (uint16_t)(pk[f / 2] >> 16);
            }
            // O^T and the sums hold the earlier stages at the old maxima (the
            // products of stage ms - 1 have run, those of stage ms wait for P)
            if (rescale && s > 0) {
                // every product of the previous stage (warps 0-1 waited for half)
                if (!poll(B_PVDONE, (ms - 1) & 1)) late_fail = true;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c <= G::NDC; ++c) {     // O^T blocks, then the sums
#pragma unroll
                    for (int q4 = 0; q4 < NC / 16; ++q4) {
                        uint32_t o[16];
                        const uint32_t ta = tl + TM_O + NC * c + 16 * q4;
                        tmem_ld16(ta, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha_sm[16 * q4 + j]);
                        tmem_st16(ta, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars, B_PFULL));
        }
        if (stop) break;

        // ---- epilogue: 1 / l per column, then O^T from TMEM
        const uint32_t ml = n + (uint32_t)nst - 1;
        if (!wait_all(B_PVDONE, ml & 1)) break;
        tc_fence_after();
        uint32_t lr[NC];
#pragma unroll
        for (int q4 = 0; q4 < NC / 16; ++q4)
            tmem_ld16(tl + G::TM_L + 16 * q4, *reinterpret_cast<uint32_t(*)[16]>(&lr[16 * q4]));
        tmem_ld_wait();
        float inv[NC];
        float Lt = 0.f;                             // column tid's sum, for the LSE
#pragma unroll
        for (int f = 0; f < NC; ++f) {
            const float L = __uint_as_float(lr[f]);
            if (f == tid) Lt = L;
            // only an exactly empty sum means "no keys"; NaN in attended K / V
            // reaches the output as in the definition
            inv[f] = (L == 0.f) ? 0.f : __frcp_rn(L);
        }
        const int64_t r0 = (int64_t)x.b * p.Hq + x.h0;          // output row of column 0
        bool bad_store = false;
#pragma unroll 1
        for (int c = 0; c < G::NDC; ++c) {
#pragma unroll
            for (int q4 = 0; q4 < NC / 16; ++q4) {
                uint32_t o[16];
                tmem_ld16(tl + TM_O + NC * c + 16 * q4, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int f = 16 * q4 + j;
                    if (f >= x.nvalid) continue;
                    const float v = __uint_as_float(o[j]) * inv[f];
                    if (single) {
                        if (GA_CHK((r0 + f + 1) * D <= p.out_elems))
                            p.out[(r0 + f) * D + 128 * c + tid] = __float2bfloat16_rn(v);
                        else
                            bad_store = true;
                    } else if (GA_CHK(x.rc < p.rc_capacity && p.partial_o != nullptr)) {
                        p.partial_o[(x.rc * p.Hq + x.h0 + f) * (int64_t)D + 128 * c + tid] = v;
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bars, B_OFREE));
        if (bad_store) report(p.err_word, kErrSelfCheck);
        if (!single && tid < x.nvalid && GA_CHK(x.rc < p.rc_capacity)) {
            const float mm = m_sm[tid];            // natural-log LSE of column tid
            p.partial_lse[x.rc * p.Hq + x.h0 + tid] =
                (Lt == 0.f) ? -CUDART_INF_F : (mm + log2f(Lt)) * CUDART_LN2_F;
        }
        n += (uint32_t)nst;
    }
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    mq_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmQ, const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    __shared__ uint32_t tmem_slot;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    using G = Geo<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* pre = reinterpret_cast<int32_t*>(smem + G::OFF_PREFIX);
    const uint32_t base = smem_addr(smem);
    const uint32_t bars = base + G::OFF_BARS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NKS; ++s) {
            mbar_init(bar(bars, B_KFULL + s), 1);      // producer's arm (+ copied bytes)
            mbar_init(bar(bars, B_KEMPTY + s), 1);     // QK commit
        }
        for (int s = 0; s < NVS; ++s) {
            mbar_init(bar(bars, B_VFULL + s), 1);      // producer's arm (+ copied bytes)
            mbar_init(bar(bars, B_VEMPTY + s), 1);     // PV commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(bars, B_SFULL + i), 1);      // QK commit
            mbar_init(bar(bars, B_SFREE + i), NSW);    // each softmax warp read S
            mbar_init(bar(bars, B_QFULL + i), 1);      // producer's arm (+ copied bytes)
            mbar_init(bar(bars, B_QFREE + i), 1);      // QK commit
        }
        mbar_init(bar(bars, B_PFULL), NSW);            // each softmax warp wrote P
        mbar_init(bar(bars, B_PHALF), 1);              // PV commit after pages 0..3
        mbar_init(bar(bars, B_PVDONE), 1);             // PV commit
        mbar_init(bar(bars, B_OFREE), NSW);            // each softmax warp read O^T
        mbar_init(bar(bars, B_FIN), 2);                // both issuers' last commits
        mbar_init_fence();
        abort_flag = 0;
    }
    // the all-ones operand of the sums (bf16 1.0 = 0x3F80)
    for (int i = threadIdx.x; i < ONES_BYTES / 16; i += NTHREADS)
        reinterpret_cast<uint4*>(smem + G::OFF_ONES)[i] =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_shared();
    if (warp == KP_WARP && lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmQ);
    }
    if (warp == VP_WARP && lane == 0) prefetch_tensormap(&tmV);
    int64_t total_rc = 0;
    if (!build_row_prefix(p, pre, NTHREADS, &total_rc)) return;
    const int64_t U = total_rc * p.Hkv * p.HG;
    if (warp == QK_WARP) tmem_alloc(smem_addr(&tmem_slot), G::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (warp < NSW) {
        softmax_warps<G>(p, pre, U, smem, bars, tmem, &abort_flag);
    } else if (warp == QK_WARP || warp == PV_WARP) {
        if (warp == QK_WARP) {
            if (lane == 0) qk_issuer<G>(p, pre, U, base, bars, tmem, &abort_flag);
        } else {
            pv_warp<G>(p, pre, U, smem, base, bars, tmem, &abort_flag);
        }
        if (lane == 0) {
            // every product this thread issued has completed before TMEM is freed
            tc_commit(bar(bars, B_FIN));
            if (!mbar_wait(bar(bars, B_FIN), 0)) {
                report(p.err_word, kErrTimeout);
                abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == KP_WARP) {
        producer<G, true>(&tmK, &tmQ, p, pre, U, base, bars, &abort_flag);
    } else if (warp == VP_WARP) {
        producer<G, false>(&tmV, &tmQ, p, pre, U, base, bars, &abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == QK_WARP) tmem_dealloc(tmem, G::TMEM_COLS);
}

}  // namespace mq

// ------------------------------------------------------------------ host

template <int D>
static int run_mq(const DecodeArgs& a) {
    const ga_plan& pl = *a.plan;
    const int32_t S = pl.q_len;
    auto kern = &mq::mq_tc_kernel<D>;
    constexpr int kSmem = mq::Geo<D>::SMEM_BYTES;
    int rc = ensure_smem_attr(reinterpret_cast<const void*>(kern), kSmem, D == 256 ? 20 : 21);
    if (rc != GA_OK) return rc;
    const int64_t rows = a.num_pages * a.num_kv_heads * (int64_t)kPageSize;
    // K: one box = one 128-dim block of a page-head block ([key / 8][64-dim
    // region][key % 8], 4 KB); V: one box = a whole page-head block; q: one
    // 64-dim region of a unit's 64 rows
    CUtensorMap tmK, tmV, tmQ;
    rc = encode_region_map(&tmK, a.k_pool, GA_KV_BF16, a.num_pages * a.num_kv_heads, D,
                           mq::K_REGIONS);
    if (rc != GA_OK) return rc;
    rc = encode_rows_map(&tmV, a.v_pool, GA_KV_BF16, rows, D, kPageSize, 0);
    if (rc != GA_OK) return rc;
    const int64_t qrows = (int64_t)a.batch * a.num_q_heads * S;
    rc = encode_rows_map(&tmQ, a.q, GA_KV_BF16, qrows, D, mq::NC, 1);
    if (rc != GA_OK) return rc;

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.page_table = a.page_table;
    p.seq_lens = a.seq_lens;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const bool split = pl.mode != GA_SPLIT_NONE;
    p.partial_o = split ? reinterpret_cast<float*>(ws + pl.partial_o_offset) : nullptr;
    p.partial_lse = split ? reinterpret_cast<float*>(ws + pl.partial_lse_offset) : nullptr;
    p.touch_log = (pl.flags & GA_PLAN_TOUCH_LOG)
                      ? reinterpret_cast<int32_t*>(ws + pl.touch_log_offset)
                      : nullptr;
    p.err_word = a.err_word;
    p.pt_stride = a.pt_stride;
    p.num_pages = a.num_pages;
    p.rc_capacity = pl.row_chunks;
    p.B = a.batch;
    p.Hq = a.num_q_heads * S;
    p.Hkv = a.num_kv_heads;
    p.group = a.num_q_heads / a.num_kv_heads * S;
    p.TW = mq::NC;
    p.HG = (p.group + mq::NC - 1) / mq::NC;
    p.window = effective_window(a.window, S);
    p.S = S;
    p.mask_window = a.window;
    p.mode = pl.mode;
    p.splits = pl.splits;
    p.chunk_pages = pl.chunk_pages;
    p.schedule = kScheduleRoundRobin;
    p.touch_stride = pl.touch_stride;
    p.test_wait_timeout = (pl.flags & GA_PLAN_TEST_WAIT_TIMEOUT) ? 1 : 0;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.pool_rows = rows;
    p.out_elems = (int64_t)a.batch * a.num_q_heads * S * D;
    const int grid = pl.grid > 0 ? pl.grid : 1;
    kern<<<grid, mq::NTHREADS, kSmem, a.stream>>>(tmK, tmV, tmQ, p);
    if (cudaGetLastError() != cudaSuccess) return GA_ERR_CUDA;
    if (split && !(pl.flags & GA_PLAN_EXTERNAL_COMBINE))
        return launch_combine(p.partial_o, p.partial_lse, a.plan, a.seq_lens, a.out, a.err_word,
                              a.pt_stride, a.stream);
    return GA_OK;
}

int launch_mq_tc(const DecodeArgs& a) {
    if (a.kv_dtype != GA_KV_BF16 || a.k_pool == a.v_pool) return GA_ERR_UNSUPPORTED;
    if (a.head_dim == 256) return run_mq<256>(a);
    if (a.head_dim == 512) return run_mq<512>(a);
    return GA_ERR_UNSUPPORTED;
}

}  // namespace ga
