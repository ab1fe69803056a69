// ga_decode_tc.cu -- paged decode over an E4M3 KV pool (sliding-window hd256
// and full-context hd512) with both products on the fifth-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// Why a separate kernel.  With E4M3 pages a decode warp that runs its own
// m16n8k32 MMAs spends its time on per-warp latency chains (QK, softmax, P
// split, PV per 16-key page), not on bandwidth.  Here one thread issues the
// MMAs for a whole "superstage" (8 pages = 128 keys at hd256, 4 pages = 64
// keys at hd512) and four warps only run the softmax, so the warps' work per
// byte falls by an order of magnitude.  The method is unchanged: the paged
// softmax attention of the sliding family ("[Model] Gemma 4 M3 31B",
// Acceptance Criteria: windows of 1024 with the 1023 / 1024 / 1025
// boundaries; "[Model] Gemma 4 M2 26B-A4B", Proposed Plan: opt-in FP8 pool
// for the sliding family) and of the global family over the same kind of
// pool ("Gemma 4 31B on vLLM -- operating-point reference": an FP8 KV cache
// covers every layer).
//
// Layout of one superstage in shared memory: a K slot and a V slot of 32 KB.
// Each page-head block arrives as one bulk tensor copy (a 5-D box over all of
// its 128-byte regions) that lands as [key / 8][region][key % 8] rows of 128
// bytes with the 128-byte swizzle, page i of the superstage at 16 D i bytes:
// every region's 8-key groups then sit at one uniform stride (1 KB x D/128) in
// key order, so a single MMA descriptor per region spans the superstage's
// scattered pages.  K and V slots are separate rings: a K
// slot is free again as soon as its QK product has run, a V slot only after
// the softmax and the PV product, so V gets more slots (2 K + 4 V in 192 KB
// keep the copy engine busy).  With one pool for K and V (same pointer) each
// block is fetched once into a V slot that serves both products, and all six
// slots are V slots.
//
// Products (N = 2 NC, K = 32 per instruction, fp32 accumulate):
//   S   [keys x 2NC]  = K [keys x dims]  . Qs^T   (A K-major, B K-major; M = keys
//                                                  of a superstage, 128 or 64)
//   O^T [dims x 2NC] += V^T [dims x keys] . Ps^T  (A MN-major, B K-major; M = 128
//                                                  dims, one product per region)
// The 2 NC columns are a unit's NC (query, head) columns (8, or 16 when a kv
// head has more than 8) twice: q scaled per column by 448 / amax and split
// into E4M3 hi and lo parts (columns f and NC + f), and likewise P (scaled by
// 2^6) into hi and lo; a column's result is the sum of its two halves.  S sits in TMEM lanes = keys (M = 64: key r in lane
// 32 (r / 16) + r % 16), O^T in lanes = dims, so a softmax thread owns one key
// of a superstage and dim t of each 128-dim region.
//
// Roles (256 threads): warps 0-3 softmax and output, warp 4 allocates TMEM
// and its lane 0 issues the QK products, warp 7's lane 0 the PV products
// (an MMA issue holds its thread for ~100 cycles, so one thread for both
// made each product wait behind the other), warp 5 streams pages with bulk
// tensor copies, warp 6 turns each unit's q rows into the E4M3 operand one
// unit ahead.  Every role reads the next unit's length (and the producer its
// page ids) while it works on the current one, so a unit boundary waits on no
// global load.  Hand-offs are mbarriers; every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math_constants.h>

#include "ga_decode_common.cuh"

namespace ga {

namespace tc {

#ifndef GA_TC_NKS
#define GA_TC_NKS 2
#define GA_TC_NVS 4
#endif
constexpr int NKS = GA_TC_NKS;                    // K slots (freed by the QK product)
constexpr int NVS = GA_TC_NVS;                    // V slots (freed by the PV product)
constexpr int NPB = 4;                            // P buffers: the PV of a superstage
                                                  // completes well after the next one's P
constexpr int NSW = 4;                            // softmax warps
constexpr int MMA_WARP = 4, PROD_WARP = 5, Q_WARP = 6, PV_WARP = 7;
constexpr int NTHREADS = 256;
constexpr float PSCALE = 64.0f;                   // P scale: with slack 2^2, P <= 256 < 448
constexpr float MAX_SLACK = 2.0f;

constexpr int al(int x) { return (x + 127) / 128 * 128; }
// barriers: k_full / k_empty [NKS], v_full / v_empty [NVMAX], two each of
// s_full, s_free, NPB each of p_full, pv_done, two each of o_free, q_full,
// q_free, fin, and tok
constexpr int NVMAX = NKS + NVS;                  // V slots when K == V (no K ring)
constexpr int B_KFULL = 0, B_KEMPTY = NKS, B_VFULL = 2 * NKS, B_VEMPTY = 2 * NKS + NVMAX,
              B_SFULL = 2 * NKS + 2 * NVMAX, B_SFREE = B_SFULL + 2,
              B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + NPB, B_OFREE = B_PVDONE + NPB,
              B_QFULL = B_OFREE + 2, B_QFREE = B_QFULL + 2, B_FIN = B_QFREE + 2,
              B_TOK = B_FIN + 1, NBARS = B_TOK + 1;
static_assert(NKS >= 2 && NVS >= 2 && NVS <= 32 && NKS <= 32, "ring depth");

// Geometry per head dim.  Both give 32 KB K and V slots.  ALIAS: K and V
// are one pool; each block is fetched once into a V slot that serves both
// products, and the K ring's memory becomes V slots too.
//
// NC (query, head) columns per unit: 8, or 16 for a kv head with more than 8
// (several queries per row, or a GQA group above 8), so that its pages are
// streamed once for 16 columns.  Every product is then N = 2 NC wide (hi and
// lo parts), S takes two buffers of 2 NC TMEM columns, and the q and P
// operands 2 NC rows; a 16-column unit gives one V slot back to make room
// for them.
//
// HP > 1 (head_dim 256, two pools): a unit spans HP kv heads (its 8 columns
// are their query heads).  A superstage is 8 / HP pages of all HP heads, and
// page i fills rows 16 HP i .. 16 HP i + 16 HP - 1 of each region as
// [key / 8][head][key % 8] (one 5-D box of 2 HP KB per page and region), so
// a head's keys lie in groups of 8 rows, 8 HP rows apart: the QK product runs
// over all 128 rows at once (a row only counts for its own head's columns),
// the PV product runs per head (its own accumulator, K = 32 keys per
// instruction at a group stride of 1 KB x HP), so a NaN in one head's V never
// meets another head's P.
template <int D_, bool ALIAS_ = false, int HP_ = 1, int NC_ = kHeadTile>
struct Geo {
    static constexpr int D = D_;
    static constexpr bool ALIAS = ALIAS_;
    static constexpr int HP = HP_;                        // kv heads per unit
    static constexpr int NC = NC_;                        // (query, head) columns per unit
    static constexpr int NVG = NC > kHeadTile ? NVS - 1 : NVS;   // V slots, two pools
    static constexpr int NVE = ALIAS ? NKS + NVG : NVG;   // V slots in use
    static constexpr int NCH = D / 128;                  // 128-dim regions (128 B of E4M3)
    static constexpr int SSP = HP > 1 ? 8 / HP : (D == 256 ? 8 : 4);   // pages per superstage
    static constexpr int PAGE_ROWS = kPageSize * HP;      // rows a page adds to a region tile
    static constexpr int MQ = SSP * PAGE_ROWS;            // rows per superstage = QK's M
    static constexpr int CHUNK_BYTES = MQ * 128;          // one region: [MQ rows][128 B]
    static constexpr int SLOT_BYTES = NCH * CHUNK_BYTES;  // K or V of a superstage
    static constexpr int BLOCK_BYTES = kPageSize * D;     // K or V of one page-head block
    static constexpr int QREG_BYTES = 2 * NC * 128;       // one region: [2 NC rows][128 B]
    static constexpr int QBUF_BYTES = NCH * QREG_BYTES;   // [region][2 NC rows][128 B]
    static constexpr int PBUF_BYTES = 2 * NC * 128;       // [2 NC rows][up to 128 keys]
    static constexpr int TM_S = 0, TM_O = 4 * NC;         // S: 2 x 2 NC columns, then 2 O
    static constexpr int O_HEAD = 2 * NC * NCH;           // TMEM columns of one head's O
    static constexpr int O_COLS = HP * O_HEAD;            // TMEM columns of one O buffer
    static constexpr int TMEM_COLS = TM_O + 2 * O_COLS <= 128   ? 128
                                     : TM_O + 2 * O_COLS <= 256 ? 256
                                                                : 512;
    static constexpr int PV_STEPS = HP > 1 ? 4 / HP : 0;  // K = 32 products per head and region
    static_assert(HP == 1 || (D == 256 && !ALIAS && (HP == 2 || HP == 4)), "heads per unit");
    static_assert(NC == kHeadTile || (NC == 2 * kHeadTile && HP == 1), "columns per unit");
    // HP == 1: a page-head block arrives as one box over all its regions and
    // lands as [key / 8][region][key % 8] rows, page i at BLOCK_BYTES i: each
    // region's 8-key groups then sit 1 KB x NCH apart, in key order, starting
    // 1 KB x region into the slot.  HP > 1: region tiles CHUNK_BYTES apart, 8-row
    // groups 1 KB apart (rows in [key / 8][head][key % 8] order).
    static constexpr bool ILV = HP == 1;
    // where page i of a superstage starts in a slot: a whole block (HP == 1) or
    // its 16 HP rows of each region tile (HP > 1)
    static constexpr uint32_t PAGE_OFF = ILV ? BLOCK_BYTES : PAGE_ROWS * 128;
    static_assert(SSP * PAGE_OFF == (ILV ? SLOT_BYTES : CHUNK_BYTES), "pages fill a slot");
    static constexpr uint32_t REGION_OFF = ILV ? 1024 : CHUNK_BYTES;   // region c at c x this
    static constexpr uint32_t GROUP_STRIDE = ILV ? 1024 * NCH : 1024;  // QK operand SBO
    // byte offset in a slot of operand row r (the superstage's key r, HP == 1) of region c
    static __device__ __forceinline__ uint32_t row_off(int c, int r) {
        return (uint32_t)c * REGION_OFF + (uint32_t)(r >> 3) * GROUP_STRIDE +
               (uint32_t)(r & 7) * 128u;
    }
    static constexpr int OFF_RING = 0;                    // K slots, then V slots
    static constexpr int OFF_VRING = ALIAS ? OFF_RING : OFF_RING + NKS * SLOT_BYTES;
    static constexpr int OFF_Q = OFF_RING + (NKS + NVG) * SLOT_BYTES;
    static constexpr int OFF_P = OFF_Q + 2 * QBUF_BYTES;
    static constexpr int OFF_RED = OFF_P + NPB * PBUF_BYTES;              // [2][4 warps][NC]
    static constexpr int OFF_QSC = al(OFF_RED + 2 * NSW * NC * 4);        // [2][NC] q scales
    static constexpr int OFF_PREFIX = al(OFF_QSC + 2 * NC * 4);
    static constexpr int OFF_FLAGS = al(OFF_PREFIX + (kMaxBatch + 1) * 4);
    static constexpr int OFF_BARS = al(OFF_FLAGS + NVMAX * 4);
    static constexpr int SMEM_USED = al(OFF_BARS + NBARS * 8);
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0 && CHUNK_BYTES % 1024 == 0,
                  "swizzle-128B operands need 1024-byte aligned tiles");
    static_assert((MQ == 128 || MQ == 64) && SSP * NCH <= 32, "superstage shape");
    static_assert(TM_O + 2 * O_COLS <= TMEM_COLS && TMEM_COLS <= 512, "tensor memory");
};

// Two values -> two E4M3 codes (hi) and the E4M3 codes of their remainders
// (lo), low byte first: hi + lo carries ~8 bits of the value.
__device__ __forceinline__ void split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = f32x2_to_e4m3x2(a, b);
    const uint32_t h = e4m3x2_to_f16x2(hi);
    const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&h));
    lo = f32x2_to_e4m3x2(a - r.x, b - r.y);
}

// ------------------------------------------------------------------ producer

// Who writes this step's token of a unit that holds its row's last page:
// the producer itself for the CTA's first unit when that unit is short (its
// last page is copied right away, before the q warp could have written the
// token), the q warp for every other such unit.
template <class G>
__device__ __forceinline__ bool producer_writes_token(const UnitInfo& x, bool first_unit) {
    return first_unit && (x.np + G::SSP - 1) / G::SSP <= 2;
}

// Warp 5.  For each superstage m of each unit: wait until K slot m % NKS and
// V slot m % NVE are free, arm their "full" barriers with the bytes of the
// good pages, and let lanes 0..SSP-1 each copy one page, K (every 128-dim
// region) before V (K == V: only the V slot, once).  Pages with an invalid id
// are flagged (bit i of flags[m % NVE]) and not copied.
template <class G>
__device__ void producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmK1,
                         const CUtensorMap* tmV1, const DecodeParams& p, const int32_t* pre,
                         int64_t U, uint32_t ring, uint32_t bars, volatile uint32_t* flags,
                         volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    // Test hook: nothing is armed or copied for CTA 0, so the other roles'
    // bounded waits run out and report GA_DEVERR_TIMEOUT.
    if (p.test_wait_timeout && blockIdx.x == 0) return;
    const uint64_t policy = l2_evict_first_policy();
    // page ids of pages 0..31 and 32..63 of a unit, one per lane
    auto first_ids = [&](const UnitInfo& y, int32_t& a, int32_t& b) {
        const int32_t* t = p.page_table + (int64_t)y.b * p.pt_stride + y.p0;
        a = (lane < y.np) ? __ldg(t + lane) : -1;
        b = (32 + lane < y.np) ? __ldg(t + 32 + lane) : -1;
    };
    UnitCursor cur(p, pre, U);
    bool have = cur.more();
    UnitInfo x = {};
    int32_t ids = -1, ids_nxt = -1;
    if (have) {
        x = cur.take(p, pre);
        first_ids(x, ids, ids_nxt);
    }
    uint32_t seq = 0;                 // superstages armed so far
    bool stop = false;
    using Tok = TokenAppend<G::D, GA_KV_E4M3, G::HP>;
    Tok tok;                          // a token this warp writes itself
    bool tokens_written = false;      // the q warp's B_TOK arrival has been seen
    bool first_unit = true;
    while (have && !stop) {
        // The next unit: its length is on its way; once it has arrived (after
        // this unit's first superstage) its first page ids are loaded too.
        const bool has_next = cur.more();
        UnitInfo nx = {};
        int32_t nids = -1, nids_nxt = -1;
        bool nx_ready = !has_next;
        auto ready_next = [&]() {
            if (!nx_ready) {
                nx = cur.take(p, pre);
                first_ids(nx, nids, nids_nxt);
                nx_ready = true;
            }
        };
        if (has_next) {               // the next unit's q rows into L2 for the q warp
            constexpr int LPR = G::D * 2 / 128;           // 128-byte lines per q row
            for (int l = lane; l < G::NC * LPR; l += 32) {
                const int64_t r = (int64_t)unit_q_row(p, cur.nl) + l / LPR;
                if ((r + 1) * G::D <= p.out_elems)
                    prefetch_l2(reinterpret_cast<const char*>(p.q + r * G::D) + 128 * (l % LPR));
            }
        }
        const int32_t* tbl = p.page_table + (int64_t)x.b * p.pt_stride + x.p0;
        const bool log = p.touch_log != nullptr && x.c == 0 && x.hg == 0;
        const bool own_token = producer_writes_token<G>(x, first_unit);
        tok.pending = false;
        if (own_token) tok.start(p, x);
        first_unit = false;
        constexpr int SPB = 32 / G::SSP;  // superstages per batch of 32 page ids
        const int nss = (x.np + G::SSP - 1) / G::SSP;
        for (int s = 0; s < nss; ++s) {
            if (s > 0 && s % SPB == 0) {      // next batch of 32 page ids, one batch ahead
                ids = ids_nxt;
                const int nb = 32 * (s / SPB + 1) + lane;
                ids_nxt = (nb < x.np) ? __ldg(tbl + nb) : -1;
            }
            // the superstage with the row's last page: after the step's token
            if (s == nss - 1) tok.finish(p, __shfl_sync(0xffffffffu, ids, (x.np - 1) & 31));
            const bool tok_wait =
                !tokens_written && !own_token && s == nss - 1 && Tok::due(p, x);
            const uint32_t n = seq, kslot = n % NKS, vslot = n % G::NVE;
            bool ok = true;
            if (lane == 0)
                ok = !*abort_flag && (!tok_wait || wait_or_abort(bar(bars, B_TOK), 0, abort_flag)) &&
                     (G::ALIAS ||
                      wait_or_abort(bar(bars, B_KEMPTY + kslot), ((n / NKS) & 1) ^ 1, abort_flag)) &&
                     wait_or_abort(bar(bars, B_VEMPTY + vslot), ((n / G::NVE) & 1) ^ 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) {
                    report(p.err_word, kErrTimeout);
                    *abort_flag = 1;
                }
                stop = true;
                break;
            }
            tokens_written |= tok_wait;
            const int pl = lane % G::SSP;
            const int pi = G::SSP * s + pl;
            const int32_t pid = __shfl_sync(0xffffffffu, ids, (G::SSP * (s % SPB) + pl) & 31);
            const bool present = lane < G::SSP && pi < x.np;
            const bool valid_id = present && page_ok(pid, p.num_pages);
            // first row of the unit's (first) kv head in the [pages * Hkv * 16, D] view
            const int32_t y = valid_id ? page_block_row(pid, x.c * G::HP, p.Hkv * G::HP) : 0;
            const bool good =
                valid_id && GA_CHK(y >= 0 && (int64_t)y + G::PAGE_ROWS <= p.pool_rows);
            const uint32_t gm = __ballot_sync(0xffffffffu, good);
            const uint32_t pm = __ballot_sync(0xffffffffu, present);
            const uint32_t kfull = bar(bars, B_KFULL + kslot), vfull = bar(bars, B_VFULL + vslot);
            constexpr uint32_t kPageBytes = (uint32_t)(G::HP * G::BLOCK_BYTES);
            if (lane == 0) {
                flags[vslot] = pm & ~gm;
                if (!G::ALIAS) mbar_arrive_expect_tx(kfull, (uint32_t)__popc(gm) * kPageBytes);
                mbar_arrive_expect_tx(vfull, (uint32_t)__popc(gm) * kPageBytes);
            }
            __syncwarp();
            if (good) {
                const uint32_t kd = ring + kslot * G::SLOT_BYTES + (uint32_t)lane * G::PAGE_OFF;
                const uint32_t vd = ring + (uint32_t)G::OFF_VRING + vslot * G::SLOT_BYTES +
                                    (uint32_t)lane * G::PAGE_OFF;
                if constexpr (G::HP > 1) {
                    // one box per region: the page's rows of the unit's HP kv heads
                    static_assert(G::NCH == 2, "one 5-D map per 128-byte region");
                    const int32_t h0 = x.c * G::HP;
                    tma_load_5d(kd, tmK, kfull, 0, 0, h0, 0, pid, policy);
                    tma_load_5d(kd + G::CHUNK_BYTES, tmK1, kfull, 0, 0, h0, 0, pid, policy);
                    tma_load_5d(vd, tmV, vfull, 0, 0, h0, 0, pid, policy);
                    tma_load_5d(vd + G::CHUNK_BYTES, tmV1, vfull, 0, 0, h0, 0, pid, policy);
                } else {
                    // one box per page-head block over all its regions
                    const int32_t blk = y / kPageSize;
                    if (!G::ALIAS) tma_load_5d(kd, tmK, kfull, 0, 0, 0, 0, blk, policy);
                    tma_load_5d(vd, tmV, vfull, 0, 0, 0, 0, blk, policy);
                }
            } else if (present) {
                report(p.err_word, valid_id ? kErrSelfCheck : kErrPageId);
            }
            if (log && present && pi < p.touch_stride && GA_CHK(x.rc < p.rc_capacity))
                p.touch_log[x.rc * p.touch_stride + pi] = pid;
            ++seq;
            ready_next();
        }
        ready_next();                 // a unit without pages
        have = has_next;
        x = nx;
        ids = nids;
        ids_nxt = nids_nxt;
    }
    // Never leave with a copy in flight into this CTA's shared memory: wait
    // for the last round each K and V slot was armed for.
    auto drain = [&](int base, int nslots) {
        if (lane < nslots && (uint32_t)lane < seq) {
            const uint32_t last = (uint32_t)lane + ((seq - 1 - (uint32_t)lane) / nslots) * nslots;
            if (!mbar_wait(bar(bars, base + lane), (last / nslots) & 1)) {
                report(p.err_word, kErrTimeout);
                *abort_flag = 1;
            }
        }
    };
    if (!G::ALIAS) drain(B_KFULL, NKS);
    drain(B_VFULL, G::NVE);
}

// ------------------------------------------------------------------ MMA issuers

// Warp 4, lane 0: S(m) = K q^T for the CTA's superstages in order, once the
// stage's K half has landed, the S buffer is free and the unit's q operand
// is ready.
template <class G>
__device__ void qk_issuer(const DecodeParams& p, const int32_t* pre, int64_t U, uint32_t ring,
                          uint32_t qbuf, uint32_t bars, uint32_t tmem, volatile int* abort_flag) {
    constexpr uint32_t IQK = idesc_e4m3(G::MQ, 2 * G::NC, false, false);
    uint32_t m = 0, k = 0;                        // superstages, active units so far
    bool stop = false;
    UnitCursor cur(p, pre, U);
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        const int nss = (x.np + G::SSP - 1) / G::SSP;
        if (nss == 0) continue;
        const uint32_t qb = k & 1;
        if (!issuer_wait(p, bar(bars, B_QFULL + (int)qb), (k >> 1) & 1, abort_flag)) break;
        for (int s = 0; s < nss; ++s, ++m) {
            // K == V: S reads the V slot the block was fetched into
            const uint32_t slot = G::ALIAS ? m % G::NVE : m % NKS, sb = m & 1;
            if (!issuer_wait(p, bar(bars, (G::ALIAS ? B_VFULL : B_KFULL) + (int)slot),
                             (m / (G::ALIAS ? G::NVE : NKS)) & 1, abort_flag) ||
                !issuer_wait(p, bar(bars, B_SFREE + (int)sb), ((m >> 1) & 1) ^ 1, abort_flag)) {
                stop = true;
                break;
            }
            tc_fence_after();
            const uint32_t ka = ring + (uint32_t)(G::ALIAS ? G::OFF_VRING : G::OFF_RING) +
                                slot * G::SLOT_BYTES,
                           qa = qbuf + qb * G::QBUF_BYTES;
#pragma unroll
            for (int c = 0; c < G::NCH; ++c)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_e4m3(tmem + G::TM_S + 2 * G::NC * sb,
                                smem_desc_sw128(ka + c * G::REGION_OFF + 32 * kk, 16,
                                                G::GROUP_STRIDE),
                                smem_desc_sw128(qa + c * G::QREG_BYTES + 32 * kk, 16, 1024), IQK,
                                (c | kk) != 0 ? 1u : 0u);
            tc_commit(bar(bars, B_SFULL + (int)sb));
            if (!G::ALIAS) tc_commit(bar(bars, B_KEMPTY + (int)slot));  // the K slot may be refilled
        }
        ++k;
    }
}

// Warp 7, lane 0: O += V^T P^T for the CTA's superstages in order, once the
// softmax warps have written P(m) and the stage's V half has landed.  Its commit frees the V slot and the P
// buffer.  A unit's first PV overwrites its O buffer (accumulate off) once
// the epilogue two active units back has read it.
template <class G>
__device__ void pv_issuer(const DecodeParams& p, const int32_t* pre, int64_t U, uint32_t ring,
                          uint32_t pbuf, uint32_t bars, uint32_t tmem, volatile int* abort_flag) {
    constexpr uint32_t IPV = idesc_e4m3(128, 2 * G::NC, true, false);
    uint32_t m = 0, k = 0;
    bool stop = false;
    UnitCursor cur(p, pre, U);
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        const int nss = (x.np + G::SSP - 1) / G::SSP;
        if (nss == 0) continue;
        const uint32_t ob = k & 1;
        for (int s = 0; s < nss; ++s, ++m) {
            const uint32_t slot = m % G::NVE, pb = m % NPB;
            if ((s == 0 &&
                 !issuer_wait(p, bar(bars, B_OFREE + (int)ob), ((k >> 1) & 1) ^ 1, abort_flag)) ||
                !issuer_wait(p, bar(bars, B_PFULL + (int)pb), (m / NPB) & 1, abort_flag) ||
                !issuer_wait(p, bar(bars, B_VFULL + (int)slot), (m / G::NVE) & 1, abort_flag)) {
                stop = true;
                break;
            }
            tc_fence_after();
            const int nks = (min(G::SSP, x.np - G::SSP * s) + 1) / 2;   // 32 keys per MMA
            if constexpr (G::HP > 1) {
                // per head h: its 32-key steps j (pages 2j, 2j + 1), groups of 8
                // keys 8 HP rows apart, into its own accumulator; P^T holds head
                // h's keys at 128 / HP h .. in the same order
#pragma unroll
                for (int c = 0; c < G::NCH; ++c) {
                    const uint32_t va =
                        ring + (uint32_t)G::OFF_VRING + slot * G::SLOT_BYTES + c * G::CHUNK_BYTES;
#pragma unroll
                    for (int h = 0; h < G::HP; ++h) {
                        const uint32_t d =
                            tmem + G::TM_O + G::O_COLS * ob + G::O_HEAD * h + 2 * G::NC * c;
                        for (int j = 0; j < G::PV_STEPS && j < nks; ++j)
                            tc_mma_e4m3(
                                d,
                                smem_desc_sw128(va + 1024 * h + j * 4 * (1024 * G::HP),
                                                G::CHUNK_BYTES, 1024 * G::HP),
                                smem_desc_sw128(
                                    pbuf + pb * G::PBUF_BYTES + 32 * (h * G::PV_STEPS + j), 16, 1024),
                                IPV, (s == 0 && j == 0) ? 0u : 1u);
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < G::NCH; ++c) {
                    const uint32_t d = tmem + G::TM_O + G::O_COLS * ob + 2 * G::NC * c;
                    const uint32_t va =
                        ring + (uint32_t)G::OFF_VRING + slot * G::SLOT_BYTES + c * G::REGION_OFF;
                    // 32 keys per product: 4 groups of 8, GROUP_STRIDE apart
                    for (int ks = 0; ks < nks; ++ks)
                        tc_mma_e4m3(d,
                                    smem_desc_sw128(va + 4 * G::GROUP_STRIDE * ks, G::CHUNK_BYTES,
                                                    G::GROUP_STRIDE),
                                    smem_desc_sw128(pbuf + pb * G::PBUF_BYTES + 32 * ks, 16, 1024),
                                    IPV, (s == 0 && ks == 0) ? 0u : 1u);
                }
            }
            tc_commit(bar(bars, B_VEMPTY + (int)slot));  // the V slot may be refilled
            tc_commit(bar(bars, B_PVDONE + (int)pb));    // P buffer free, O up to date
        }
        ++k;
    }
}

// ------------------------------------------------------------------ q warp

// The q warp, once per launch: this step's token of every other unit of the
// CTA that holds its row's last page, written into that page (the producer
// waits on B_TOK before it copies such a page).  Lane i takes the CTA's
// units i, i + 32, ...: their page-table entries and token lines are fetched
// in parallel, then the warp writes one unit's token at a time.
template <class G>
__device__ void append_tokens(const DecodeParams& p, const int32_t* pre, int64_t U,
                              uint32_t bars) {
    using Tok = TokenAppend<G::D, GA_KV_E4M3, G::HP>;
    const int lane = threadIdx.x & 31;
    for (int64_t u0 = blockIdx.x; u0 < U; u0 += 32 * (int64_t)gridDim.x) {
        const int64_t u = u0 + (int64_t)lane * gridDim.x;
        UnitInfo x = {};
        bool due = false;
        if (u < U) {
            x = unit_info(p, pre, u);
            due = Tok::due(p, x) && !producer_writes_token<G>(x, u == blockIdx.x);
        }
        const int32_t pos = x.g.len - 1, c0 = x.c * G::HP;
        int32_t page = -1;
        if (due) {
            Tok::prefetch(p, x.b, c0, 0, 1);
            page = __ldg(Tok::page_entry(p, x.b, pos));
        }
        for (uint32_t m = __ballot_sync(0xffffffffu, due); m != 0; m &= m - 1) {
            const int j = __ffs(m) - 1;
            Tok::write(p, __shfl_sync(0xffffffffu, x.b, j), __shfl_sync(0xffffffffu, c0, j),
                       __shfl_sync(0xffffffffu, pos, j), __shfl_sync(0xffffffffu, page, j));
        }
    }
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(bars, B_TOK));
}

// One unit's q rows into a q buffer (the layout q_warp describes) and their
// scales, by the 32 lanes of the q warp: LPC lanes per column, each taking
// D / LPC consecutive dims.  LPC x NC = 32 covers all NC columns (rows of
// columns past the unit's valid ones written as zeros); LPC = 16 covers
// columns 0 and 1 only, for units of at most 2 valid columns whose other
// rows are already zero.  A lane holds at most 16 of its 16-byte pieces at
// once: with more (16-column units at hd512) it reads them twice, once for
// the column's amax and once to convert them.
template <class G, int LPC>
__device__ __forceinline__ void prep_q(const DecodeParams& p, const UnitInfo& y, uint8_t* qb_buf,
                                       float* qsc_b) {
    constexpr int DPL = G::D / LPC;                // dims per lane
    constexpr int NW = DPL / 8;                    // 16-byte loads per lane (8 dims each)
    constexpr int PW = NW < 16 ? NW : 16;          // loads held at once
    constexpr int NBLK = NW / PW;
    constexpr bool all_cols = LPC * G::NC == 32;
    static_assert(PW % 2 == 0 && NBLK * PW == NW, "16-dim pieces");
    const int lane = threadIdx.x & 31;
    const int f = lane / LPC, part = lane % LPC, d0 = DPL * part;
    const int64_t row = (int64_t)y.b * p.Hq + y.h0 + f;
    bool have = false;
    if (f < y.nvalid) {
        have = GA_CHK((row + 1) * G::D <= p.out_elems);
        if (!have) report(p.err_word, kErrSelfCheck);
    }
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (have ? row * G::D + d0 : 0));
    uint4 wv[PW];
    auto load = [&](int blk) {
#pragma unroll
        for (int i = 0; i < PW; ++i)
            wv[i] = have ? __ldg(src + PW * blk + i) : make_uint4(0u, 0u, 0u, 0u);
    };
    float am = 0.f;
#pragma unroll
    for (int blk = 0; blk < NBLK; ++blk) {
        load(blk);
#pragma unroll
        for (int i = 0; i < PW; ++i) {
            const uint32_t e[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                am = fmaxf(am, fmaxf(fabsf(bf16_lo(e[j])), fabsf(bf16_hi(e[j]))));
        }
    }
#pragma unroll
    for (int off = 1; off < LPC; off <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    if (part == 0 && f < y.nvalid && !(am < CUDART_INF_F)) report(p.err_word, kErrQRange);
    const float sc = am > 0.f ? am * (1.0f / 448.0f) : 1.0f;
    const float inv = 1.0f / sc;
    if (all_cols || f < y.nvalid) {
#pragma unroll
        for (int blk = 0; blk < NBLK; ++blk) {
            if (NBLK > 1) load(blk);
#pragma unroll
            for (int i = 0; i < PW; i += 2) {     // 16 dims: elements of wv[i], wv[i + 1]
                const uint32_t e[8] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w,
                                       wv[i + 1].x, wv[i + 1].y, wv[i + 1].z, wv[i + 1].w};
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h01, l01, h23, l23;
                    split_e4m3x2(bf16_lo(e[2 * j]) * inv, bf16_hi(e[2 * j]) * inv, h01, l01);
                    split_e4m3x2(bf16_lo(e[2 * j + 1]) * inv, bf16_hi(e[2 * j + 1]) * inv, h23,
                                 l23);
                    hw[j] = h01 | (h23 << 16);
                    lw[j] = l01 | (l23 << 16);
                }
                const int dd = d0 + 8 * (PW * blk + i);          // first dim of the piece
                const int jj = (dd & 127) >> 4;                  // 16-byte chunk of the 128-byte row
                uint8_t* region = qb_buf + (dd >> 7) * G::QREG_BYTES;
                *reinterpret_cast<uint4*>(region + f * 128 + ((jj ^ (f & 7)) << 4)) =
                    make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(region + (G::NC + f) * 128 + ((jj ^ (f & 7)) << 4)) =
                    make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
        if (part == 0) qsc_b[f] = sc;
    }
}

// Warp 6.  For each active unit (one with pages), in the order the MMA issuer
// takes them: the unit's q rows as the QK operand in buffer k % 2 -- column f
// scaled by 448 / amax_f, its E4M3 hi part in row f and lo part in row NC + f
// of each 128-dim region ([2 NC rows][128 B], 128-byte swizzle); rows of
// columns past the unit's valid ones are zero.  Lane l takes column l / LPC,
// dims D/LPC (l % LPC) .. +D/LPC-1 (LPC = 32 / NC).  Buffer k % 2 is
// rewritten once the softmax warps are done with active unit k - 2 (its
// scales read, all its S consumed).
template <class G, int NV>
__device__ void q_warp(const DecodeParams& p, const int32_t* pre, int64_t U, uint8_t* smem,
                       uint32_t bars, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    float* qsc = reinterpret_cast<float*>(smem + G::OFF_QSC);  // [2][NC]
    uint8_t* qbuf = smem + G::OFF_Q;
    // At most 2 valid columns per unit (NV = 2: one kv head of GQA group 1 or
    // 2, the same for every unit of a launch): 16 lanes per column, and the
    // rows of the other columns are zeroed once here instead of for every unit.
    constexpr bool narrow = NV == 2;
    if constexpr (narrow) {
        for (int i = lane; i < 2 * G::QBUF_BYTES / 16; i += 32)
            reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
        if (lane < 2 * G::NC) qsc[lane] = 1.0f;
    }
    UnitCursor cur(p, pre, U);
    uint32_t k = 0;
    // this step's tokens once the first unit's q is ready (or at the end)
    bool tokens = p.k_new == nullptr;
    while (cur.more()) {
        if (k == 1 && !tokens) {
            append_tokens<G>(p, pre, U, bars);
            tokens = true;
        }
        const UnitInfo y = cur.take(p, pre);
        if (y.np == 0) continue;
        const uint32_t qb = k & 1;
        bool ok = k < 2 || wait_or_abort(bar(bars, B_QFREE + (int)qb), ((k - 2) >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) {
                report(p.err_word, kErrTimeout);
                *abort_flag = 1;
            }
            break;
        }
        prep_q<G, narrow ? 16 : 32 / G::NC>(p, y, qbuf + qb * G::QBUF_BYTES, qsc + qb * G::NC);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bars, B_QFULL + (int)qb));
        ++k;
    }
    if (!tokens) append_tokens<G>(p, pre, U, bars);
}

// ------------------------------------------------------------------ softmax warps

// N consecutive TMEM columns of this warp's 32 lanes, 16 at a time.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N % 16 == 0, "whole 16-column loads");
#pragma unroll
    for (int i = 0; i < N / 16; ++i)
        tmem_ld16(taddr + 16 * i, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * i));
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N % 16 == 0, "whole 16-column stores");
#pragma unroll
    for (int i = 0; i < N / 16; ++i)
        tmem_st16(taddr + 16 * i, *reinterpret_cast<const uint32_t(*)[16]>(r + 16 * i));
}

// Warps 0-3.  Thread t owns one key of every superstage (M = 128: key t;
// M = 64: key 16 w + lane for lanes 0..15 of warp w, the TMEM lanes the
// product writes) and dim t of each 128-dim region of O.  Per superstage:
// read S, mask, online
// softmax in base 2 (the running max is raised only when a score exceeds it
// by more than MAX_SLACK; then O is rescaled in TMEM), write P's hi / lo
// E4M3 parts as the PV operand, zero V rows the PV reads but no query
// attends.  At the end of a unit: read O and write the output (or a split
// partial and its LSE).  NV (2, 4, 8, or 16 for 16-column units) bounds the
// valid (query, head) columns of every unit; columns NV.. of P stay zero.
// Column f's hi part is TMEM / operand column f, its lo part NC + f.
template <class G, int NV>
__device__ void softmax_warps(const DecodeParams& p, const int32_t* pre, int64_t U, uint8_t* smem,
                              uint32_t bars, uint32_t tmem, volatile uint32_t* flags,
                              volatile int* abort_flag) {
    constexpr int D = G::D;
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const uint32_t tl = tmem + ((uint32_t)(32 * w) << 16);     // this warp's TMEM lanes
    constexpr int NC = G::NC;
    float* red = reinterpret_cast<float*>(smem + G::OFF_RED);  // [max | sum][4 warps][NC]
    const float* qsc = reinterpret_cast<const float*>(smem + G::OFF_QSC);
    uint8_t* pbuf = smem + G::OFF_P;
    uint8_t* ring = smem + G::OFF_RING;
    // This thread's key within a superstage.  M = 128: key t of thread t.
    // M = 64: the product writes key 16 w + r to lane r < 16 of warp w's TMEM
    // lanes, so lanes r and 16 + r share that key and split its columns
    // (SPLIT): lane r takes columns 0 .. CW - 1 of the unit, lane 16 + r
    // columns CW .. 2 CW - 1, its S values passed over by shuffles.  Every
    // thread still holds the running maxima of all columns (O^T's rescale
    // needs them); the V rows of unattended keys are zeroed by lanes < 16.
    constexpr bool SPLIT = G::MQ == 64;
    constexpr int CW = SPLIT ? NV / 2 : NV;         // columns of this thread
    static_assert(!SPLIT || (G::HP == 1 && NV % 2 == 0), "column split");
    const bool upper = SPLIT && lane >= 16;
    const int cb = upper ? CW : 0;                  // this thread's first column
    const bool zero_lane = G::MQ == 128 || lane < 16;
    const int kss = G::MQ == 128 ? tid : 16 * w + (lane & 15);
    bool stop = false;

    // P columns past NV are never written: zero them once.
    for (int i = tid; i < NPB * G::PBUF_BYTES / 16; i += 128)
        reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);

    // A wait polled by one lane per warp, with one outcome for all 128 threads
    // (the named barrier also orders the lanes after the poller).
    auto poll = [&](int b, uint32_t parity) -> bool {
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(bar(bars, b), parity, abort_flag);
        return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    auto settle = [&](bool ok) -> bool {
        if (named_barrier_or(1, 128, !ok)) {
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
                for (int c = 0; c < G::NCH; ++c)
                    p.out[r * D + 128 * c + tid] = __float2bfloat16_rn(0.f);
            } else if (GA_CHK(x.rc < p.rc_capacity && p.partial_o != nullptr)) {
                float* po = p.partial_o + (x.rc * p.Hq + h) * (int64_t)D;
#pragma unroll
                for (int c = 0; c < G::NCH; ++c) po[128 * c + tid] = 0.f;
            }
        }
        if (!single && tid < x.nvalid && GA_CHK(x.rc < p.rc_capacity))
            p.partial_lse[x.rc * p.Hq + x.h0 + tid] = -CUDART_INF_F;
    };

    constexpr int GQ = NV / G::HP;              // (query, head) columns per kv head of a unit
    uint32_t n = 0, k = 0;                      // superstages, active units so far
    UnitCursor cur(p, pre, U);
    float nks[G::HP], nvs[G::HP];               // the pending unit's K / V scales, per kv head
    auto load_scales = [&]() {
#pragma unroll
        for (int h = 0; h < G::HP; ++h) {
            nks[h] = __ldg(p.k_scale + cur.nl.c * G::HP + h);
            nvs[h] = __ldg(p.v_scale + cur.nl.c * G::HP + h);
        }
    };
#pragma unroll
    for (int h = 0; h < G::HP; ++h) nks[h] = nvs[h] = 1.f;
    if (cur.more()) load_scales();
    while (cur.more() && !stop) {
        const UnitInfo x = cur.take(p, pre);
        float ksc[G::HP], vsc[G::HP];
#pragma unroll
        for (int h = 0; h < G::HP; ++h) {
            ksc[h] = nks[h];
            vsc[h] = nvs[h];
        }
        if (cur.more()) load_scales();
        const bool single = (x.g.chunks == 1);
        const int nss = (x.np + G::SSP - 1) / G::SSP;
        if (nss == 0) {
            write_empty(x, single);
            continue;
        }
        const uint32_t qb = k & 1;
        if (!wait_all(B_QFULL + (int)qb, (k >> 1) & 1)) break;     // this unit's q scales
        float kf[CW], l[CW], m[NV];             // m: every column's running max
        int32_t clo[CW], chi[CW];
#pragma unroll
        for (int j = 0; j < CW; ++j) {
            const int f = cb + j;
            kf[j] = p.scale_log2 * ksc[SPLIT ? 0 : j / GQ] * qsc[qb * NC + f];
            // query i = column % S sits at position L - S + i: keys [clo, chi)
            const int32_t pos = x.g.len - p.S + (x.hg * NC + f) % p.S;
            chi[j] = f < x.nvalid ? pos + 1 : 0;
            clo[j] = f < x.nvalid ? (p.mask_window > 0 ? max(0, pos - p.mask_window + 1) : 0) : 0;
            l[j] = 0.f;
        }
#pragma unroll
        for (int f = 0; f < NV; ++f) m[f] = -CUDART_INF_F;
        // this thread's column j's running max (compile-time indexes only)
        auto mcol = [&](int j) -> float { return upper ? m[CW + j] : m[j]; };
        const uint32_t ob = k & 1;
        const uint32_t to = tl + G::TM_O + G::O_COLS * ob;   // this unit's O^T columns
        for (int s = 0; s < nss; ++s) {
            const uint32_t ms = n + (uint32_t)s, slot = ms % G::NVE, sb = ms & 1, pbi = ms % NPB;
            // S of this superstage, the stage's V copies (they carry the
            // flags, and V rows may be zeroed below) and the P buffer's
            // previous PV
            bool ok = true;
            if (lane == 0)
                ok = wait_or_abort(bar(bars, B_SFULL + (int)sb), (ms >> 1) & 1, abort_flag) &&
                     wait_or_abort(bar(bars, B_VFULL + (int)slot), (ms / G::NVE) & 1, abort_flag) &&
                     (ms < NPB || wait_or_abort(bar(bars, B_PVDONE + (int)pbi),
                                                ((ms - NPB) / NPB) & 1, abort_flag));
            if (!settle(__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0)) break;
            tc_fence_after();
            uint32_t sr[2 * NC];
            tmem_ld_cols(tl + G::TM_S + 2 * NC * sb, sr);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars, B_SFREE + (int)sb));
            // this thread's row: page pg of the superstage, key of that page,
            // and (HP > 1) which of the unit's kv heads it belongs to
            const int pg = kss / G::PAGE_ROWS;
            const int rr = kss % G::PAGE_ROWS;
            const int khi = G::HP > 1 ? rr / (8 * G::HP) : 0;
            const int key = G::HP > 1 ? 8 * khi + (kss & 7) : (kss & 15);
            const int hrow = G::HP > 1 ? (rr >> 3) % G::HP : 0;
            const int npg = min(G::SSP, x.np - G::SSP * s);
            const bool present = pg < npg && !((flags[slot] >> pg) & 1u);
            const int32_t kj = (x.p0 + G::SSP * s + pg) * kPageSize + key;
            // this thread's columns: hi and lo parts of their scores
            float shi[CW], slo[CW];
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                if constexpr (SPLIT) {
                    const uint32_t a = __shfl_sync(0xffffffffu, sr[CW + j], lane & 15);
                    const uint32_t b = __shfl_sync(0xffffffffu, sr[NC + CW + j], lane & 15);
                    shi[j] = __uint_as_float(upper ? a : sr[j]);
                    slo[j] = __uint_as_float(upper ? b : sr[NC + j]);
                } else {
                    shi[j] = __uint_as_float(sr[j]);
                    slo[j] = __uint_as_float(sr[NC + j]);
                }
            }
            float sc[CW];
            bool grow = false;
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                const bool valid =
                    present && (G::HP == 1 || j / GQ == hrow) && kj >= clo[j] && kj < chi[j];
                sc[j] = valid ? (shi[j] + slo[j]) * kf[j] : -CUDART_INF_F;
                grow |= sc[j] > mcol(j) + MAX_SLACK;
            }
            // lanes holding one column's scores of a warp: 16 (SPLIT) or 32
            constexpr int XOR0 = SPLIT ? 8 : 16;
            const bool col_writer = (lane & (2 * XOR0 - 1)) == 0;
            if (named_barrier_or(1, 128, grow)) {
                float alpha[NV];
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    float mx = sc[j];
#pragma unroll
                    for (int off = XOR0; off > 0; off >>= 1)
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    if (col_writer) red[w * NC + cb + j] = mx;
                }
                named_barrier(1, 128);
#pragma unroll
                for (int f = 0; f < NV; ++f) {
                    const float M =
                        fmaxf(m[f], fmaxf(fmaxf(red[f], red[NC + f]),
                                          fmaxf(red[2 * NC + f], red[3 * NC + f])));
                    alpha[f] = (m[f] == -CUDART_INF_F) ? 0.f : exp2f(m[f] - M);
                    m[f] = M;
                }
#pragma unroll
                for (int j = 0; j < CW; ++j) l[j] *= upper ? alpha[CW + j] : alpha[j];
                named_barrier(1, 128);          // maxima read before anyone rewrites them
                if (s > 0) {                    // O holds this unit's earlier superstages
                    const uint32_t mp = ms - 1;
                    if (!wait_all(B_PVDONE + (int)(mp % NPB), (mp / NPB) & 1)) break;
                    tc_fence_after();
                    // (HP > 1: every head's accumulator; a head's columns of the
                    // other heads hold nothing used)
#pragma unroll
                    for (int h = 0; h < G::HP; ++h)
#pragma unroll
                    for (int c = 0; c < G::NCH; ++c) {
                        uint32_t o[2 * NC];
                        tmem_ld_cols(to + G::O_HEAD * h + 2 * NC * c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int f = 0; f < NV; ++f) {
                            o[f] = __float_as_uint(__uint_as_float(o[f]) * alpha[f]);
                            o[NC + f] = __float_as_uint(__uint_as_float(o[NC + f]) * alpha[f]);
                        }
                        tmem_st_cols(to + G::O_HEAD * h + 2 * NC * c, o);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
            }
            // P = 2^(s - m) x 2^6 as E4M3 hi (row f) and lo (row NC + f)
            uint32_t hb[(CW + 1) / 2], lb[(CW + 1) / 2];   // two columns' bytes each
#pragma unroll
            for (int j = 0; j < CW; j += 2) {
                const float mj0 = mcol(j);
                const float m0 = (mj0 == -CUDART_INF_F) ? 0.f : mj0;
                const float p0 = exp2f(sc[j] - m0);
                l[j] += p0;
                float p1 = 0.f;
                if (j + 1 < CW) {
                    const float mj1 = mcol(j + 1);
                    const float m1 = (mj1 == -CUDART_INF_F) ? 0.f : mj1;
                    p1 = exp2f(sc[j + 1] - m1);
                    l[j + 1] += p1;
                }
                split_e4m3x2(p0 * PSCALE, p1 * PSCALE, hb[j / 2], lb[j / 2]);
            }
            uint8_t* pb = pbuf + pbi * G::PBUF_BYTES;
            // P^T position of this key: its head's keys together, in the
            // order the head's PV product reads them (HP > 1)
            const int kpos =
                G::HP > 1 ? (128 / G::HP) * hrow + 8 * (2 * pg + khi) + (kss & 7) : kss;
            const int kc = kpos >> 4, kb = kpos & 15;
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                const int f = cb + j, sh = 8 * (j & 1);
                pb[f * 128 + (((kc ^ (f & 7)) << 4) | kb)] = (uint8_t)(hb[j / 2] >> sh);
                pb[(NC + f) * 128 + (((kc ^ (f & 7)) << 4) | kb)] = (uint8_t)(lb[j / 2] >> sh);
            }
            // V rows inside the PV's 32-key steps that no query of the row
            // attends (window edges, a flagged page, the page after an odd
            // last one) may hold anything, NaN included: zero them
            const int nks = (npg + 1) / 2;
            if (zero_lane && pg < 2 * nks && !(present && kj >= x.g.lo && kj < x.g.len)) {
#pragma unroll
                for (int c = 0; c < G::NCH; ++c) {
                    uint4* vr = reinterpret_cast<uint4*>(ring + G::OFF_VRING + slot * G::SLOT_BYTES +
                                                         G::row_off(c, kss));
#pragma unroll
                    for (int i = 0; i < 8; ++i) vr[i] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars, B_PFULL + (int)pbi));
        }
        if (stop) break;
        __syncwarp();                           // q buffer qb: scales read, all S consumed
        if (lane == 0) mbar_arrive(bar(bars, B_QFREE + (int)qb));

        // ---- epilogue: column sums, then O^T from TMEM
        {
            constexpr int XOR0 = SPLIT ? 8 : 16;
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                float v = l[j];
#pragma unroll
                for (int off = XOR0; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if ((lane & (2 * XOR0 - 1)) == 0) red[NSW * NC + w * NC + cb + j] = v;
            }
        }
        const uint32_t ml = n + (uint32_t)nss - 1;
        if (!wait_all(B_PVDONE + (int)(ml % NPB), (ml / NPB) & 1)) break;   // also publishes red
        float Lt[NV];
#pragma unroll
        for (int f = 0; f < NV; ++f) {
            const float* r = red + NSW * NC + f;
            Lt[f] = f < x.nvalid ? ((r[0] + r[NC]) + (r[2 * NC] + r[3 * NC])) : 0.f;
        }
        // only an exactly empty sum means "no keys"; NaN in attended K / V
        // reaches the output as in the definition
        float fac[NV];
#pragma unroll
        for (int f = 0; f < NV; ++f)
            fac[f] = (Lt[f] == 0.f) ? 0.f : __fdividef(vsc[f / GQ], Lt[f] * PSCALE);
        const int64_t r0 = (int64_t)x.b * p.Hq + x.h0;          // output row of column 0
        bool bad_store = false;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < G::HP; ++h)         // HP > 1: head h's columns from its accumulator
#pragma unroll
        for (int c = 0; c < G::NCH; ++c) {
            uint32_t o[2 * NC];
            tmem_ld_cols(to + G::O_HEAD * h + 2 * NC * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int f = 0; f < NV; ++f) {
                if (f >= x.nvalid || f / GQ != h) continue;
                const float v = (Lt[f] == 0.f)
                                    ? 0.f
                                    : (__uint_as_float(o[f]) + __uint_as_float(o[NC + f])) * fac[f];
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bars, B_OFREE + (int)ob));
        if (bad_store) report(p.err_word, kErrSelfCheck);
        if (!single && tid < x.nvalid && GA_CHK(x.rc < p.rc_capacity)) {
            float mm = -CUDART_INF_F, LL = 0.f;      // natural-log LSE of column tid
#pragma unroll
            for (int f = 0; f < NV; ++f)
                if (f == tid) {
                    mm = m[f];
                    LL = Lt[f];
                }
            p.partial_lse[x.rc * p.Hq + x.h0 + tid] =
                (LL == 0.f) ? -CUDART_INF_F : (mm + log2f(LL)) * CUDART_LN2_F;
        }
        n += (uint32_t)nss;
        ++k;
    }
}

// ------------------------------------------------------------------ kernel

// tmK / tmV: the pools' 3-D maps (HP = 1), or their 5-D maps of region 0 and
// tmK1 / tmV1 those of region 1 (HP > 1; unused otherwise).
template <int D, int NV, bool ALIAS, int HP>
__global__ void __launch_bounds__(NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmK1,
                     const __grid_constant__ CUtensorMap tmV1, const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    __shared__ uint32_t tmem_slot;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    using G = Geo<D, ALIAS, HP, (NV > kHeadTile ? 2 * kHeadTile : kHeadTile)>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* pre = reinterpret_cast<int32_t*>(smem + G::OFF_PREFIX);
    volatile uint32_t* flags = reinterpret_cast<volatile uint32_t*>(smem + G::OFF_FLAGS);
    const uint32_t ring = smem_addr(smem + G::OFF_RING);
    const uint32_t bars = smem_addr(smem + G::OFF_BARS);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NKS; ++s) {
            mbar_init(bar(bars, B_KFULL + s), 1);      // producer's arm (+ copied K bytes)
            mbar_init(bar(bars, B_KEMPTY + s), 1);     // QK commit
        }
        for (int s = 0; s < NVMAX; ++s) {
            mbar_init(bar(bars, B_VFULL + s), 1);      // producer's arm (+ copied V bytes)
            mbar_init(bar(bars, B_VEMPTY + s), 1);     // PV commit
        }
        for (int i = 0; i < NPB; ++i) {
            mbar_init(bar(bars, B_PFULL + i), NSW);    // each softmax warp wrote P
            mbar_init(bar(bars, B_PVDONE + i), 1);     // PV commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(bars, B_SFULL + i), 1);      // QK commit
            mbar_init(bar(bars, B_SFREE + i), NSW);    // each softmax warp read S
            mbar_init(bar(bars, B_OFREE + i), NSW);    // each softmax warp read O
            mbar_init(bar(bars, B_QFULL + i), 1);      // the q warp wrote q
            mbar_init(bar(bars, B_QFREE + i), NSW);    // each softmax warp is done with it
        }
        mbar_init(bar(bars, B_FIN), 2);                // both issuers' last commits
        mbar_init(bar(bars, B_TOK), 1);                // the q warp wrote the step's tokens
        mbar_init_fence();
        abort_flag = 0;
    }
    if (warp == PROD_WARP && lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        if (HP > 1) {
            prefetch_tensormap(&tmK1);
            prefetch_tensormap(&tmV1);
        }
    }
    int64_t total_rc = 0;
    if (!build_row_prefix(p, pre, NTHREADS, &total_rc)) return;
    const int64_t U = total_rc * p.Hkv * p.HG;
    if (warp == MMA_WARP) tmem_alloc(smem_addr(&tmem_slot), G::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (warp < NSW) {
        softmax_warps<G, NV>(p, pre, U, smem, bars, tmem, flags, &abort_flag);
    } else if (warp == MMA_WARP || warp == PV_WARP) {
        if (lane == 0) {
            if (warp == MMA_WARP)
                qk_issuer<G>(p, pre, U, ring, smem_addr(smem + G::OFF_Q), bars, tmem, &abort_flag);
            else
                pv_issuer<G>(p, pre, U, ring, smem_addr(smem + G::OFF_P), bars, tmem, &abort_flag);
            // every MMA this thread issued has completed before TMEM is freed
            tc_commit(bar(bars, B_FIN));
            if (!mbar_wait(bar(bars, B_FIN), 0)) {
                report(p.err_word, kErrTimeout);
                abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == PROD_WARP) {
        producer<G>(&tmK, &tmV, &tmK1, &tmV1, p, pre, U, ring, bars, flags, &abort_flag);
    } else if (warp == Q_WARP) {
        q_warp<G, NV>(p, pre, U, smem, bars, &abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, G::TMEM_COLS);
}

}  // namespace tc

// ------------------------------------------------------------------ host

template <int D, bool ALIAS, int HP = 1>
static int run_tc(const DecodeArgs& a) {
    const ga_plan& pl = *a.plan;
    const int32_t S = pl.q_len;
    // (query, head) columns of a kv head: units of 16 when the plan was made
    // for them (more than 8 columns), else of at most 8; HP > 1: the unit's 8
    // columns are the query heads of HP kv heads
    const int32_t cols = a.num_q_heads / a.num_kv_heads * S;
    const bool wide = HP == 1 && pl.col_tile == 2 * kHeadTile;
    const int tw = wide ? 2 * kHeadTile : kHeadTile;
    const int nv = HP > 1 ? 8 : wide ? 16 : cols <= 2 ? 2 : cols <= 4 ? 4 : 8;
    auto pick = [nv]() {
        if constexpr (HP > 1) {
            (void)nv;
            return &tc::decode_tc_kernel<D, 8, ALIAS, HP>;
        } else {
            return nv == 2   ? &tc::decode_tc_kernel<D, 2, ALIAS, 1>
                   : nv == 4 ? &tc::decode_tc_kernel<D, 4, ALIAS, 1>
                   : nv == 8 ? &tc::decode_tc_kernel<D, 8, ALIAS, 1>
                             : &tc::decode_tc_kernel<D, 16, ALIAS, 1>;
        }
    };
    auto kern = pick();
    int smem = tc::Geo<D, ALIAS, HP>::SMEM_BYTES;
    if constexpr (HP == 1)
        if (wide) smem = tc::Geo<D, ALIAS, 1, 2 * kHeadTile>::SMEM_BYTES;
    // attribute slots 8..19: (head dim, alias, column count); 22, 23: HP = 2,
    // 4; 24..27: (head dim, alias) of 16-column units
    int rc = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem,
                              HP > 1 ? (HP == 2 ? 22 : 23)
                              : wide ? 24 + (D == 256 ? 0 : 2) + (ALIAS ? 1 : 0)
                                     : 8 + (D == 256 ? 0 : 6) + (ALIAS ? 3 : 0) +
                                           (nv == 2 ? 0 : nv == 4 ? 1 : 2));
    if (rc != GA_OK) return rc;
    const int64_t rows = a.num_pages * a.num_kv_heads * (int64_t)kPageSize;
    CUtensorMap tmK, tmV, tmK1, tmV1;
    if constexpr (HP > 1) {
        // one box = one 128-dim region of a page's blocks of HP kv heads
        rc = encode_heads_map(&tmK, a.k_pool, 0, a.num_kv_heads, a.num_pages, a.head_dim, HP);
        if (rc == GA_OK)
            rc = encode_heads_map(&tmK1, a.k_pool, 1, a.num_kv_heads, a.num_pages, a.head_dim, HP);
        if (rc == GA_OK)
            rc = encode_heads_map(&tmV, a.v_pool, 0, a.num_kv_heads, a.num_pages, a.head_dim, HP);
        if (rc == GA_OK)
            rc = encode_heads_map(&tmV1, a.v_pool, 1, a.num_kv_heads, a.num_pages, a.head_dim, HP);
        if (rc != GA_OK) return rc;
    } else {
        // one box = a whole page-head block, [key / 8][128-dim region][key % 8]
        const int64_t blocks = a.num_pages * a.num_kv_heads;
        rc = encode_region_map(&tmK, a.k_pool, a.kv_dtype, blocks, a.head_dim, D / 128);
        if (rc != GA_OK) return rc;
        rc = encode_region_map(&tmV, a.v_pool, a.kv_dtype, blocks, a.head_dim, D / 128);
        if (rc != GA_OK) return rc;
        tmK1 = tmK;
        tmV1 = tmV;
    }

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.page_table = a.page_table;
    p.seq_lens = a.seq_lens;
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const bool split = pl.mode != GA_SPLIT_NONE;
    p.partial_o = split ? reinterpret_cast<float*>(ws + pl.partial_o_offset) : nullptr;
    p.partial_lse = split ? reinterpret_cast<float*>(ws + pl.partial_lse_offset) : nullptr;
    p.touch_log = (pl.flags & GA_PLAN_TOUCH_LOG)
                      ? reinterpret_cast<int32_t*>(ws + pl.touch_log_offset)
                      : nullptr;
    p.k_new = static_cast<const uint4*>(a.k_new);
    p.v_new = static_cast<const uint4*>(a.v_new);
    p.k_pool = const_cast<void*>(a.k_pool);
    p.v_pool = const_cast<void*>(a.v_pool);
    p.err_word = a.err_word;
    p.pt_stride = a.pt_stride;
    p.num_pages = a.num_pages;
    p.rc_capacity = pl.row_chunks;
    p.B = a.batch;
    p.Hq = a.num_q_heads * S;
    // units over groups of HP kv heads (columns: their query heads)
    p.Hkv = a.num_kv_heads / HP;
    p.group = a.num_q_heads / a.num_kv_heads * S * HP;
    p.TW = tw;
    p.HG = (p.group + tw - 1) / tw;
    p.window = effective_window(a.window, S);
    p.S = S;
    p.mask_window = a.window;
    p.mode = pl.mode;
    p.splits = pl.splits;
    p.chunk_pages = pl.chunk_pages;
    p.schedule = kernel_schedule(pl.schedule, pl.mode);
    p.touch_stride = pl.touch_stride;
    p.test_wait_timeout = (pl.flags & GA_PLAN_TEST_WAIT_TIMEOUT) ? 1 : 0;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.pool_rows = rows;
    p.out_elems = (int64_t)a.batch * a.num_q_heads * S * a.head_dim;
    const int grid = pl.grid > 0 ? pl.grid : 1;
    kern<<<grid, tc::NTHREADS, smem, a.stream>>>(tmK, tmV, tmK1, tmV1, p);
    if (cudaGetLastError() != cudaSuccess) return GA_ERR_CUDA;
    if (split && !(pl.flags & GA_PLAN_EXTERNAL_COMBINE))
        return launch_combine(p.partial_o, p.partial_lse, a.plan, a.seq_lens, a.out, a.err_word,
                              a.pt_stride, a.stream);
    return GA_OK;
}

int launch_decode_tc(const DecodeArgs& a) {
    // one pool for K and V (same pointer): fetch each block once
    const bool alias = a.k_pool == a.v_pool;
    if (a.head_dim == 256 && !alias) {
        // the plan's unit width (checked against the geometry at the entry)
        const int32_t hp = a.plan->kv_heads_per_unit;
        if (hp == 4) return run_tc<256, false, 4>(a);
        if (hp == 2) return run_tc<256, false, 2>(a);
    }
    if (a.head_dim == 256) return alias ? run_tc<256, true>(a) : run_tc<256, false>(a);
    if (a.head_dim == 512) return alias ? run_tc<512, true>(a) : run_tc<512, false>(a);
    return GA_ERR_UNSUPPORTED;
}

}  // namespace ga
