// ga_decode.cu -- paged split-KV GQA decode attention for sm_103a.
//
// One templated kernel body serves both KV families (local hd256 window,
// global hd512 full context) and both KV element types (bf16, E4M3), so the
// hd512 path is never a hand-copied twin of the hd256 one ("[Model] Gemma 4
// M2 26B-A4B", Proposed Plan: one home for the paged-KV launch bodies).
//
// Work decomposition.  A unit is (row-chunk, kv head, head group of <= 8
// query heads).  A row's attended pages (only the window's pages for the
// local family: "Gemma 4 31B on vLLM -- operating-point reference", Three
// load-bearing facts, sliding-window tile pruning) are cut into chunks by the
// split plan; each chunk of each kv head is one unit.  The grid is
// persistent: CTA i takes units i, i + grid, ...
//
// Inside a CTA (NCW + 1 warps):
//   * the producer warp reads page ids from the page table, checks them,
//     and issues one 3-D bulk tensor copy (TMA, 128-byte swizzle) per K and per
//     V page-head block into a ring of NS shared-memory stages, each completing
//     on that stage's "full" mbarrier (one instruction per block: small 2-D
//     boxes issued from one thread capped the stream well below HBM speed);
//   * NCW consumer warps take the unit's pages round-robin.  Per 16-key page a
//     warp computes S^T = K Q^T with m16n8k16 tensor-core MMAs (16 keys x 8
//     query heads), applies the window mask, runs the online softmax on
//     fp32 scores (warp shuffles across the 8 lanes sharing a head column),
//     transposes P with movmatrix and accumulates O^T += V^T P^T (V read with
//     ldmatrix.trans).  The stage is then released on its "empty" mbarrier.
//   * at the end of a unit the consumer warps merge their (m, l, O) in shared
//     memory in a fixed order (deterministic) and write either the final bf16
//     output (row in one chunk) or an fp32 partial plus its log-sum-exp.
// The S=1 decode has no causal mask ("visible-cx/Gemma-4-31B-CoreAI",
// "--metal-sdpa is mandatory here"); the window mask only touches the first
// and last page of the attended range.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math_constants.h>

#include <type_traits>

#include "ga_decode_common.cuh"

namespace ga {


template <int D_, int KV_, int NCW_, int NS_, bool ALIAS_ = false, bool COLPAR_ = false>
struct DecodeCfg {
    static constexpr int D = D_;
    static constexpr int KV = KV_;                  // GA_KV_BF16 / GA_KV_E4M3
    static constexpr int NCW = NCW_;                // consumer warps
    static constexpr int NS = NS_;                  // ring stages (one page each)
    // K and V are one pool (K == V, e.g. a shared K/V projection): each page-head
    // block is fetched once and serves both products.
    static constexpr bool ALIAS = ALIAS_;
    // Column-parallel: a unit holds NCW tiles of 8 (query, head) columns and
    // warp w owns tile w over every page of the unit (each page is read once
    // for all of them; no cross-warp merge).  Page-parallel (default): a unit
    // is one tile of 8 columns and the warps share out its pages.
    static constexpr bool COLPAR = COLPAR_;
    static constexpr int TW = COLPAR ? 8 * NCW : kHeadTile;     // columns per unit

    static constexpr int NCT = NCW * 32;            // consumer threads
    static constexpr int NTHREADS = NCT + 32;
    static constexpr int ESZ = KV == GA_KV_BF16 ? 2 : 1;
    static constexpr int TILE_ELEMS = 128 / ESZ;    // elements per 128-byte box row
    static constexpr int NTILES = D * ESZ / 128;    // boxes per page-head block
    static constexpr int TILE_BYTES = kPageSize * 128;
    static constexpr int BLOCK_BYTES = NTILES * TILE_BYTES;
    static constexpr int STAGE_BYTES = (ALIAS ? 1 : 2) * BLOCK_BYTES;   // K block (+ V block)
    static constexpr int KSTEPS = D / 16;
    static constexpr int MTILES = D / 16;
    static constexpr bool Q_IN_REGS = (D <= 256);
    // E4M3 runs its MMAs on E4M3 operands: P is scaled by PSCALE so that with a
    // max slack of 2^MAX_SLACK it stays within E4M3's range (<= 256 < 448).
    static constexpr float MAX_SLACK = KV == GA_KV_BF16 ? 8.0f : 2.0f;
    static constexpr float PSCALE = KV == GA_KV_BF16 ? 1.0f : 64.0f;
    static constexpr int MSTRIDE = D + 4;           // floats per head row of the merge buffer
    // shared-memory map; every region starts on a 128-byte boundary (the
    // mbarriers need 8, the float4 / uint2 accesses 16)
    static constexpr int al(int x) { return (x + 127) / 128 * 128; }
    // The unit's q rows land as one 3-D box like a page-head block: D/64
    // tiles of [8 heads][128 bytes], 128-byte swizzled.  The E4M3 path turns
    // them into fragments in place (same size).
    static constexpr int Q_BYTES = TW * D * 2;
    static constexpr int QTILE_STRIDE = TW * 128;   // bytes per 64-element column tile
    // The merge buffer: one region of [8 heads][MSTRIDE] floats per consumer
    // warp when shared memory allows (each warp writes its own, one barrier),
    // else one region the warps add into in turn.
    static constexpr int REGION_FLOATS = kHeadTile * MSTRIDE;
    static constexpr int BEFORE_MERGE = al(al(NS * STAGE_BYTES) + Q_BYTES);
    static constexpr int AFTER_MERGE = al(2 * NCW * kHeadTile * 4) + al(2 * kHeadTile * 4) +
                                       al((kMaxBatch + 1) * 4) + al(NS * 4) + al((2 * NS + 1) * 8);
    static constexpr int MREG =
        COLPAR ? 0
        : (BEFORE_MERGE + al(NCW * REGION_FLOATS * 4) + AFTER_MERGE + 1024 <= 227 * 1024) ? NCW
                                                                                         : 1;
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_Q = al(OFF_RING + NS * STAGE_BYTES);
    static constexpr int OFF_MERGE = al(OFF_Q + Q_BYTES);
    static constexpr int OFF_ML = al(OFF_MERGE + MREG * REGION_FLOATS * 4);
    static constexpr int OFF_QSC = al(OFF_ML + 2 * NCW * kHeadTile * 4);   // [2][8] q amax / scale
    static constexpr int OFF_PREFIX = al(OFF_QSC + 2 * kHeadTile * 4);
    static constexpr int OFF_FLAGS = al(OFF_PREFIX + (kMaxBatch + 1) * 4);
    static constexpr int OFF_BARS = al(OFF_FLAGS + NS * 4);
    static constexpr int SMEM_USED = al(OFF_BARS + (2 * NS + 1) * 8);   // full, empty, q tile
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    static_assert(D % 128 == 0 && NTILES >= 1, "head_dim (the merge takes m-tiles 8 at a time)");
    static_assert(OFF_BARS % 8 == 0 && OFF_Q % 1024 == 0 && OFF_MERGE % 16 == 0, "alignment");
    static_assert(KV != GA_KV_E4M3 || (KSTEPS * 32 * 8 == Q_BYTES && !COLPAR),
                  "E4M3 fragments reuse the q tile (page-parallel only)");
    static_assert(REGION_FLOATS % 4 == 0 && MSTRIDE % 4 == 0, "float4 access to merge regions");
    static_assert(STAGE_BYTES % 1024 == 0, "swizzle-128B boxes need 1024-byte aligned stages");
    // Every ring slot must always be consumed by the same warp: page n sits in
    // slot n % NS and, within a unit, goes to warp n % NCW (up to the unit's
    // offset).  A warp waiting on round r of a slot has then consumed round r-1
    // of that slot itself, so the parity wait cannot be satisfied by an older
    // phase of the same parity; unit boundaries are ordered by the merge
    // barrier.  With NS % NCW != 0 a fast warp could see a stale completion.
    // (Column-parallel: every warp consumes every slot, so any depth works.)
    static_assert(COLPAR || NS % NCW == 0, "ring stages must be a multiple of consumer warps");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// ------------------------------------------------------------------ producer

template <class C>
__device__ void producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const DecodeParams& p,
                         const int32_t* pre, int64_t U, uint32_t ring, uint32_t bars,
                         volatile uint32_t* flags, volatile int* abort_flag) {
    // Lanes 0 .. kIssueLanes-1 each take one of that many consecutive pages:
    // the per-page chain (wait for a free stage, arm its barrier, issue the two
    // bulk copies) runs for several stages at once.
    constexpr int kIssueLanes = 4;
    static_assert(C::NS >= kIssueLanes && C::NS <= 32, "ring depth");
    const int lane = threadIdx.x & 31;
    // Test hook: nothing is armed or copied for CTA 0, so its consumers' bounded
    // waits run out and report GA_DEVERR_TIMEOUT (no copy is left in flight).
    if (p.test_wait_timeout && blockIdx.x == 0) return;
    const uint64_t policy = l2_evict_first_policy();
    uint32_t seq = 0;                 // pages handed to the ring so far
    bool stop = false;
    // Look-ahead: while a unit's pages are issued, the next unit's length and
    // first page ids are already on their way, so moving to it costs no
    // dependent global loads.
    auto first_ids = [&](const UnitInfo& y, int32_t& a, int32_t& b) {
        const int32_t* t = p.page_table + (int64_t)y.b * p.pt_stride + y.p0;
        a = (lane < y.np) ? __ldg(t + lane) : -1;
        b = (32 + lane < y.np) ? __ldg(t + 32 + lane) : -1;
    };
    int64_t u = blockIdx.x;
    UnitInfo x = {};
    int32_t id_cur = -1, id_nxt = -1;
    TokenAppend<C::D, C::KV, 1> tok;
    if (u < U) {
        x = unit_info(p, pre, u);
        first_ids(x, id_cur, id_nxt);
    }
    while (u < U && !stop) {
        const int64_t un = u + gridDim.x;
        UnitLoc nl = {};
        int32_t nlen = 0;
        if (un < U) {
            nl = locate_unit(p, pre, un);
            nlen = __ldg(p.seq_lens + nl.b);
        }
        UnitInfo nx = x;
        int32_t nid_cur = -1, nid_nxt = -1;
        bool nx_ready = !(un < U);
        auto ready_next = [&]() {
            if (!nx_ready) {
                nx = finish_unit(p, pre, nl, nlen);
                first_ids(nx, nid_cur, nid_nxt);
                nx_ready = true;
            }
        };
        const int32_t* tbl = p.page_table + (int64_t)x.b * p.pt_stride;
        // the unit's q rows (heads h0 .. h0+nvalid-1, contiguous) into L2 ahead
        // of the consumers' bulk copy of them
        if (((int64_t)x.b * p.Hq + x.h0 + x.nvalid) * C::D <= p.out_elems) {
            const char* qrow = reinterpret_cast<const char*>(
                p.q + ((int64_t)x.b * p.Hq + x.h0) * C::D);
            for (int l = lane; l * 128 < x.nvalid * C::D * 2; l += 32) prefetch_l2(qrow + 128 * l);
        }
        const bool log = p.touch_log != nullptr && x.c == 0 && x.hg == 0;
        tok.start(p, x);               // this step's token, written before its page's copy
        // page ids of this unit, 32 at a time (the next batch loads one batch ahead)
        for (int i0 = 0; i0 < x.np && !stop; i0 += 32) {
            const int cnt = min(32, x.np - i0);
            for (int k = 0; k < cnt && !stop; k += kIssueLanes) {
                if (i0 + k + kIssueLanes >= x.np)     // the group with the last page
                    tok.finish(p, __shfl_sync(0xffffffffu, id_cur, (x.np - 1 - i0) & 31));
                const int32_t pid = __shfl_sync(0xffffffffu, id_cur, (k + lane) & 31);
                bool fail = false;
                if (lane < kIssueLanes && k + lane < cnt) {
                    const uint32_t n = seq + (uint32_t)(k + lane);
                    const uint32_t slot = n % C::NS;
                    const uint32_t round = n / C::NS;
                    const uint32_t full = bars + 8 * slot;
                    const uint32_t empty = bars + 8 * (C::NS + slot);
                    if (*abort_flag || !mbar_wait(empty, (round & 1) ^ 1)) {
                        report(p.err_word, kErrTimeout);
                        *abort_flag = 1;
                        fail = true;
                    } else if (page_ok(pid, p.num_pages) &&
                               GA_CHK(page_block_row(pid, x.c, p.Hkv) >= 0 &&
                                      page_block_row(pid, x.c, p.Hkv) + kPageSize <= p.pool_rows)) {
                        flags[slot] = 0;
                        mbar_arrive_expect_tx(full, C::STAGE_BYTES);
                        const int32_t y = page_block_row(pid, x.c, p.Hkv);
                        const uint32_t dst = ring + slot * C::STAGE_BYTES;
                        // one 3-D box per block: the whole page-head block of K, then V
                        tma_load_3d(dst, tmK, full, 0, y, 0, policy);
                        if constexpr (!C::ALIAS)
                            tma_load_3d(dst + C::BLOCK_BYTES, tmV, full, 0, y, 0, policy);
                    } else {
                        flags[slot] = 1;
                        report(p.err_word, page_ok(pid, p.num_pages) ? kErrSelfCheck : kErrPageId);
                        mbar_arrive(full);
                    }
                    if (log && i0 + k + lane < p.touch_stride && GA_CHK(x.rc < p.rc_capacity))
                        p.touch_log[x.rc * p.touch_stride + i0 + k + lane] = pid;
                }
                stop = __any_sync(0xffffffffu, fail);
                ready_next();          // after the first group: its length has arrived
            }
            seq += (uint32_t)cnt;
            id_cur = id_nxt;
            id_nxt = (i0 + 64 + lane < x.np) ? __ldg(tbl + x.p0 + i0 + 64 + lane) : -1;
        }
        ready_next();                  // a unit without pages
        u = un;
        x = nx;
        id_cur = nid_cur;
        id_nxt = nid_nxt;
    }
    // Never leave with a copy in flight into this CTA's shared memory: wait
    // for the last round each stage was armed for (already complete unless
    // the kernel is aborting, and bounded either way).
    if (lane < C::NS && (uint32_t)lane < seq) {
        const uint32_t last = (uint32_t)lane + ((seq - 1 - (uint32_t)lane) / C::NS) * C::NS;
        if (!mbar_wait(bars + 8 * lane, (last / C::NS) & 1)) {
            report(p.err_word, kErrTimeout);
            *abort_flag = 1;
        }
    }
}

// ------------------------------------------------------------------ consumer

// B fragments of Q^T, per lane: n = lane/4 the head column, t = lane%4.
//  bf16 (m16n8k16): b0 = q[n][16ks+2t .. +1], b1 = q[n][16ks+2t+8 .. +9],
//   read with ldmatrix straight from the unit's q tile.
//  E4M3 (m16n8k32, K = the 16 dims of chunk ks twice): q of head n is scaled
//   by 448 / amax_n and split into two E4M3 parts, hi = E4M3(q') and
//   lo = E4M3(q' - hi); b0 = hi[n][16ks+4t .. +3], b1 = lo[n][16ks+4t .. +3],
//   so one MMA against the K codes stacked twice yields K (hi + lo).  The
//   scale amax_n / 448 goes to qsc[8 + n] and multiplies the scores.
//   fill_qfrags_e4m3 writes qf[ks][lane] = {b0, b1} over the q tile itself.
// The q tile holds piece (n, j) = dims 8j .. 8j+7 of head n at tile j/8, row
// n, 16-byte chunk (j%8) ^ n.
template <class C>
__device__ __forceinline__ void fill_qfrags_e4m3(const DecodeParams& p, const UnitInfo& x,
                                                 uint8_t* qtile, float* qsc, int tid) {
    constexpr int D8 = C::D / 8;
    constexpr int PIECES = kHeadTile * D8;
    constexpr int PER = (PIECES + C::NCT - 1) / C::NCT;
    uint4 w[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int e = tid + k * C::NCT;
        const int n = e / D8, j = e % D8;
        w[k] = make_uint4(0u, 0u, 0u, 0u);
        if (e < PIECES && n < x.nvalid)
            w[k] = *reinterpret_cast<const uint4*>(qtile + (j >> 3) * 1024 + n * 128 +
                                                   (((j & 7) ^ n) << 4));
    }
    unsigned* amax = reinterpret_cast<unsigned*>(qsc);
    if (tid < kHeadTile) amax[tid] = 0u;
    named_barrier(1, C::NCT);        // also: the whole tile is read before fragments overwrite it
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int e = tid + k * C::NCT;
        if (e < PIECES && e / D8 < x.nvalid) {
            const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                m = fmaxf(m, fmaxf(fabsf(bf16_lo(ww[i])), fabsf(bf16_hi(ww[i]))));
            atomicMax(amax + e / D8, __float_as_uint(m));   // non-negative floats order as ints
        }
    }
    named_barrier(1, C::NCT);
    if (tid < kHeadTile) {
        const float am = __uint_as_float(amax[tid]);
        if (tid < x.nvalid && !(am < CUDART_INF_F)) report(p.err_word, kErrQRange);
        qsc[kHeadTile + tid] = (am > 0.f) ? am * (1.0f / 448.0f) : 1.0f;
    }
    named_barrier(1, C::NCT);
    // piece (n, j): ks = j/2; dims 0..3 -> lane t = 2 (j%2), dims 4..7 -> t + 1
    uint32_t* qf = reinterpret_cast<uint32_t*>(qtile);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int e = tid + k * C::NCT;
        if (e < PIECES) {
            const int n = e / D8, j = e % D8;
            const float inv = 1.0f / qsc[kHeadTile + n];
            const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
            uint32_t* dst = qf + ((j >> 1) * 32 + n * 4 + 2 * (j & 1)) * 2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float f[4] = {bf16_lo(ww[2 * h]) * inv, bf16_hi(ww[2 * h]) * inv,
                                    bf16_lo(ww[2 * h + 1]) * inv, bf16_hi(ww[2 * h + 1]) * inv};
                const uint32_t h01 = f32x2_to_e4m3x2(f[0], f[1]);
                const uint32_t h23 = f32x2_to_e4m3x2(f[2], f[3]);
                const uint32_t d01 = e4m3x2_to_f16x2(h01), d23 = e4m3x2_to_f16x2(h23);
                const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&d01));
                const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&d23));
                const uint32_t l01 = f32x2_to_e4m3x2(f[0] - g01.x, f[1] - g01.y);
                const uint32_t l23 = f32x2_to_e4m3x2(f[2] - g23.x, f[3] - g23.y);
                dst[2 * h] = h01 | (h23 << 16);
                dst[2 * h + 1] = l01 | (l23 << 16);
            }
        }
    }
    named_barrier(1, C::NCT);
}

template <class C>
__device__ void consumer(const CUtensorMap* tmQ, const DecodeParams& p, const int32_t* pre,
                         int64_t U, uint8_t* smem, uint32_t ring, uint32_t bars,
                         volatile uint32_t* flags, volatile int* abort_flag,
                         volatile int* q_issued) {
    const int tid = threadIdx.x;            // 0 .. NCT-1
    const int w = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, t = lane & 3;
    // ldmatrix row / 16-byte-chunk selectors of this lane
    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8, khi = lane >> 4;
    const int vrow = (lane & 7) + ((lane >> 4) & 1) * 8, vhi = (lane >> 3) & 1;
    const uint32_t koff = krow * 128, kx = krow & 7;
    const uint32_t voff = vrow * 128, vx = vrow & 7;

    uint8_t* qtile = smem + C::OFF_Q;
    const uint32_t qtile_s = smem_addr(qtile);
    const uint32_t qbar = bars + 8 * (2 * C::NS);
    const uint2* qf = reinterpret_cast<const uint2*>(qtile);   // E4M3 fragments, over the tile
    // ldmatrix selectors for the q tile: lanes 8m .. 8m+7 give the rows (heads)
    // of matrix m = (k-step ks + m/2, half m%2); column-parallel warps read
    // their own 8 rows (one 128-byte swizzle atom of each column tile)
    const int qrow = lane & 7, qmat = lane >> 3;
    const uint32_t qrow_base = C::COLPAR ? 8u * (uint32_t)w : 0u;
    auto q_addr = [&](int ks) -> uint32_t {        // fragments of k-steps ks, ks+1 (ks even)
        const int ksi = ks + (qmat >> 1);
        const uint32_t ch = (uint32_t)(((ksi & 3) << 1) + (qmat & 1));
        return qtile_s + (uint32_t)(ksi >> 2) * (uint32_t)C::QTILE_STRIDE +
               (qrow_base + (uint32_t)qrow) * 128u + ((ch ^ (uint32_t)qrow) << 4);
    };
    const uint64_t qpolicy = l2_evict_last_policy();
    float* merge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
    float* mlw = reinterpret_cast<float*>(smem + C::OFF_ML);   // [2][NCW][8]
    float* qsc = reinterpret_cast<float*>(smem + C::OFF_QSC);  // [8] amax bits, [8] q scale

    uint32_t seq_base = 0;
    uint32_t kunit = 0;                       // units done by this CTA: the q tile's phase
    // The next unit's coordinates, length and scales, loaded one unit ahead
    // (before the merge) so that a unit starts without a dependent load.
    UnitLoc nl = {};
    int32_t nlen = 0;
    float nks = 1.0f, nvs = 1.0f;
    auto locate_next = [&](int64_t un) {
        nl = locate_unit(p, pre, un);
        nlen = __ldg(p.seq_lens + nl.b);
        if constexpr (C::KV == GA_KV_E4M3) {
            nks = __ldg(p.k_scale + nl.c);
            nvs = __ldg(p.v_scale + nl.c);
        }
    };
    if (blockIdx.x < U) locate_next(blockIdx.x);
    for (int64_t u = blockIdx.x; u < U; u += gridDim.x, ++kunit) {
        const UnitInfo x = finish_unit(p, pre, nl, nlen);
        const bool single = (x.g.chunks == 1);
        // This lane's two columns (2t, 2t+1) of the unit: query i = column % S
        // sits at position L - S + i and attends keys [clo, chi) (causal in
        // the chunk; the window ends at its own position).  Pages needing a
        // mask reach below the last query's window start or past the first
        // query's position: for S = 1 the first and last page of the range.
        int32_t clo0, chi0, clo1, chi1;
        {
            const int32_t f0 = x.hg * C::TW + (C::COLPAR ? 8 * w : 0) + 2 * t;
            const int32_t pos0 = x.g.len - p.S + f0 % p.S;
            const int32_t pos1 = x.g.len - p.S + (f0 + 1) % p.S;
            chi0 = pos0 + 1;
            chi1 = pos1 + 1;
            clo0 = p.mask_window > 0 ? max(0, pos0 - p.mask_window + 1) : 0;
            clo1 = p.mask_window > 0 ? max(0, pos1 - p.mask_window + 1) : 0;
        }
        const int32_t plo = p.mask_window > 0 ? max(0, x.g.len - p.mask_window) : 0;
        const int32_t phi = x.g.len - p.S + 1;
        float kfac = p.scale_log2, vfac = 1.0f;
        if (C::KV == GA_KV_E4M3) {
            kfac *= nks;
            vfac = nvs;
        }
        // This unit's q tile (copied during the previous unit's merge).  The
        // wait is bounded and taken even when aborting, whenever a copy was
        // issued: none may be left in flight into shared memory.  q_issued is
        // CTA-uniform here (written before a merge barrier).
        if ((kunit == 0 || *q_issued) && !mbar_wait(qbar, kunit & 1)) {
            if (lane == 0) report(p.err_word, kErrTimeout);
            *abort_flag = 1;
        }
        if constexpr (C::KV == GA_KV_E4M3) fill_qfrags_e4m3<C>(p, x, qtile, qsc, tid);
        float kf0 = kfac, kf1 = kfac;                 // per head column (2t, 2t+1)
        if constexpr (C::KV == GA_KV_E4M3) {
            kf0 *= qsc[kHeadTile + 2 * t];
            kf1 *= qsc[kHeadTile + 2 * t + 1];
        }

        // Head columns past the unit's valid ones read other heads' rows of the
        // tile (or its zero fill): their q is zeroed.  wvalid: valid columns
        // of this warp's tile (column-parallel), else of the unit.
        const int wvalid = C::COLPAR ? min(max(x.nvalid - 8 * w, 0), 8) : x.nvalid;
        uint32_t qr[C::Q_IN_REGS ? C::KSTEPS : 1][2];
        if constexpr (C::Q_IN_REGS) {
            if constexpr (C::KV == GA_KV_BF16) {
                const uint32_t keep = (gid < wvalid) ? 0xffffffffu : 0u;
#pragma unroll
                for (int ks = 0; ks < C::KSTEPS; ks += 2) {
                    uint32_t r[4];
                    ldsm_x4(q_addr(ks), r);
                    qr[ks][0] = r[0] & keep;
                    qr[ks][1] = r[1] & keep;
                    qr[ks + 1][0] = r[2] & keep;
                    qr[ks + 1][1] = r[3] & keep;
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < C::KSTEPS; ++ks) {
                    const uint2 v = qf[ks * 32 + lane];
                    qr[ks][0] = v.x;
                    qr[ks][1] = v.y;
                }
            }
        } else if constexpr (C::KV == GA_KV_BF16 && C::COLPAR) {
            if (wvalid < 8) {                  // warp-uniform: zero this warp's rows past the valid ones
                constexpr int QT = C::D / 64;
                const int nz = (8 - wvalid) * QT * 8;
                for (int e = lane; e < nz; e += 32) {
                    const int n = 8 * w + wvalid + e / (QT * 8), tl = (e / 8) % QT, c = e % 8;
                    *reinterpret_cast<uint4*>(qtile + tl * C::QTILE_STRIDE + n * 128 + c * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
        } else if constexpr (C::KV == GA_KV_BF16) {
            if (x.nvalid < kHeadTile) {        // unit-uniform: zero those rows of the tile once
                constexpr int QT = C::D / 64;
                const int nz = (kHeadTile - x.nvalid) * QT * 8;
                for (int e = tid; e < nz; e += C::NCT) {
                    const int n = x.nvalid + e / (QT * 8), tl = (e / 8) % QT, c = e % 8;
                    *reinterpret_cast<uint4*>(qtile + tl * C::QTILE_STRIDE + n * 128 + c * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                named_barrier(1, C::NCT);
            }
        }

        float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
        float o[C::MTILES][4];
#pragma unroll
        for (int mt = 0; mt < C::MTILES; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

        // page-parallel: warp w takes pages w, w + NCW, ...; column-parallel:
        // every warp takes every page
        for (int i = C::COLPAR ? 0 : w; i < x.np; i += C::COLPAR ? 1 : C::NCW) {
            const uint32_t n = seq_base + (uint32_t)i;
            const uint32_t slot = n % C::NS;
            const uint32_t full = bars + 8 * slot;
            bool ready = false;
            if (!*abort_flag) {
                ready = mbar_wait(full, (n / C::NS) & 1);
                if (!ready) {
                    if (lane == 0) report(p.err_word, kErrTimeout);
                    *abort_flag = 1;
                }
            }
            ready = __all_sync(0xffffffffu, ready);
            if (ready && flags[slot] == 0 && (!C::COLPAR || wvalid > 0)) {
                const uint32_t kb = ring + slot * C::STAGE_BYTES;
                const uint32_t vb = C::ALIAS ? kb : kb + C::BLOCK_BYTES;
                // ---- S^T = K Q^T (16 keys x 8 heads), 4 independent chains
                float sa[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r) sa[r][0] = sa[r][1] = sa[r][2] = sa[r][3] = 0.f;
                if constexpr (C::KV == GA_KV_BF16) {
#pragma unroll
                    for (int ks0 = 0; ks0 < C::KSTEPS; ks0 += 2) {
                        uint32_t qb[4];
                        if constexpr (C::Q_IN_REGS) {
                            qb[0] = qr[ks0][0];
                            qb[1] = qr[ks0][1];
                            qb[2] = qr[ks0 + 1][0];
                            qb[3] = qr[ks0 + 1][1];
                        } else {
                            ldsm_x4(q_addr(ks0), qb);
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int ks = ks0 + h;
                            uint32_t a[4];
                            const uint32_t ch = (uint32_t)(((ks & 3) << 1) + khi);
                            ldsm_x4(kb + (ks >> 2) * C::TILE_BYTES + koff + ((ch ^ kx) << 4), a);
                            mma_bf16(sa[ks & 3], a, qb[2 * h], qb[2 * h + 1]);
                        }
                    }
                } else {
                    // K codes feed the E4M3 MMA directly: ldmatrix gives, per
                    // 16-dim chunk, the A fragment rows (keys) x k 0..15; K of the
                    // MMA carries the chunk twice (hi and lo parts of q).
#pragma unroll
                    for (int kp = 0; kp < C::KSTEPS / 2; ++kp) {
                        uint32_t r[4];
                        const uint32_t ch = (uint32_t)(((kp & 3) << 1) + khi);
                        ldsm_x4(kb + (kp >> 2) * C::TILE_BYTES + koff + ((ch ^ kx) << 4), r);
#pragma unroll
                        for (int hs = 0; hs < 2; ++hs) {
                            const int ks = 2 * kp + hs;
                            uint32_t b0, b1;
                            if constexpr (C::Q_IN_REGS) {
                                b0 = qr[ks][0];
                                b1 = qr[ks][1];
                            } else {
                                const uint2 v = qf[ks * 32 + lane];
                                b0 = v.x;
                                b1 = v.y;
                            }
                            mma_e4m3(sa[ks & 3], r[2 * hs], r[2 * hs + 1], r[2 * hs],
                                     r[2 * hs + 1], b0, b1);
                        }
                    }
                }
                float s[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    s[r] = ((sa[0][r] + sa[1][r]) + (sa[2][r] + sa[3][r])) * ((r & 1) ? kf1 : kf0);
                // ---- window / length mask (first and last page of the range only)
                const int32_t key0 = (x.p0 + i) * kPageSize;
                const bool partial = key0 < plo || key0 + kPageSize > phi;
                uint32_t mk01 = 0xffffffffu, mk89 = 0xffffffffu;
                if (partial) {
                    // scores: per (key, column); V rows: keys no query of the row
                    // attends (outside [lo, L) of the union window) hold no data
                    const int32_t ka = key0 + gid, kb8 = key0 + gid + 8;
                    if (!(ka >= clo0 && ka < chi0)) s[0] = -CUDART_INF_F;
                    if (!(ka >= clo1 && ka < chi1)) s[1] = -CUDART_INF_F;
                    if (!(kb8 >= clo0 && kb8 < chi0)) s[2] = -CUDART_INF_F;
                    if (!(kb8 >= clo1 && kb8 < chi1)) s[3] = -CUDART_INF_F;
                    auto valid = [&](int k) {
                        const int32_t kk = key0 + k;
                        return kk >= x.g.lo && kk < x.g.len;
                    };
                    if constexpr (C::KV == GA_KV_BF16) {
                        mk01 = (valid(2 * t) ? 0x0000ffffu : 0u) |
                               (valid(2 * t + 1) ? 0xffff0000u : 0u);
                        mk89 = (valid(2 * t + 8) ? 0x0000ffffu : 0u) |
                               (valid(2 * t + 9) ? 0xffff0000u : 0u);
                    } else {   // E4M3 V fragment bytes hold keys 2t, 2t+1, 2t+8, 2t+9
                        mk01 = (valid(2 * t) ? 0x000000ffu : 0u) |
                               (valid(2 * t + 1) ? 0x0000ff00u : 0u) |
                               (valid(2 * t + 8) ? 0x00ff0000u : 0u) |
                               (valid(2 * t + 9) ? 0xff000000u : 0u);
                    }
                }
                // ---- online softmax (base 2) over this page, per head column.
                // The running max m is only raised when some score exceeds it by
                // more than MAX_SLACK, so p <= 2^MAX_SLACK between updates; the
                // common page needs one warp vote instead of a shuffle reduction
                // and an O rescale.  m stays uniform across the 8 lanes of a
                // column because it only changes on the warp-uniform slow path.
                {
                    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
                    const bool grow = (mx0 > m0 + C::MAX_SLACK) || (mx1 > m1 + C::MAX_SLACK);
                    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                        for (int off = 4; off < 32; off <<= 1) {
                            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                        }
                        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                        const float al0 = (m0 == -CUDART_INF_F) ? 0.f : exp2f(m0 - mn0);
                        const float al1 = (m1 == -CUDART_INF_F) ? 0.f : exp2f(m1 - mn1);
                        m0 = mn0;
                        m1 = mn1;
                        l0 *= al0;
                        l1 *= al1;
#pragma unroll
                        for (int mt = 0; mt < C::MTILES; ++mt) {
                            o[mt][0] *= al0;
                            o[mt][1] *= al1;
                            o[mt][2] *= al0;
                            o[mt][3] *= al1;
                        }
                    }
                }
                const float ms0 = (m0 == -CUDART_INF_F) ? 0.f : m0;
                const float ms1 = (m1 == -CUDART_INF_F) ? 0.f : m1;
                const float p0 = exp2f(s[0] - ms0), p1 = exp2f(s[1] - ms1);
                const float p2 = exp2f(s[2] - ms0), p3 = exp2f(s[3] - ms1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // ---- P^T fragments: rows = keys, cols = heads -> transpose
                uint32_t pb0, pb1;
                if constexpr (C::KV == GA_KV_BF16) {
                    pb0 = movmatrix_t(pack_bf16x2(p0, p1));
                    pb1 = movmatrix_t(pack_bf16x2(p2, p3));
                } else {
                    // (keys 2t, 2t+1) and (keys 2t+8, 2t+9) of head column g in f16,
                    // scaled by PSCALE, split into E4M3 hi + lo parts: b0 / b1 of the
                    // PV MMA, whose K carries these four keys twice.
                    const uint32_t h01 = movmatrix_t(pack_f16x2(p0 * C::PSCALE, p1 * C::PSCALE));
                    const uint32_t h89 = movmatrix_t(pack_f16x2(p2 * C::PSCALE, p3 * C::PSCALE));
                    const uint32_t e01 = f16x2_to_e4m3x2(h01), e89 = f16x2_to_e4m3x2(h89);
                    const uint32_t r01 = e4m3x2_to_f16x2(e01), r89 = e4m3x2_to_f16x2(e89);
                    const __half2 d01 = __hsub2(*reinterpret_cast<const __half2*>(&h01),
                                                *reinterpret_cast<const __half2*>(&r01));
                    const __half2 d89 = __hsub2(*reinterpret_cast<const __half2*>(&h89),
                                                *reinterpret_cast<const __half2*>(&r89));
                    const uint32_t l01 = f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t*>(&d01));
                    const uint32_t l89 = f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t*>(&d89));
                    pb0 = e01 | (e89 << 16);
                    pb1 = l01 | (l89 << 16);
                }
                // ---- O^T += V^T P^T (V rows of unattended slots zeroed on partial pages)
                auto pv = [&](auto masked) {
                    constexpr bool kMask = decltype(masked)::value;
                    if constexpr (C::KV == GA_KV_BF16) {
#pragma unroll
                        for (int mt = 0; mt < C::MTILES; ++mt) {
                            uint32_t a[4];
                            const uint32_t ch = (uint32_t)(((mt & 3) << 1) + vhi);
                            ldsm_x4_t(vb + (mt >> 2) * C::TILE_BYTES + voff + ((ch ^ vx) << 4), a);
                            if constexpr (kMask) {
                                a[0] &= mk01;
                                a[1] &= mk01;
                                a[2] &= mk89;
                                a[3] &= mk89;
                            }
                            mma_bf16(o[mt], a, pb0, pb1);
                        }
                    } else {
                        // V^T fragments from ldmatrix.trans: per 32-dim group the
                        // b16 transpose gives, per lane, keys (2t, 2t+1) x dims
                        // (2g, 2g+1) of two 8-key halves; one byte_perm per register
                        // forms the A rows of the even-dim (E) and odd-dim (O)
                        // m-tiles with K order keys 2t, 2t+1, 2t+8, 2t+9 (twice).
#pragma unroll
                        for (int mp = 0; mp < C::MTILES / 2; ++mp) {
                            uint32_t r[4];
                            const uint32_t ch = (uint32_t)(((mp & 3) << 1) + vhi);
                            ldsm_x4_t(vb + (mp >> 2) * C::TILE_BYTES + voff + ((ch ^ vx) << 4), r);
                            uint32_t e0 = __byte_perm(r[0], r[2], 0x6420u);
                            uint32_t e1 = __byte_perm(r[1], r[3], 0x6420u);
                            uint32_t o0 = __byte_perm(r[0], r[2], 0x7531u);
                            uint32_t o1 = __byte_perm(r[1], r[3], 0x7531u);
                            if constexpr (kMask) {
                                e0 &= mk01; e1 &= mk01; o0 &= mk01; o1 &= mk01;
                            }
                            mma_e4m3(o[2 * mp], e0, e1, e0, e1, pb0, pb1);
                            mma_e4m3(o[2 * mp + 1], o0, o1, o0, o1, pb0, pb1);
                        }
                    }
                };
                if (partial)
                    pv(std::true_type{});
                else
                    pv(std::false_type{});
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (C::NS + slot));
        }
        seq_base += (uint32_t)x.np;
        const int64_t un = u + gridDim.x;
        if (un < U) locate_next(un);
        // generic writes to the q tile (E4M3 fragments, zeroed rows) are ordered
        // before the next bulk copy into it (reads need no proxy fence)
        if (C::KV == GA_KV_E4M3 || (!C::Q_IN_REGS && x.nvalid < C::TW))
            fence_proxy_async_shared();

        // ---- merge the warps' (m, l, O) in a fixed order
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if constexpr (C::COLPAR) {
            // Column-parallel: each warp holds the whole softmax of its own
            // columns; after the q tile is released, it scales and stores them.
            named_barrier(1, C::NCT);
            if (tid == 0) {
                const int issue = (un < U && !*abort_flag) ? 1 : 0;
                *q_issued = issue;
                if (issue) {
                    mbar_arrive_expect_tx(qbar, C::Q_BYTES);
                    tma_load_3d(qtile_s, tmQ, qbar, 0, unit_q_row(p, nl), 0, qpolicy);
                }
            }
            const float fa0 = (l0 == 0.f) ? 0.f : __fdividef(vfac, l0 * C::PSCALE);
            const float fa1 = (l1 == 0.f) ? 0.f : __fdividef(vfac, l1 * C::PSCALE);
            const bool c0 = 2 * t < wvalid, c1 = 2 * t + 1 < wvalid;
            const int64_t h = x.h0 + 8 * w + 2 * t;          // column 2t of this lane
            const int64_t r0 = (int64_t)x.b * p.Hq + h;      // its output row
            const bool ok0 = c0 && GA_CHK((r0 + 1) * C::D <= p.out_elems &&
                                          (single || (x.rc < p.rc_capacity && p.partial_o)));
            const bool ok1 = c1 && GA_CHK((r0 + 2) * C::D <= p.out_elems &&
                                          (single || (x.rc < p.rc_capacity && p.partial_o)));
            if ((c0 && !ok0) || (c1 && !ok1)) report(p.err_word, kErrSelfCheck);
#pragma unroll
            for (int mt = 0; mt < C::MTILES; ++mt) {
                const int d0 = 16 * mt + gid, d1 = d0 + 8;
                if (single) {
                    if (ok0) {
                        p.out[r0 * C::D + d0] = __float2bfloat16_rn(o[mt][0] * fa0);
                        p.out[r0 * C::D + d1] = __float2bfloat16_rn(o[mt][2] * fa0);
                    }
                    if (ok1) {
                        p.out[(r0 + 1) * C::D + d0] = __float2bfloat16_rn(o[mt][1] * fa1);
                        p.out[(r0 + 1) * C::D + d1] = __float2bfloat16_rn(o[mt][3] * fa1);
                    }
                } else {
                    float* po = p.partial_o + (x.rc * p.Hq + h) * (int64_t)C::D;
                    if (ok0) {
                        po[d0] = o[mt][0] * fa0;
                        po[d1] = o[mt][2] * fa0;
                    }
                    if (ok1) {
                        po[C::D + d0] = o[mt][1] * fa1;
                        po[C::D + d1] = o[mt][3] * fa1;
                    }
                }
            }
            if (!single && gid == 0) {        // natural-log LSE of each column
                if (ok0)
                    p.partial_lse[x.rc * p.Hq + h] =
                        (l0 == 0.f) ? -CUDART_INF_F : (m0 + log2f(l0)) * CUDART_LN2_F;
                if (ok1)
                    p.partial_lse[x.rc * p.Hq + h + 1] =
                        (l1 == 0.f) ? -CUDART_INF_F : (m1 + log2f(l1)) * CUDART_LN2_F;
            }
            continue;
        }
        if (gid == 0) {
            mlw[w * kHeadTile + 2 * t] = m0;
            mlw[w * kHeadTile + 2 * t + 1] = m1;
            mlw[C::NCW * kHeadTile + w * kHeadTile + 2 * t] = l0;
            mlw[C::NCW * kHeadTile + w * kHeadTile + 2 * t + 1] = l1;
        }
        named_barrier(1, C::NCT);
        // every warp is past its pages: the next unit's q tile can be fetched
        // while the merge runs
        if (tid == 0) {
            const int issue = (un < U && !*abort_flag) ? 1 : 0;
            *q_issued = issue;
            if (issue) {
                mbar_arrive_expect_tx(qbar, C::Q_BYTES);
                tma_load_3d(qtile_s, tmQ, qbar, 0, unit_q_row(p, nl), 0, qpolicy);
            }
        }
        float fac[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = 2 * t + e;
            float M = -CUDART_INF_F;
            for (int ww = 0; ww < C::NCW; ++ww) M = fmaxf(M, mlw[ww * kHeadTile + col]);
            const float Ms = (M == -CUDART_INF_F) ? 0.f : M;
            float Lt = 0.f;
            for (int ww = 0; ww < C::NCW; ++ww)
                Lt += mlw[C::NCW * kHeadTile + ww * kHeadTile + col] *
                      exp2f(mlw[ww * kHeadTile + col] - Ms);
            const float mown = (e == 0) ? m0 : m1;
            // only an exactly empty sum means "no keys"; NaN in attended K / V
            // propagates to the output as in the definition
            fac[e] = (Lt == 0.f) ? 0.f : exp2f(mown - Ms) * __fdividef(vfac, Lt * C::PSCALE);
        }
        // natural-log LSE of the chunk's scaled scores for head tid (read here:
        // the next unit may overwrite the per-warp (m, l) once past the merge)
        float lse = -CUDART_INF_F;
        if (!single && tid < x.nvalid) {
            float M = -CUDART_INF_F;
            for (int ww = 0; ww < C::NCW; ++ww) M = fmaxf(M, mlw[ww * kHeadTile + tid]);
            const float Ms = (M == -CUDART_INF_F) ? 0.f : M;
            float Lt = 0.f;
            for (int ww = 0; ww < C::NCW; ++ww)
                Lt += mlw[C::NCW * kHeadTile + ww * kHeadTile + tid] *
                      exp2f(mlw[ww * kHeadTile + tid] - Ms);
            lse = (Lt == 0.f) ? -CUDART_INF_F : (Ms + log2f(Lt)) * CUDART_LN2_F;
        }
        // Each warp's scaled O goes to its own region, summed in warp order by
        // the output loop; with one shared region the warps add into it in
        // turn.  Either way the order is fixed: deterministic results.  Every
        // lane writes both its head columns: rows of heads past the unit's
        // valid ones are never read, and straight-line code lets the loads of
        // a batch issue together.
        if (!GA_CHK(2 * t + 1 < kHeadTile)) report(p.err_word, kErrSelfCheck);
        float* r0 = merge + (C::MREG > 1 ? w * C::REGION_FLOATS : 0) + (2 * t) * C::MSTRIDE;
        float* r1 = r0 + C::MSTRIDE;
        auto dims = [](int mt, int& d0, int& d1) {
            if constexpr (C::KV == GA_KV_BF16) {
                d0 = 16 * mt + (threadIdx.x & 31) / 4;
                d1 = d0 + 8;
            } else {   // E4M3 m-tile pairs hold even / odd dims of 32-dim groups
                d0 = 32 * (mt >> 1) + 2 * ((threadIdx.x & 31) / 4) + (mt & 1);
                d1 = d0 + 16;
            }
        };
        if constexpr (C::MREG > 1) {
#pragma unroll
            for (int mt = 0; mt < C::MTILES; ++mt) {
                int d0, d1;
                dims(mt, d0, d1);
                r0[d0] = o[mt][0] * fac[0];
                r1[d0] = o[mt][1] * fac[1];
                r0[d1] = o[mt][2] * fac[0];
                r1[d1] = o[mt][3] * fac[1];
            }
            named_barrier(1, C::NCT);
        } else {
            if (w == 0) {
#pragma unroll
                for (int mt = 0; mt < C::MTILES; ++mt) {
                    int d0, d1;
                    dims(mt, d0, d1);
                    r0[d0] = o[mt][0] * fac[0];
                    r1[d0] = o[mt][1] * fac[1];
                    r0[d1] = o[mt][2] * fac[0];
                    r1[d1] = o[mt][3] * fac[1];
                }
            }
            named_barrier(1, C::NCT);
            for (int ww = 1; ww < C::NCW; ++ww) {
                if (w == ww) {
                    constexpr int MB = 8;
#pragma unroll
                    for (int m0b = 0; m0b < C::MTILES; m0b += MB) {
                        float prev[MB][4];
#pragma unroll
                        for (int i = 0; i < MB; ++i) {
                            int d0, d1;
                            dims(m0b + i, d0, d1);
                            prev[i][0] = r0[d0];
                            prev[i][1] = r1[d0];
                            prev[i][2] = r0[d1];
                            prev[i][3] = r1[d1];
                        }
#pragma unroll
                        for (int i = 0; i < MB; ++i) {
                            int d0, d1;
                            dims(m0b + i, d0, d1);
                            r0[d0] = prev[i][0] + o[m0b + i][0] * fac[0];
                            r1[d0] = prev[i][1] + o[m0b + i][1] * fac[1];
                            r0[d1] = prev[i][2] + o[m0b + i][2] * fac[0];
                            r1[d1] = prev[i][3] + o[m0b + i][3] * fac[1];
                        }
                    }
                }
                named_barrier(1, C::NCT);
            }
        }
        constexpr int D8 = C::D / 8;
        for (int e = tid; e < x.nvalid * D8; e += C::NCT) {
            const int n = e / D8, d = (e % D8) * 8;
            const float4* src = reinterpret_cast<const float4*>(merge + n * C::MSTRIDE + d);
            float4 a = src[0], b = src[1];
#pragma unroll
            for (int r = 1; r < C::MREG; ++r) {
                const float4* sr = src + r * (C::REGION_FLOATS / 4);
                const float4 ar = sr[0], br = sr[1];
                a.x += ar.x; a.y += ar.y; a.z += ar.z; a.w += ar.w;
                b.x += br.x; b.y += br.y; b.z += br.z; b.w += br.w;
            }
            const int h = x.h0 + n;
            if (!GA_CHK(((int64_t)x.b * p.Hq + h) * C::D + d + 8 <= p.out_elems &&
                        (single || (x.rc < p.rc_capacity && p.partial_o != nullptr)))) {
                report(p.err_word, kErrSelfCheck);
                continue;
            }
            if (single) {
                uint4 v;
                v.x = pack_bf16x2(a.x, a.y);
                v.y = pack_bf16x2(a.z, a.w);
                v.z = pack_bf16x2(b.x, b.y);
                v.w = pack_bf16x2(b.z, b.w);
                *reinterpret_cast<uint4*>(p.out + ((int64_t)x.b * p.Hq + h) * C::D + d) = v;
            } else {
                float4* dst = reinterpret_cast<float4*>(
                    p.partial_o + (x.rc * p.Hq + h) * (int64_t)C::D + d);
                dst[0] = a;
                dst[1] = b;
            }
        }
        if (!single && tid < x.nvalid && GA_CHK(x.rc < p.rc_capacity))
            p.partial_lse[x.rc * p.Hq + x.h0 + tid] = lse;
    }
}

// ------------------------------------------------------------------ kernel

template <class C>
__global__ void __launch_bounds__(C::NTHREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    __shared__ int q_issued;          // the q tile of the next unit was requested
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* pre = reinterpret_cast<int32_t*>(smem + C::OFF_PREFIX);
    volatile uint32_t* flags = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_FLAGS);
    const uint32_t ring = smem_addr(smem + C::OFF_RING);
    const uint32_t bars = smem_addr(smem + C::OFF_BARS);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bars + 8 * s, 1);
            mbar_init(bars + 8 * (C::NS + s), C::COLPAR ? C::NCW : 1);   // consumers of a stage
        }
        mbar_init(bars + 8 * (2 * C::NS), 1);      // q tile
        mbar_init_fence();
        abort_flag = 0;
    }
    if (warp == C::NCW && lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmQ);
    }
    int64_t total_rc = 0;
    if (!build_row_prefix(p, pre, C::NTHREADS, &total_rc)) return;
    const int64_t U = total_rc * p.Hkv * p.HG;
    // the first unit's q tile; later ones are fetched during each merge
    if (threadIdx.x == 0 && (int64_t)blockIdx.x < U) {
        mbar_arrive_expect_tx(bars + 8 * (2 * C::NS), C::Q_BYTES);
        tma_load_3d(smem_addr(smem + C::OFF_Q), &tmQ, bars + 8 * (2 * C::NS), 0,
                    unit_q_row(p, locate_unit(p, pre, blockIdx.x)), 0, l2_evict_last_policy());
    }
    if (warp == C::NCW)
        producer<C>(&tmK, &tmV, p, pre, U, ring, bars, flags, &abort_flag);
    else
        consumer<C>(&tmQ, p, pre, U, smem, ring, bars, flags, &abort_flag, &q_issued);
}

// ------------------------------------------------------------------ host

template <class C>
static int run(const DecodeArgs& a, int slot) {
    const void* fn = reinterpret_cast<const void*>(&decode_kernel<C>);
    int rc = ensure_smem_attr(fn, C::SMEM_BYTES, slot);
    if (rc != GA_OK) return rc;
    const ga_plan& pl = *a.plan;
    const int32_t S = pl.q_len;
    const int64_t rows = a.num_pages * a.num_kv_heads * (int64_t)kPageSize;
    CUtensorMap tmK, tmV, tmQ;
    rc = encode_rows_map(&tmK, a.k_pool, a.kv_dtype, rows, a.head_dim, kPageSize);
    if (rc != GA_OK) return rc;
    rc = encode_rows_map(&tmV, a.v_pool, a.kv_dtype, rows, a.head_dim, kPageSize);
    if (rc != GA_OK) return rc;
    // q as [B * Hq * S, D] bf16, boxes of one group of 8 (query, head)
    // columns (rows past the end read as zeros)
    rc = encode_rows_map(&tmQ, a.q, GA_KV_BF16, (int64_t)a.batch * a.num_q_heads * S, a.head_dim,
                         C::TW);
    if (rc != GA_OK) return rc;

    DecodeParams p;
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
    p.Hkv = a.num_kv_heads;
    p.group = a.num_q_heads / a.num_kv_heads * S;
    p.TW = C::TW;
    p.HG = (p.group + C::TW - 1) / C::TW;
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
    p.pool_rows = a.num_pages * a.num_kv_heads * (int64_t)kPageSize;
    p.out_elems = (int64_t)a.batch * a.num_q_heads * S * a.head_dim;
    const int grid = pl.grid > 0 ? pl.grid : 1;
    decode_kernel<C><<<grid, C::NTHREADS, C::SMEM_BYTES, a.stream>>>(tmK, tmV, tmQ, p);
    if (cudaGetLastError() != cudaSuccess) return GA_ERR_CUDA;
    if (split && !(pl.flags & GA_PLAN_EXTERNAL_COMBINE))
        return launch_combine(p.partial_o, p.partial_lse, a.plan, a.seq_lens, a.out, a.err_word,
                              a.pt_stride, a.stream);
    return GA_OK;
}

// Tuned shapes per (head_dim, KV type): consumer warps, ring stages (a
// multiple of the warps).  The macros let a build sweep them.
#ifndef GA_LB_NCW
#define GA_LB_NCW 3
#define GA_LB_NS 9
#endif
#ifndef GA_LE_NCW
#define GA_LE_NCW 7
#define GA_LE_NS 14
#endif
#ifndef GA_GB_NCW
#define GA_GB_NCW 4
#define GA_GB_NS 4
#endif
#ifndef GA_GE_NCW
#define GA_GE_NCW 6
#define GA_GE_NS 12
#endif
using CfgLocalBf16 = DecodeCfg<256, GA_KV_BF16, GA_LB_NCW, GA_LB_NS>;
using CfgLocalE4m3 = DecodeCfg<256, GA_KV_E4M3, GA_LE_NCW, GA_LE_NS>;
using CfgGlobalBf16 = DecodeCfg<512, GA_KV_BF16, GA_GB_NCW, GA_GB_NS>;
using CfgGlobalE4m3 = DecodeCfg<512, GA_KV_E4M3, GA_GE_NCW, GA_GE_NS>;
// K == V (one pool): half-size stages; four per-warp merge regions fit.
#ifndef GA_GA_NCW
#define GA_GA_NCW 4
#define GA_GA_NS 8
#endif
using CfgGlobalBf16Alias = DecodeCfg<512, GA_KV_BF16, GA_GA_NCW, GA_GA_NS, true>;
// Column-parallel (4 tiles of 8 columns per unit, every warp on every page).
#ifndef GA_CL_NS
#define GA_CL_NS 12
#endif
#ifndef GA_CG_NS
#define GA_CG_NS 5
#endif
using CfgLocalBf16Col = DecodeCfg<256, GA_KV_BF16, 4, GA_CL_NS, false, true>;
using CfgGlobalBf16Col = DecodeCfg<512, GA_KV_BF16, 4, GA_CG_NS, false, true>;
using CfgGlobalE4m3Alias = DecodeCfg<512, GA_KV_E4M3, GA_GE_NCW, 2 * GA_GE_NS, true>;

int launch_decode(const DecodeArgs& a) {
    // the rows-by-size schedule: one-query plans, unsplit or in fixed-size
    // chunks, whose sorted arrays and counters fit after the row prefix
    if (a.plan->schedule != kScheduleRoundRobin &&
        (a.plan->schedule != kScheduleSorted || a.plan->q_len != 1 ||
         !(a.plan->mode == kSplitNone    ? sorted_schedule_fits(a.batch)
           : a.plan->mode == kSplitChunk ? sorted_chunk_schedule_fits(a.batch)
                                         : false)))
        return GA_ERR_INVALID_ARG;
    // many (query, head) columns per kv head (multi-query decode) and a plan
    // made for 64-column units: the tensor-core kernel
#ifndef GA_MQ_MMA_SYNC
    if (a.plan->col_tile == kTcColTile && a.kv_dtype == GA_KV_BF16 && a.k_pool != a.v_pool)
        return launch_mq_tc(a);
#endif
    // more than one tile of (query, head) columns per kv head and a plan made
    // for wider units: column-parallel mma.sync units of 4 x 8 columns
    const bool colpar = a.plan->col_tile > kHeadTile && a.kv_dtype == GA_KV_BF16 &&
                        a.k_pool != a.v_pool;
    if (colpar)
        return a.head_dim == 256 ? run<CfgLocalBf16Col>(a, 6) : run<CfgGlobalBf16Col>(a, 7);
    if (a.head_dim == 256) {
#ifndef GA_E4M3_LOCAL_MMA_SYNC
        if (a.kv_dtype == GA_KV_E4M3) return launch_decode_tc(a);
#endif
        return a.kv_dtype == GA_KV_BF16 ? run<CfgLocalBf16>(a, 0) : run<CfgLocalE4m3>(a, 1);
    }
    if (a.head_dim == 512 && a.k_pool == a.v_pool) {
#ifndef GA_E4M3_GLOBAL_MMA_SYNC
        if (a.kv_dtype == GA_KV_E4M3) return launch_decode_tc(a);
#endif
        return a.kv_dtype == GA_KV_BF16 ? run<CfgGlobalBf16Alias>(a, 4)
                                        : run<CfgGlobalE4m3Alias>(a, 5);
    }
    if (a.head_dim == 512) {
#ifndef GA_E4M3_GLOBAL_MMA_SYNC
        if (a.kv_dtype == GA_KV_E4M3) return launch_decode_tc(a);
#endif
        return a.kv_dtype == GA_KV_BF16 ? run<CfgGlobalBf16>(a, 2) : run<CfgGlobalE4m3>(a, 3);
    }
    return GA_ERR_UNSUPPORTED;
}

}  // namespace ga
