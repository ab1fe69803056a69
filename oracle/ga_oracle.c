/*
 * ga_oracle.c -- plain CPU fp64 oracle for paged split-KV GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table or constant with the CUDA path under
 * paged_split_kv_gqa_gb300/ and never includes anything from it.
 *
 * What it computes (plain definitions, written out, no blocking or fusion):
 *
 *   decode  -- for every row b and query head h:
 *              kv head c = floor(h / g), g = Hq / Hkv  (block-GQA mapping;
 *              "visible-cx/Gemma-4-31B-CoreAI", hybrid-pf64 numerics gate,
 *              32 query heads over 4 global KV heads);
 *              key set J = [lo, L_b), lo = max(0, L_b - W) for the local
 *              sliding-window family, lo = 0 for the global family
 *              ("[Model] Gemma 4 M3 31B", Acceptance Criteria: window
 *              boundaries 1023 / 1024 / 1025);
 *              key j lives in physical page page_table[b][j / P], slot j % P
 *              ("[Model] Gemma 4 M1 12B", Description: paged decode over two
 *              KV groups with their own head counts and cache shapes);
 *              s_j = scale * <q, k_j>;  o = sum_j e^{s_j - m} v_j / sum_j e^{s_j - m},
 *              m = max_j s_j;  lse = m + ln sum_j e^{s_j - m}.
 *              Everything in double.  bf16 -> double is exact; an fp8 code
 *              decodes exactly and is multiplied by its per-head fp32 scale in
 *              double (exact: 4-bit x 24-bit significands).
 *   split   -- the same key set cut into page-aligned chunks; each chunk gives
 *              (o_s, lse_s); they are merged by o = sum_s e^{lse_s - M} o_s /
 *              sum_s e^{lse_s - M}, M = max_s lse_s, empty chunks (lse = -inf)
 *              weigh nothing ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa
 *              is mandatory here": flash-decode with split factor 8).
 *   multi-query decode -- S query tokens per row, the last S positions of the
 *              row: query i (0 <= i < S) sits at position p_i = L_b - S + i
 *              and attends exactly the keys a one-query decode of a row of
 *              length p_i + 1 would: causal inside the chunk, and for the
 *              sliding family the window ends at its own position
 *              ("visible-cx/Gemma-4-31B-CoreAI", hybrid-pf64/ bundles: the prefill entry has
 *              a query axis with an intra-chunk causal mask, and the chunk
 *              parity gate -- chunked and token-by-token walks must agree;
 *              "Gemma 4 31B on vLLM", LIGHT recipe: EAGLE3 verify of 3
 *              speculative tokens).  A query with p_i < 0 attends nothing.
 *   append  -- writes token position pos_b into page page_table[b][pos_b / P],
 *              slot pos_b % P, for every kv head; the fp8 pool stores
 *              E4M3FN(RNE, saturate-to-finite)(fp32(x) / scale[c])
 *              ("[Model] Gemma 4 M2 26B-A4B", Proposed Plan: opt-in FP8 KV pool
 *              for the sliding family).
 *   e4m3    -- OCP 8-bit floating point, E4M3 "FN" variant: bias 7, no
 *              infinities, S.1111.111 is NaN, largest finite 448, subnormals
 *              m * 2^-9.  Encoder rounds to nearest, ties to even, and
 *              saturates finite overflow and +-inf to +-448; NaN -> 0x7F.
 *
 * Layouts (all row-major, C order):
 *   q           [B, Hq, D]            bf16 bit patterns (uint16)
 *   pools       [num_pages, Hkv, P, D] bf16 bit patterns or e4m3 codes (uint8)
 *   page_table  [B, pt_stride]         int32
 *   seq_lens    [B]                    int32 (keys attended end at L_b - 1)
 *   out         [nrows, Hq, D]         double
 *   multi-query: q [B, Hq, S, D], out [B, Hq, S, D], lse [B, Hq, S]
 *
 * Return value: 0 on success, a negative number for an argument the
 * definition cannot evaluate (bad page id, length beyond the table, ...).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_KV_BF16 0
#define ORACLE_KV_E4M3 1

/* Threads of one call: nthreads > 0 as asked, else the process default.
 * Passed per parallel region, so one call never changes the next one's. */
static int oracle_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* ---------------------------------------------------------------- numbers */

double oracle_bf16_to_double(uint16_t bits) {
    /* bf16 is the top half of an IEEE binary32: widen and reinterpret. */
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

double oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round-to-nearest-even of a non-negative double to an integer. */
static double rne(double a) {
    double f = floor(a);
    double r = a - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;          /* saturate (incl. +-inf) */
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid m * 2^-9, m = 0..8; m = 8 is the smallest normal,
           whose code 0b0001000 is exactly 8. */
        double m = rne(a / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int e2;
    double frac = frexp(a, &e2);                 /* a = frac * 2^e2, frac in [0.5,1) */
    int e = e2 - 1;                              /* a = (2*frac) * 2^e, 2*frac in [1,2) */
    double mant = rne((2.0 * frac - 1.0) * 8.0); /* 3 fraction bits */
    if (mant >= 8.0) { mant = 0.0; e += 1; }
    int field = e + 7;
    if (field > 15 || (field == 15 && mant >= 7.0)) return sign | 0x7E;
    return sign | (uint8_t)((field << 3) | (int)mant);
}

/* ---------------------------------------------------------------- key sets */

/* Keys attended by the query of a row of length L: [*lo, *hi).
   W <= 0 means the global family (whole context). */
void oracle_key_range(int32_t L, int32_t W, int32_t* lo, int32_t* hi) {
    int32_t l = 0;
    if (L < 0) L = 0;
    if (W > 0 && L > W) l = L - W;
    *lo = l;
    *hi = L;
}

/* Logical pages holding those keys: first logical page and count. */
void oracle_logical_pages(int32_t L, int32_t W, int32_t P, int32_t* first, int32_t* count) {
    int32_t lo, hi;
    oracle_key_range(L, W, &lo, &hi);
    if (hi <= lo) { *first = 0; *count = 0; return; }
    *first = lo / P;
    *count = (hi - 1) / P - lo / P + 1;
}

/* ---------------------------------------------------------------- gather */

typedef struct {
    const void* k_pool;
    const void* v_pool;
    int kv_dtype;
    const float* k_scale;
    const float* v_scale;
    const int32_t* page_table;
    int64_t pt_stride;
    int32_t Hkv, D, P;
    int64_t num_pages;
} pool_view;

/* Element d of key/value slot (page, c, slot) as a double, scale applied. */
static double pool_elem(const pool_view* pv, const void* pool, const float* sc,
                        int64_t page, int32_t c, int32_t slot, int32_t d) {
    int64_t idx = (((page * pv->Hkv) + c) * (int64_t)pv->P + slot) * (int64_t)pv->D + d;
    if (pv->kv_dtype == ORACLE_KV_BF16)
        return oracle_bf16_to_double(((const uint16_t*)pool)[idx]);
    return oracle_e4m3_decode(((const uint8_t*)pool)[idx]) * (double)sc[c];
}

/* Gather keys [lo, hi) of row b, kv head c into dense K, V [n, D]. */
static int gather(const pool_view* pv, int32_t b, int32_t c, int32_t lo, int32_t hi,
                  double* K, double* V) {
    for (int32_t j = lo; j < hi; ++j) {
        int64_t lp = j / pv->P;
        if (lp >= pv->pt_stride) return -2;
        int64_t page = pv->page_table[(int64_t)b * pv->pt_stride + lp];
        if (page < 0 || page >= pv->num_pages) return -3;
        int32_t slot = j % pv->P;
        for (int32_t d = 0; d < pv->D; ++d) {
            K[(int64_t)(j - lo) * pv->D + d] = pool_elem(pv, pv->k_pool, pv->k_scale, page, c, slot, d);
            V[(int64_t)(j - lo) * pv->D + d] = pool_elem(pv, pv->v_pool, pv->v_scale, page, c, slot, d);
        }
    }
    return 0;
}

/* Softmax attention of one query over n dense keys.  o[D]; returns lse. */
static double attend(const double* q, const double* K, const double* V, int64_t n,
                     int32_t D, double scale, double* s, double* o) {
    if (n <= 0) {
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        return -INFINITY;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int32_t d = 0; d < D; ++d) acc += q[d] * K[j * D + d];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double w = exp(s[j] - m);
        l += w;
        for (int32_t d = 0; d < D; ++d) o[d] += w * V[j * D + d];
    }
    for (int32_t d = 0; d < D; ++d) o[d] /= l;
    return m + log(l);
}

/* ---------------------------------------------------------------- decode */

/*
 * Full decode.  rows: optional list of nrows row indices (NULL = all B rows,
 * nrows ignored).  out [nrows, Hq, D], lse_out [nrows, Hq] (may be NULL).
 * chunk_pages > 0 computes every row as page-aligned chunks of that many
 * pages and merges them by log-sum-exp (split mode); 0 = one pass.
 * nthreads <= 0 uses the OpenMP default.
 */
int oracle_decode(const uint16_t* q, const void* k_pool, const void* v_pool, int kv_dtype,
                  const float* k_scale, const float* v_scale,
                  const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                  int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t W, int32_t P,
                  int64_t num_pages, double scale, const int32_t* rows, int32_t nrows,
                  int32_t chunk_pages, double* out, double* lse_out, int32_t nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0) return -1;
    if (kv_dtype != ORACLE_KV_BF16 && kv_dtype != ORACLE_KV_E4M3) return -1;
    pool_view pv = {k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride,
                    Hkv, D, P, num_pages};
    const int32_t g = Hq / Hkv;
    const int32_t nr = rows ? nrows : B;
    int status = 0;
    const int nt = oracle_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t unit = 0; unit < (int64_t)nr * Hkv; ++unit) {
        int32_t r = (int32_t)(unit / Hkv);
        int32_t c = (int32_t)(unit % Hkv);
        int32_t b = rows ? rows[r] : r;
        if (b < 0 || b >= B) {
#pragma omp atomic write
            status = -4;
            continue;
        }
        int32_t lo, hi;
        oracle_key_range(seq_lens[b], W, &lo, &hi);
        int64_t n = hi - lo;
        double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
        double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double* qd = (double*)malloc(sizeof(double) * D);
        int rc = gather(&pv, b, c, lo, hi, K, V);
        if (rc) {
#pragma omp atomic write
            status = rc;
        }
        for (int32_t i = 0; i < g && rc == 0; ++i) {
            int32_t h = c * g + i;
            for (int32_t d = 0; d < D; ++d)
                qd[d] = oracle_bf16_to_double(q[((int64_t)b * Hq + h) * D + d]);
            double* o = out + ((int64_t)r * Hq + h) * D;
            double lse;
            if (chunk_pages <= 0) {
                lse = attend(qd, K, V, n, D, scale, s, o);
            } else {
                /* chunks: logical pages [first + j*cp, first + (j+1)*cp) */
                int32_t first = n > 0 ? lo / P : 0;
                int32_t npages = n > 0 ? (hi - 1) / P - first + 1 : 0;
                int32_t nch = (npages + chunk_pages - 1) / chunk_pages;
                double M = -INFINITY;
                double* lses = (double*)malloc(sizeof(double) * (size_t)(nch > 0 ? nch : 1));
                double* os = (double*)malloc(sizeof(double) * (size_t)(nch > 0 ? nch : 1) * D);
                for (int32_t j = 0; j < nch; ++j) {
                    int64_t k0 = (int64_t)(first + j * chunk_pages) * P;
                    int64_t k1 = (int64_t)(first + (j + 1) * chunk_pages) * P;
                    if (k0 < lo) k0 = lo;
                    if (k1 > hi) k1 = hi;
                    lses[j] = attend(qd, K + (k0 - lo) * D, V + (k0 - lo) * D,
                                     k1 - k0, D, scale, s, os + (int64_t)j * D);
                    if (lses[j] > M) M = lses[j];
                }
                double den = 0.0;
                for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int32_t j = 0; j < nch; ++j) {
                    if (lses[j] == -INFINITY) continue;
                    double w = exp(lses[j] - M);
                    den += w;
                    for (int32_t d = 0; d < D; ++d) o[d] += w * os[(int64_t)j * D + d];
                }
                if (den > 0.0) {
                    for (int32_t d = 0; d < D; ++d) o[d] /= den;
                    lse = M + log(den);
                } else {
                    lse = -INFINITY;
                }
                free(lses);
                free(os);
            }
            if (lse_out) lse_out[(int64_t)r * Hq + h] = lse;
        }
        free(K); free(V); free(s); free(qd);
    }
    return status;
}

/*
 * Multi-query decode: S query tokens per row at positions L_b - S .. L_b - 1.
 * q [B, Hq, S, D] bf16; out [B, Hq, S, D]; lse_out [B, Hq, S] (may be NULL).
 * Query i of row b is the one-query decode of a row of length L_b - S + i + 1
 * over the same pages.
 */
int oracle_decode_mq(const uint16_t* q, const void* k_pool, const void* v_pool, int kv_dtype,
                     const float* k_scale, const float* v_scale,
                     const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                     int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t W, int32_t P,
                     int64_t num_pages, int32_t S, double scale, double* out,
                     double* lse_out, int32_t nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0 || S <= 0) return -1;
    if (kv_dtype != ORACLE_KV_BF16 && kv_dtype != ORACLE_KV_E4M3) return -1;
    pool_view pv = {k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, pt_stride,
                    Hkv, D, P, num_pages};
    const int32_t g = Hq / Hkv;
    int status = 0;
    const int nt = oracle_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t unit = 0; unit < (int64_t)B * Hkv; ++unit) {
        int32_t b = (int32_t)(unit / Hkv);
        int32_t c = (int32_t)(unit % Hkv);
        int32_t L = seq_lens[b];
        /* keys any of the S queries attends: from the first query's window
           start to the last query's position */
        int32_t lo0, hi0, loS, hiS;
        oracle_key_range(L - S + 1, W, &lo0, &hi0);
        oracle_key_range(L, W, &loS, &hiS);
        int32_t glo = lo0, ghi = hiS;
        int64_t n = ghi > glo ? ghi - glo : 0;
        double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
        double* sbuf = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double* qd = (double*)malloc(sizeof(double) * D);
        int rc = n > 0 ? gather(&pv, b, c, glo, ghi, K, V) : 0;
        if (rc) {
#pragma omp atomic write
            status = rc;
        }
        for (int32_t hj = 0; hj < g && rc == 0; ++hj) {
            int32_t h = c * g + hj;
            for (int32_t i = 0; i < S; ++i) {
                int64_t row = ((int64_t)b * Hq + h) * S + i;
                for (int32_t d = 0; d < D; ++d)
                    qd[d] = oracle_bf16_to_double(q[row * D + d]);
                /* query i: the keys of a one-query row of length L - S + i + 1 */
                int32_t lo, hi;
                oracle_key_range(L - S + i + 1, W, &lo, &hi);
                double lse;
                if (hi <= lo) {
                    for (int32_t d = 0; d < D; ++d) out[row * D + d] = 0.0;
                    lse = -INFINITY;
                } else {
                    lse = attend(qd, K + (int64_t)(lo - glo) * D, V + (int64_t)(lo - glo) * D,
                                 hi - lo, D, scale, sbuf, out + row * D);
                }
                if (lse_out) lse_out[row] = lse;
            }
        }
        free(K); free(V); free(sbuf); free(qd);
    }
    return status;
}

/* Log-sum-exp merge of S partials: po [S, D], plse [S] (natural log) -> o [D]. */
double oracle_combine(const double* po, const double* plse, int32_t S, int32_t D, double* o) {
    double M = -INFINITY;
    for (int32_t s = 0; s < S; ++s)
        if (plse[s] > M) M = plse[s];
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (M == -INFINITY) return -INFINITY;
    double den = 0.0;
    for (int32_t s = 0; s < S; ++s) {
        if (plse[s] == -INFINITY) continue;
        double w = exp(plse[s] - M);
        den += w;
        for (int32_t d = 0; d < D; ++d) o[d] += w * po[(int64_t)s * D + d];
    }
    for (int32_t d = 0; d < D; ++d) o[d] /= den;
    return M + log(den);
}

/* ---------------------------------------------------------------- append */

/*
 * Writes the new token of every row b with positions[b] >= 0 into the pools.
 * k_new, v_new [B, Hkv, D] bf16 bits; pools as above (bf16 bits or e4m3).
 * Returns -2 / -3 when a position or page id is outside the table / pool
 * (that row is skipped).
 */
int oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new, void* k_pool, void* v_pool,
                     int kv_dtype, const float* k_scale, const float* v_scale,
                     const int32_t* page_table, int64_t pt_stride, const int32_t* positions,
                     int32_t B, int32_t Hkv, int32_t D, int32_t P, int64_t num_pages) {
    int status = 0;
    for (int32_t b = 0; b < B; ++b) {
        int32_t pos = positions[b];
        if (pos < 0) continue;
        int64_t lp = pos / P;
        if (lp >= pt_stride) { status = -2; continue; }
        int64_t page = page_table[(int64_t)b * pt_stride + lp];
        if (page < 0 || page >= num_pages) { status = -3; continue; }
        int32_t slot = pos % P;
        for (int32_t c = 0; c < Hkv; ++c) {
            int64_t dst = ((page * Hkv + c) * (int64_t)P + slot) * (int64_t)D;
            int64_t src = ((int64_t)b * Hkv + c) * D;
            for (int32_t d = 0; d < D; ++d) {
                if (kv_dtype == ORACLE_KV_BF16) {
                    ((uint16_t*)k_pool)[dst + d] = k_new[src + d];
                    ((uint16_t*)v_pool)[dst + d] = v_new[src + d];
                } else {
                    float xk = (float)oracle_bf16_to_double(k_new[src + d]);
                    float xv = (float)oracle_bf16_to_double(v_new[src + d]);
                    float qk = xk / k_scale[c];   /* IEEE binary32 division */
                    float qv = xv / v_scale[c];
                    ((uint8_t*)k_pool)[dst + d] = oracle_e4m3_encode(qk);
                    ((uint8_t*)v_pool)[dst + d] = oracle_e4m3_encode(qv);
                }
            }
        }
    }
    return status;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
