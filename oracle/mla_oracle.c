/*
 * fp64 CPU oracle for MLA decoding over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the package smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (plain definition, no blocking, no fusion, no reordering):
 *
 *   For batch b, query token i in [0, s_q), query head h in [0, h_q):
 *     g   = h / (h_q / h_kv)                          shared latent KV head
 *     T   = cache_seqlens[b]                          (causal == 0)
 *     T   = cache_seqlens[b] - s_q + i + 1            (causal != 0)
 *     k_j = kcache[block_table[b][j / page]][j % page][g][0 .. d)   j < T
 *     s_j = scale * sum_{c < d} q[b][i][h][c] * k_j[c]
 *     LSE = M + ln( sum_j exp(s_j - M) ),  M = max_j s_j
 *     O[v] = sum_j exp(s_j - LSE) * k_j[v]                           v < dv
 *   A row with T <= 0 has no visible key: O = 0 and LSE = -inf.
 *
 * Sources:
 *  - "Novita AI, H100 및 H200에서 FlashMLA 평가", section "MLA란 무엇인가요?",
 *    table "MHA vs MQA vs GQA vs MLA": every query head shares one compressed
 *    (latent) key-value vector per token, with a decoupled RoPE part.  Hence
 *    one cached row of d = 512 latent + 64 RoPE dims serves as K, and V is its
 *    first dv = 512 dims (the reading this library adopts).
 *  - "FlashMLA란 무엇인가?" (topnet.top article 5338), section "FlashMLA의 주요
 *    특성": bf16 data and a paged KV cache with block size 64.
 *  - same page, section "FlashMLA 설치 및 사용", steps 2 and 3: the decode call
 *    takes q, the cache, block_table, cache_seqlens, dv, the scheduler output
 *    and a causal flag, and returns the output and the log-sum-exp.  The LSE is
 *    read as the natural log of sum_j exp(s_j) with the softmax scale inside.
 *  - causal rule for several query tokens per step ("병렬 디코딩", section
 *    "FlashMLA의 기술 구현"): query i sees keys at positions < T - s_q + i + 1.
 *
 * Inputs arrive as raw bf16 bit patterns (uint16) and are widened to double
 * exactly; all arithmetic is fp64.
 *
 * The cache may instead be packed e4m3 pages with per-token scales
 * (oracle_mla_decode_fp8).  The page "[flashinfer] FlashInfer, SM120 GPU를
 * 위한 희소 MLA 커널 추가로 LLM 추론 속도 향상" (item 5) names a packed KV cache
 * whose scale format is a parameter, and "[vllm] Blackwell을 위한 새로운 MLA
 * 백엔드: TOKENSPEED_MLA 분석" (section "들어가며") an FP8 KV cache; neither gives
 * a layout.  The reading taken: a page is 64 rows of d e4m3 codes followed by
 * 64 little-endian fp32 scales, and row j is k_j[c] = scale_j * e4m3(code_jc),
 * formed exactly in fp64; the attention above is then applied to these rows
 * unchanged.  e4m3 is the OCP 8-bit float E4M3: sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent 0 encodes subnormals m/8 * 2^-6; S.1111.111
 * is NaN; there are no infinities (largest finite value 448).
 *
 * Sparse top-k decode (oracle_mla_decode_sparse).  "[flashinfer] FlashInfer,
 * SM120 GPU를 위한 희소 MLA 커널 추가로 LLM 추론 속도 향상" (section "왜 이게
 * 좋은가?", item 2) describes sparse MLA as attention over only some tokens of
 * the KV cache, chosen by top-k selection, for paged caches with d_qk = 576
 * and 512; it gives no interface.  The reading taken: query token i of
 * sequence b carries a list indices[b][i][0 .. topk) of token positions in
 * the sequence, shared by all of its heads; entries outside [0, T_b) (T_b =
 * cache_seqlens[b]; -1 pads short lists) are ignored, every other entry is one
 * term of the softmax (a position listed twice counts twice), and no causal
 * mask applies on top of the list:
 *     s_t = scale * <q, k_{indices[t]}>,  LSE = ln sum_t exp(s_t),
 *     O = sum_t exp(s_t - LSE) * v_{indices[t]}       over the valid entries t.
 * A row with no valid entry has O = 0 and LSE = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_BLOCK (-2)
#define ORACLE_ERR_NOMEM (-3)

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One OCP e4m3 code as a double (definition in the header comment). */
double oracle_e4m3_to_double(uint8_t code) {
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);        /* m/8 * 2^(1-7) */
    else v = ldexp((double)(8 + m), e - 10);     /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Where cached rows come from: bf16 rows, or packed e4m3 pages. */
typedef struct {
    const uint16_t *bf16;   /* [num_blocks][page][h_kv][d] bf16 bits, or NULL */
    const uint8_t *e4m3;    /* [num_blocks][page * d + page * 4] packed pages (h_kv = 1), or NULL */
} cache_view;

/* Cached row `t` of page `blk`, KV head g, as d doubles (exact). */
static void load_row(const cache_view *cv, int64_t blk, int page, int64_t t, int h_kv, int64_t g, int d,
                     double *row) {
    if (cv->bf16) {
        const uint16_t *krow = cv->bf16 + ((blk * page + t) * h_kv + g) * (int64_t)d;
        for (int c = 0; c < d; ++c) row[c] = bf16_bits_to_double(krow[c]);
    } else {
        const uint8_t *pg = cv->e4m3 + blk * ((int64_t)page * d + (int64_t)page * 4);
        float sc;
        memcpy(&sc, pg + (int64_t)page * d + 4 * t, sizeof sc);
        for (int c = 0; c < d; ++c) row[c] = (double)sc * oracle_e4m3_to_double(pg[t * d + c]);
    }
}

/* One output row: flat row index r = (b * s_q + i) * h_q + h. */
static int oracle_one_row(const uint16_t *q, const cache_view *cv, int64_t num_blocks,
                          int page, const int32_t *block_table, int max_blocks,
                          const int32_t *cache_seqlens, int s_q, int h_q, int h_kv, int d,
                          int dv, double scale, int causal, int64_t r, double *o_row,
                          double *lse_row, double *scores, double *krow) {
    int64_t h = r % h_q;
    int64_t i = (r / h_q) % s_q;
    int64_t b = r / ((int64_t)h_q * s_q);
    int64_t g = h / (h_q / h_kv);
    int64_t T = cache_seqlens[b];
    if (causal) T = T - s_q + i + 1;

    for (int v = 0; v < dv; ++v) o_row[v] = 0.0;
    if (T <= 0) {
        *lse_row = -INFINITY;
        return ORACLE_OK;
    }
    const uint16_t *qrow = q + r * (int64_t)d;

    /* scores s_j = scale * <q, k_j>, gathered page by page through block_table */
    for (int64_t j = 0; j < T; ++j) {
        int64_t blk = block_table[b * max_blocks + j / page];
        if (blk < 0 || blk >= num_blocks) return ORACLE_ERR_BLOCK;
        load_row(cv, blk, page, j % page, h_kv, g, d, krow);
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += bf16_bits_to_double(qrow[c]) * krow[c];
        scores[j] = scale * acc;
    }

    /* log-sum-exp with the maximum shifted out */
    double M = scores[0];
    for (int64_t j = 1; j < T; ++j)
        if (scores[j] > M) M = scores[j];
    double sum = 0.0;
    for (int64_t j = 0; j < T; ++j) sum += exp(scores[j] - M);
    double lse = M + log(sum);
    *lse_row = lse;

    /* O = sum_j softmax_j * V_j, V_j = first dv dims of the cached row */
    for (int64_t j = 0; j < T; ++j) {
        int64_t blk = block_table[b * max_blocks + j / page];
        load_row(cv, blk, page, j % page, h_kv, g, d, krow);
        double w = exp(scores[j] - lse);
        for (int v = 0; v < dv; ++v) o_row[v] += w * krow[v];
    }
    return ORACLE_OK;
}

static int decode_rows(const uint16_t *q, const cache_view *cv, int64_t num_blocks, int page,
                       const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                       int batch, int s_q, int h_q, int h_kv, int d, int dv, double scale,
                       int causal, const int64_t *rows, int64_t n_rows, double *o, double *lse,
                       int nthreads) {
    if (!q || !block_table || !cache_seqlens || !o || !lse) return ORACLE_ERR_ARG;
    if (batch < 0 || s_q <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv || d <= 0 || dv <= 0 ||
        dv > d || page <= 0 || max_blocks < 0)
        return ORACLE_ERR_ARG;
    int64_t total_rows = (int64_t)batch * s_q * h_q;
    if (!rows) n_rows = total_rows;
    int64_t max_T = 0;
    for (int b = 0; b < batch; ++b) {
        if (cache_seqlens[b] < 0) return ORACLE_ERR_ARG;
        if ((int64_t)cache_seqlens[b] > (int64_t)max_blocks * page) return ORACLE_ERR_ARG;
        if (cache_seqlens[b] > max_T) max_T = cache_seqlens[b];
    }
    for (int64_t n = 0; rows && n < n_rows; ++n)
        if (rows[n] < 0 || rows[n] >= total_rows) return ORACLE_ERR_ARG;

    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(max_T > 0 ? max_T : 1));
        double *krow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!scores || !krow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_ERR_NOMEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t n = 0; n < n_rows; ++n) {
            if (!scores || !krow) continue;
            int64_t r = rows ? rows[n] : n;
            int st = oracle_one_row(q, cv, num_blocks, page, block_table, max_blocks,
                                    cache_seqlens, s_q, h_q, h_kv, d, dv, scale, causal, r,
                                    o + n * (int64_t)dv, lse + n, scores, krow);
            if (st != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                status = st;
            }
        }
        free(scores);
        free(krow);
    }
    return status;
}

/*
 * Compute the requested rows over a bf16 cache.
 *   q            [batch, s_q, h_q, d]            bf16 bits
 *   kcache       [num_blocks, page, h_kv, d]     bf16 bits
 *   block_table  [batch, max_blocks]             int32 physical page ids
 *   cache_seqlens[batch]                         int32
 *   rows         n_rows flat row ids (b*s_q+i)*h_q+h, or NULL for all rows
 *   o            [n_rows, dv] fp64 out;  lse [n_rows] fp64 out
 *   nthreads     OpenMP threads (<= 0: runtime default)
 * Returns 0, or a negative error (bad argument, page id out of range, no memory).
 */
int oracle_mla_decode(const uint16_t *q, const uint16_t *kcache, int64_t num_blocks, int page,
                      const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                      int batch, int s_q, int h_q, int h_kv, int d, int dv, double scale,
                      int causal, const int64_t *rows, int64_t n_rows, double *o, double *lse,
                      int nthreads) {
    if (!kcache) return ORACLE_ERR_ARG;
    cache_view cv = {kcache, NULL};
    return decode_rows(q, &cv, num_blocks, page, block_table, max_blocks, cache_seqlens, batch, s_q, h_q,
                       h_kv, d, dv, scale, causal, rows, n_rows, o, lse, nthreads);
}

/*
 * The same over packed e4m3 pages: kv_pages [num_blocks][page * d + page * 4]
 * bytes (codes, then fp32 scales), one KV head (h_kv must be 1).
 */
int oracle_mla_decode_fp8(const uint16_t *q, const uint8_t *kv_pages, int64_t num_blocks, int page,
                          const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                          int batch, int s_q, int h_q, int h_kv, int d, int dv, double scale,
                          int causal, const int64_t *rows, int64_t n_rows, double *o, double *lse,
                          int nthreads) {
    if (!kv_pages || h_kv != 1) return ORACLE_ERR_ARG;
    cache_view cv = {NULL, kv_pages};
    return decode_rows(q, &cv, num_blocks, page, block_table, max_blocks, cache_seqlens, batch, s_q, h_q,
                       h_kv, d, dv, scale, causal, rows, n_rows, o, lse, nthreads);
}

/* One output row of the sparse decode (definition in the header comment). */
static int oracle_one_row_sparse(const uint16_t *q, const cache_view *cv, int64_t num_blocks, int page,
                                 const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                                 const int32_t *indices, int topk, int s_q, int h_q, int h_kv, int d, int dv,
                                 double scale, int64_t r, double *o_row, double *lse_row, double *scores,
                                 int64_t *keys, double *krow) {
    int64_t h = r % h_q;
    int64_t i = (r / h_q) % s_q;
    int64_t b = r / ((int64_t)h_q * s_q);
    int64_t g = h / (h_q / h_kv);
    int64_t T = cache_seqlens[b];
    const int32_t *list = indices + (b * s_q + i) * (int64_t)topk;
    const uint16_t *qrow = q + r * (int64_t)d;

    for (int v = 0; v < dv; ++v) o_row[v] = 0.0;
    /* the valid entries, in list order */
    int n = 0;
    for (int t = 0; t < topk; ++t)
        if (list[t] >= 0 && list[t] < T) keys[n++] = list[t];
    if (n == 0) {
        *lse_row = -INFINITY;
        return ORACLE_OK;
    }
    for (int t = 0; t < n; ++t) {
        int64_t j = keys[t];
        int64_t blk = block_table[b * max_blocks + j / page];
        if (blk < 0 || blk >= num_blocks) return ORACLE_ERR_BLOCK;
        load_row(cv, blk, page, j % page, h_kv, g, d, krow);
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += bf16_bits_to_double(qrow[c]) * krow[c];
        scores[t] = scale * acc;
    }
    double M = scores[0];
    for (int t = 1; t < n; ++t)
        if (scores[t] > M) M = scores[t];
    double sum = 0.0;
    for (int t = 0; t < n; ++t) sum += exp(scores[t] - M);
    double lse = M + log(sum);
    *lse_row = lse;
    for (int t = 0; t < n; ++t) {
        int64_t j = keys[t];
        int64_t blk = block_table[b * max_blocks + j / page];
        load_row(cv, blk, page, j % page, h_kv, g, d, krow);
        double w = exp(scores[t] - lse);
        for (int v = 0; v < dv; ++v) o_row[v] += w * krow[v];
    }
    return ORACLE_OK;
}

/*
 * Sparse top-k decode over a bf16 cache: as oracle_mla_decode, plus
 *   indices  [batch, s_q, topk] int32 token positions per query token
 * (no causal flag: the lists decide what each query token sees).
 */
int oracle_mla_decode_sparse(const uint16_t *q, const uint16_t *kcache, int64_t num_blocks, int page,
                             const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                             const int32_t *indices, int topk, int batch, int s_q, int h_q, int h_kv, int d,
                             int dv, double scale, const int64_t *rows, int64_t n_rows, double *o, double *lse,
                             int nthreads) {
    if (!q || !kcache || !block_table || !cache_seqlens || !indices || !o || !lse) return ORACLE_ERR_ARG;
    if (batch < 0 || s_q <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv || d <= 0 || dv <= 0 || dv > d ||
        page <= 0 || max_blocks < 0 || topk < 0)
        return ORACLE_ERR_ARG;
    int64_t total_rows = (int64_t)batch * s_q * h_q;
    if (!rows) n_rows = total_rows;
    for (int b = 0; b < batch; ++b)
        if (cache_seqlens[b] < 0 || (int64_t)cache_seqlens[b] > (int64_t)max_blocks * page) return ORACLE_ERR_ARG;
    for (int64_t n = 0; rows && n < n_rows; ++n)
        if (rows[n] < 0 || rows[n] >= total_rows) return ORACLE_ERR_ARG;
    cache_view cv = {kcache, NULL};
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        size_t nk = (size_t)(topk > 0 ? topk : 1);
        double *scores = (double *)malloc(sizeof(double) * nk);
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * nk);
        double *krow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!scores || !keys || !krow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_ERR_NOMEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t n = 0; n < n_rows; ++n) {
            if (!scores || !keys || !krow) continue;
            int64_t r = rows ? rows[n] : n;
            int st = oracle_one_row_sparse(q, &cv, num_blocks, page, block_table, max_blocks, cache_seqlens,
                                           indices, topk, s_q, h_q, h_kv, d, dv, scale, r, o + n * (int64_t)dv,
                                           lse + n, scores, keys, krow);
            if (st != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                status = st;
            }
        }
        free(scores);
        free(keys);
        free(krow);
    }
    return status;
}

/* Threads the oracle will use by default (for reporting the CPU baseline). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
