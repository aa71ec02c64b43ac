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

/* One output row: flat row index r = (b * s_q + i) * h_q + h. */
static int oracle_one_row(const uint16_t *q, const uint16_t *kcache, int64_t num_blocks,
                          int page, const int32_t *block_table, int max_blocks,
                          const int32_t *cache_seqlens, int s_q, int h_q, int h_kv, int d,
                          int dv, double scale, int causal, int64_t r, double *o_row,
                          double *lse_row, double *scores) {
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
        const uint16_t *krow = kcache + ((blk * page + j % page) * h_kv + g) * (int64_t)d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
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
        const uint16_t *krow = kcache + ((blk * page + j % page) * h_kv + g) * (int64_t)d;
        double w = exp(scores[j] - lse);
        for (int v = 0; v < dv; ++v) o_row[v] += w * bf16_bits_to_double(krow[v]);
    }
    return ORACLE_OK;
}

/*
 * Compute the requested rows.
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
    if (!q || !kcache || !block_table || !cache_seqlens || !o || !lse) return ORACLE_ERR_ARG;
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
        if (!scores) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_ERR_NOMEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t n = 0; n < n_rows; ++n) {
            if (!scores) continue;
            int64_t r = rows ? rows[n] : n;
            int st = oracle_one_row(q, kcache, num_blocks, page, block_table, max_blocks,
                                    cache_seqlens, s_q, h_q, h_kv, d, dv, scale, causal, r,
                                    o + n * (int64_t)dv, lse + n, scores);
            if (st != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                status = st;
            }
        }
        free(scores);
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
