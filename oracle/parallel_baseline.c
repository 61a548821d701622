/*
 * A multi-core CPU program doing the MoeReRoutingV2 moves -- BENCHMARK INFRASTRUCTURE ONLY.
 *
 * This is not the oracle: mrr_oracle.c is the definition (nested loops, one thread) that the GPU
 * path is checked against.  This file is a plain parallel program for the same moves, timed by the
 * benchmark's CPU comparison line to show what the host's cores reach.  Only bench.py loads it.
 *
 * What it computes follows the article "CANN ops-transformer MoeReRoutingV2" (m.nlpx.cn/news/59074),
 * section 计算公式: segment (i, j) of counts[i][j] rows moves from its row-major exclusive prefix
 * offset to its column-major exclusive prefix offset, with the scale rows and top-k weights, and the
 * gather (idx_type 0) or scatter (1) index; expert_token_num[j] is the column sum (count mode).
 *
 * Parallel layout: the offsets are two serial prefix walks over N*E counts; the moves are split
 * into blocks of at most 256 rows inside each segment (a block is contiguous at both ends, so it
 * is one memcpy), handed to OpenMP threads dynamically, so one huge segment still spreads over
 * every core.  Counts are assumed valid (the benchmark feeds the same checked inputs as the GPU).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <omp.h>

#define BLOCK_ROWS 256

int mrr_cpu_parallel_run(const uint8_t *tokens, int64_t A, int64_t rb, const void *counts,
                         int count_is_i64, int64_t N, int64_t E, const uint8_t *scales, int64_t sb,
                         const float *topk, uint8_t *out_tokens, uint8_t *out_scales, int32_t *idx,
                         void *etn, float *out_topk, int64_t idx_type, int threads)
{
    const int64_t NE = N * E;
    int64_t *cnt = malloc(sizeof(int64_t) * (size_t)(NE > 0 ? NE : 1));
    int64_t *src = malloc(sizeof(int64_t) * (size_t)(NE > 0 ? NE : 1));
    int64_t *dst = malloc(sizeof(int64_t) * (size_t)(NE > 0 ? NE : 1));
    if (!cnt || !src || !dst) {
        free(cnt);
        free(src);
        free(dst);
        return 1;
    }
    int64_t units = 0;
    for (int64_t q = 0; q < NE; ++q) {
        cnt[q] = count_is_i64 ? ((const int64_t *)counts)[q] : ((const int32_t *)counts)[q];
        units += (cnt[q] + BLOCK_ROWS - 1) / BLOCK_ROWS;
    }
    int64_t run = 0;
    for (int64_t q = 0; q < NE; ++q) {  /* rank outer, expert inner */
        src[q] = run;
        run += cnt[q];
    }
    run = 0;
    for (int64_t j = 0; j < E; ++j) {  /* expert outer, rank inner */
        int64_t col = 0;
        for (int64_t i = 0; i < N; ++i) {
            dst[i * E + j] = run;
            run += cnt[i * E + j];
            col += cnt[i * E + j];
        }
        if (count_is_i64)
            ((int64_t *)etn)[j] = col;
        else
            ((int32_t *)etn)[j] = (int32_t)col;
    }
    /* work units: (segment, first row) */
    int64_t *uq = malloc(sizeof(int64_t) * (size_t)(units > 0 ? units : 1));
    int64_t *uk = malloc(sizeof(int64_t) * (size_t)(units > 0 ? units : 1));
    if (!uq || !uk) {
        free(cnt);
        free(src);
        free(dst);
        free(uq);
        free(uk);
        return 1;
    }
    int64_t u = 0;
    for (int64_t q = 0; q < NE; ++q)
        for (int64_t k = 0; k < cnt[q]; k += BLOCK_ROWS) {
            uq[u] = q;
            uk[u] = k;
            ++u;
        }
#pragma omp parallel for schedule(dynamic, 4) num_threads(threads)
    for (int64_t w = 0; w < units; ++w) {
        const int64_t q = uq[w], k0 = uk[w];
        const int64_t n = cnt[q] - k0 < BLOCK_ROWS ? cnt[q] - k0 : BLOCK_ROWS;
        const int64_t s = src[q] + k0, d = dst[q] + k0;
        memcpy(out_tokens + d * rb, tokens + s * rb, (size_t)(n * rb));
        if (scales && out_scales)
            memcpy(out_scales + d * sb, scales + s * sb, (size_t)(n * sb));
        if (topk && out_topk)
            memcpy(out_topk + d, topk + s, (size_t)n * sizeof(float));
        for (int64_t r = 0; r < n; ++r) {
            if (idx_type == 0)
                idx[d + r] = (int32_t)(s + r);
            else
                idx[s + r] = (int32_t)(d + r);
        }
    }
    free(cnt);
    free(src);
    free(dst);
    free(uq);
    free(uk);
    (void)A;
    return 0;
}
