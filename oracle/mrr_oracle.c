/*
 * CPU oracle for the MoeReRoutingV2 re-routing step.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * The CUDA library never links, includes or calls anything here, and this file uses
 * nothing from the CUDA library.
 *
 * It is the plain definition of the op, written as the nested loops the pages state:
 *
 *   "CANN ops-transformer MoeReRoutingV2" article (m.nlpx.cn/news/59074):
 *     - section 计算公式 (formulas): SrcOffset is a double sum over the count matrix with
 *       the rank index outermost; DstOffset is the same double sum with the expert index
 *       outermost.  permute_tokens[DstOffset+k] = tokens[SrcOffset+k], and the same move
 *       for per_token_scales and expert_topk_weight, for 0 <= k < the segment's count.
 *     - section 参数说明 / 参数取值细节 (parameters): counts[i,j] = tokens this rank got
 *       from rank i for expert j; permute_token_idx is int32, idx_type 0 = gather index,
 *       1 = scatter index; expert_token_num is [E] in the counts' integer type and, in
 *       count mode (expert_token_num_type = 1), holds the tokens per expert.
 *     - section 约束说明 (constraints): Sum(counts) = A; every count > 0.
 *
 * The formulas lost their comparison signs in extraction.  Reading adopted: the offsets
 * are linearised exclusive prefixes -- SrcOffset(i,j) is the sum of every count that
 * precedes (i,j) in a row-major walk (rank outer, expert inner), DstOffset(i,j) the sum of
 * every count that precedes (i,j) in a column-major walk (expert outer, rank inner).  Only
 * that reading makes the moves a permutation of the A rows.
 *
 * Payloads are treated as opaque bytes: nothing is computed on them, so every output is
 * defined bit for bit.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* return codes */
#define ORC_OK 0
#define ORC_ERR_ARG 1          /* a required pointer or size is invalid            */
#define ORC_ERR_COUNT_NONPOS 2 /* some counts[i,j] <= 0 (section 参数说明: must be > 0) */
#define ORC_ERR_COUNT_SUM 3    /* Sum(counts) != A (section 约束说明)                */

static int64_t count_at(const void *counts, int count_is_i64, int64_t E, int64_t i, int64_t j)
{
    if (count_is_i64)
        return ((const int64_t *)counts)[i * E + j];
    return (int64_t)((const int32_t *)counts)[i * E + j];
}

/*
 * Validation (section 约束说明 and 参数说明): every count > 0 and the counts sum to A, which
 * must fit the int32 index output (section 算子 IR 原型: permute_token_idx is INT32).
 */
int mrr_oracle_validate(const void *counts, int count_is_i64, int64_t N, int64_t E, int64_t A)
{
    int64_t sum = 0;
    if (A < 0 || A > INT32_MAX || N < 0 || E < 0)
        return ORC_ERR_ARG;
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < E; ++j) {
            int64_t c = count_at(counts, count_is_i64, E, i, j);
            if (c <= 0)
                return ORC_ERR_COUNT_NONPOS;
            if (c > A)
                return ORC_ERR_COUNT_SUM;
            sum += c;
            if (sum > A)
                return ORC_ERR_COUNT_SUM;
        }
    return sum == A ? ORC_OK : ORC_ERR_COUNT_SUM;
}

/*
 * SrcOffset and DstOffset for every segment (i,j), section 计算公式.
 * src_off[i*E+j]: rank-outer walk; dst_off[i*E+j]: expert-outer walk.
 */
void mrr_oracle_offsets(const void *counts, int count_is_i64, int64_t N, int64_t E,
                        int64_t *src_off, int64_t *dst_off)
{
    int64_t run = 0;
    for (int64_t i = 0; i < N; ++i)         /* cur_rank outer   */
        for (int64_t j = 0; j < E; ++j) {   /* cur_expert inner */
            src_off[i * E + j] = run;
            run += count_at(counts, count_is_i64, E, i, j);
        }
    run = 0;
    for (int64_t j = 0; j < E; ++j)         /* cur_expert outer */
        for (int64_t i = 0; i < N; ++i) {   /* cur_rank inner   */
            dst_off[i * E + j] = run;
            run += count_at(counts, count_is_i64, E, i, j);
        }
}

/*
 * The whole op.  Row payloads are byte rows: row_bytes per token row (H elements times the
 * token width), scale_row_bytes per scale row (0 when per_token_scales is absent).
 * topk_w / permute_topk_w are [A] float32 (the [A,1] tensors), NULL when absent.
 * expert_token_num is written in the counts' type, count mode.
 * On any error nothing is written.
 */
int mrr_oracle_run(const uint8_t *tokens, int64_t A, int64_t row_bytes,
                   const void *counts, int count_is_i64, int64_t N, int64_t E,
                   const uint8_t *scales, int64_t scale_row_bytes,
                   const float *topk_w,
                   uint8_t *permute_tokens, uint8_t *permute_scales,
                   int32_t *permute_token_idx, void *expert_token_num,
                   float *permute_topk_w, int64_t idx_type)
{
    int rc;
    int64_t *src_off, *dst_off;

    if (!counts && N * E > 0)
        return ORC_ERR_ARG;
    if (row_bytes <= 0 || (A > 0 && (!tokens || !permute_tokens || !permute_token_idx)))
        return ORC_ERR_ARG;
    if (E > 0 && !expert_token_num)
        return ORC_ERR_ARG;
    if (idx_type != 0 && idx_type != 1)
        return ORC_ERR_ARG;
    if ((topk_w == NULL) != (permute_topk_w == NULL))
        return ORC_ERR_ARG;
    if (scales && (!permute_scales || scale_row_bytes <= 0))
        return ORC_ERR_ARG;
    rc = mrr_oracle_validate(counts, count_is_i64, N, E, A);
    if (rc != ORC_OK)
        return rc;

    src_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N * E + 1));
    dst_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N * E + 1));
    if (!src_off || !dst_off) {
        free(src_off);
        free(dst_off);
        return ORC_ERR_ARG;
    }
    mrr_oracle_offsets(counts, count_is_i64, N, E, src_off, dst_off);

    /* the three move equations share one (SrcOffset, DstOffset) pair per segment */
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < E; ++j) {
            int64_t n = count_at(counts, count_is_i64, E, i, j);
            for (int64_t k = 0; k < n; ++k) {
                int64_t s = src_off[i * E + j] + k;
                int64_t d = dst_off[i * E + j] + k;
                memcpy(permute_tokens + d * row_bytes, tokens + s * row_bytes, (size_t)row_bytes);
                if (scales)
                    memcpy(permute_scales + d * scale_row_bytes, scales + s * scale_row_bytes,
                           (size_t)scale_row_bytes);
                if (topk_w)
                    permute_topk_w[d] = topk_w[s];
                if (idx_type == 0)
                    permute_token_idx[d] = (int32_t)s;   /* gather: out[d] = in[idx[d]]  */
                else
                    permute_token_idx[s] = (int32_t)d;   /* scatter: out[idx[s]] = in[s] */
            }
        }

    /* expert_token_num, count mode: tokens handled by each expert = column sums */
    for (int64_t j = 0; j < E; ++j) {
        int64_t total = 0;
        for (int64_t i = 0; i < N; ++i)
            total += count_at(counts, count_is_i64, E, i, j);
        if (count_is_i64)
            ((int64_t *)expert_token_num)[j] = total;
        else
            ((int32_t *)expert_token_num)[j] = (int32_t)total;
    }

    free(src_off);
    free(dst_off);
    return ORC_OK;
}

/*
 * The inverse move, for the combine side of the MoE layer: rows that sit expert-major (as the
 * forward op left them) go back to the rank-major order they arrived in, so they can be
 * returned to their source ranks.  The pages place the op just before the expert FFN and name
 * finalize/combine ops after it ("CANN ops-transformer MoeReRoutingV2" article, section
 * 数据流定位); the inverse reuses the same segments: for every (i,j) and 0 <= k < counts[i,j],
 *   tokens[SrcOffset(i,j) + k] = permute_tokens[DstOffset(i,j) + k]
 * and the same for the scale rows and top-k weights.  Same validation as mrr_oracle_run; on
 * any error nothing is written.
 */
int mrr_oracle_unroute(const uint8_t *permute_tokens, int64_t A, int64_t row_bytes,
                       const void *counts, int count_is_i64, int64_t N, int64_t E,
                       const uint8_t *permute_scales, int64_t scale_row_bytes,
                       const float *permute_topk_w,
                       uint8_t *tokens, uint8_t *scales, float *topk_w)
{
    int rc;
    int64_t *src_off, *dst_off;

    if (!counts && N * E > 0)
        return ORC_ERR_ARG;
    if (row_bytes <= 0 || (A > 0 && (!permute_tokens || !tokens)))
        return ORC_ERR_ARG;
    if ((permute_topk_w == NULL) != (topk_w == NULL))
        return ORC_ERR_ARG;
    if (permute_scales && (!scales || scale_row_bytes <= 0))
        return ORC_ERR_ARG;
    rc = mrr_oracle_validate(counts, count_is_i64, N, E, A);
    if (rc != ORC_OK)
        return rc;

    src_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N * E + 1));
    dst_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N * E + 1));
    if (!src_off || !dst_off) {
        free(src_off);
        free(dst_off);
        return ORC_ERR_ARG;
    }
    mrr_oracle_offsets(counts, count_is_i64, N, E, src_off, dst_off);

    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < E; ++j) {
            int64_t n = count_at(counts, count_is_i64, E, i, j);
            for (int64_t k = 0; k < n; ++k) {
                int64_t s = src_off[i * E + j] + k;   /* rank-major position  */
                int64_t d = dst_off[i * E + j] + k;   /* expert-major position */
                memcpy(tokens + s * row_bytes, permute_tokens + d * row_bytes, (size_t)row_bytes);
                if (permute_scales)
                    memcpy(scales + s * scale_row_bytes, permute_scales + d * scale_row_bytes,
                           (size_t)scale_row_bytes);
                if (permute_topk_w)
                    topk_w[s] = permute_topk_w[d];
            }
        }

    free(src_off);
    free(dst_off);
    return ORC_OK;
}

/*
 * expert_token_num in either mode ("CANN ops-transformer MoeReRoutingV2" article, section
 * 参数说明: 0 = cumsum mode, 1 = count mode; the dispatch page, parameter
 * expert_token_nums_type: 0 = prefix sum of the tokens each expert received, 1 = the count).
 *   count mode:  out[j] = sum over ranks i of counts[i][j]
 *   cumsum mode: out[j] = sum over experts j' <= j of the count-mode value (inclusive, so the
 *                last entry is A)
 * Written in the counts' integer type.  Returns ORC_ERR_ARG for a mode other than 0 or 1.
 */
int mrr_oracle_expert_token_num(const void *counts, int count_is_i64, int64_t N, int64_t E,
                                int64_t expert_token_num_type, void *out)
{
    int64_t running = 0;
    if (expert_token_num_type != 0 && expert_token_num_type != 1)
        return ORC_ERR_ARG;
    for (int64_t j = 0; j < E; ++j) {
        int64_t total = 0;
        for (int64_t i = 0; i < N; ++i)
            total += count_at(counts, count_is_i64, E, i, j);
        running += total;
        const int64_t v = expert_token_num_type == 1 ? total : running;
        if (count_is_i64)
            ((int64_t *)out)[j] = v;
        else
            ((int32_t *)out)[j] = (int32_t)v;
    }
    return ORC_OK;
}
