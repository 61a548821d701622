/*
 * mrr_gating.h -- C ABI of the MoE gating top-k op (the routing decision upstream of the
 * re-routing op), for GB300 (sm_103a).
 *
 * Definition: the article "CANN 自定义算子详解：npu_moe_gating_top_k 实现 MoE 路由与 TopK 专家选择"
 * (m.qwbw.cn/news/316089):
 *   - section 归一化公式: normOut = Softmax(x) (norm_type 0), Sigmoid(x) (1) or Softplus(x) (2);
 *     normOut += bias, and rows whose additional_token_mask is true use additional_bias instead;
 *   - section 分组排序公式: normOut splits into group_count groups; each is scored by its maximum
 *     (group_select_mode 0) or the sum of its two largest values (1); the k_group best are kept;
 *   - section 专家选择公式: with input_ids and tid2eid the experts are tid2eid[input_ids[t]]
 *     (hash routing); otherwise the k largest normOut values inside the kept groups;
 *   - section 路由权重缩放公式: y_out = y / (sum(y) + eps) * routed_scaling_factor;
 *   - sections 参数说明 / 约束说明: x [T, e] float16/bfloat16/float32, k <= min(e, 64),
 *     renorm only 0, 1 <= k_group <= group_count, k <= e / group_count * k_group, bias and
 *     additional_bias [e] in x's dtype, additional_token_mask [T] bool, input_ids [T] int64,
 *     tid2eid [n, k] int32; expert_idx int32; the normalised output is float32.
 *
 * Choices where the page is silent: normOut is computed and compared in float32 (the precision
 * the page stores it in) and equal scores go to the lower group / expert index; y and the
 * normalised output include the bias; experts are listed in descending score order; y_out has
 * x's dtype; e must be a multiple of group_count and, for group_select_mode 1, groups hold at
 * least 2 experts.  This implementation handles e <= 1024.  A row holding a NaN logit gets
 * unspecified experts.
 *
 * Asking for norm_out can change which path scores a row, and so, in rare rows, the result.
 * Without norm_out, rows with no bias, no groups and no hash table are ranked by their logits
 * and only the chosen experts are scored; with norm_out every expert is scored and the scores
 * are ranked.  The two agree (same experts, same order, same y_out bits) wherever CUDA's float32
 * exp / log1p are monotone across the logits involved.  CUDA does not document them as
 * monotone, so where two nearly equal logits round the other way round, the experts or their
 * order may differ between the two modes; the ranking by logit is then the one exact arithmetic
 * gives.
 */
#ifndef MRR_GATING_H
#define MRR_GATING_H

#include "mrr_v2.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mrr_gate_dtype {
    MRR_GATE_F16 = 0,
    MRR_GATE_BF16 = 1,
    MRR_GATE_F32 = 2
} mrr_gate_dtype;

/* largest number of experts (x's last dimension) mrr_gating_topk_run handles */
#define MRR_GATE_MAX_EXPERTS 1024

/*
 * mrr_gating_topk_run -- enqueue the gating op on `stream` (current device).
 *   x                     [T, e] in dt                                         (read)
 *   bias                  [e] in dt, or NULL                                   (read)
 *   input_ids, tid2eid    [T] int64 and [n_vocab, k] int32, both or neither (hash routing)
 *   additional_bias       [e] in dt; used only together with additional_token_mask
 *   additional_token_mask [T] bool (one byte per row, nonzero = true), or NULL
 *   y_out                 [T, k] in dt                                         (written)
 *   expert_idx            [T, k] int32                                         (written)
 *   norm_out              [T, e] float32, or NULL (the page's out_flag = false) (written)
 *   workspace             >= 4096 device bytes, 256-byte aligned: status words; read them
 *                         with mrr_v2_read_status (MRR_ERR_INDEX: an input_ids or tid2eid
 *                         value out of range; that row's outputs are then unspecified)
 * Host-side errors (returned at once, nothing enqueued): MRR_ERR_NULL, MRR_ERR_SHAPE (T < 0,
 * e outside 1..1024, k, grouping), MRR_ERR_DTYPE, MRR_ERR_ATTR (modes, renorm != 0),
 * MRR_ERR_TOPK_PAIR (only one of input_ids / tid2eid), MRR_ERR_WORKSPACE, MRR_ERR_CUDA.
 */
mrr_status mrr_gating_topk_run(const void *x, mrr_gate_dtype dt, int64_t T, int64_t e, int64_t k,
                               const void *bias, const int64_t *input_ids, const int32_t *tid2eid,
                               int64_t n_vocab, const void *additional_bias,
                               const uint8_t *additional_token_mask, int64_t k_group,
                               int64_t group_count, float routed_scaling_factor, float eps,
                               int64_t group_select_mode, int64_t renorm, int64_t norm_type,
                               void *y_out, int32_t *expert_idx, float *norm_out,
                               void *workspace, size_t workspace_bytes, mrr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MRR_GATING_H */
