// Host entry point of the MoE gating top-k op (include/mrr_gating.h): argument checks, the
// shared-memory layout and the choice of kernel instance.  The kernel is in gating_kernel.cuh.
//
// What it computes ("CANN 自定义算子详解：npu_moe_gating_top_k" article, sections 归一化公式,
// 分组排序公式, 专家选择公式, 路由权重缩放公式): per token row, normalised scores (softmax,
// sigmoid or softplus) plus a bias, a ranking of expert groups by their maximum or top-2 sum, the
// k best experts inside the k_group best groups (or a table lookup for hash routing), and the
// chosen scores scaled to sum to routed_scaling_factor.
#include "gating_kernel.cuh"

using namespace mrr_gate;

namespace {

constexpr int kVplChoices[] = {1, 2, 4, 6, 8, 12, 16, 24, 32};

int choose_vpl(int64_t e)
{
    const int64_t need = (e + 31) / 32;
    for (int v : kVplChoices)
        if (v >= need)
            return v;
    return 32;
}

}  // namespace

extern "C" mrr_status mrr_gating_topk_run(const void *x, mrr_gate_dtype dt, int64_t T, int64_t e, int64_t k,
                                          const void *bias, const int64_t *input_ids, const int32_t *tid2eid,
                                          int64_t n_vocab, const void *additional_bias,
                                          const uint8_t *additional_token_mask, int64_t k_group,
                                          int64_t group_count, float routed_scaling_factor, float eps,
                                          int64_t group_select_mode, int64_t renorm, int64_t norm_type,
                                          void *y_out, int32_t *expert_idx, float *norm_out, void *workspace,
                                          size_t workspace_bytes, mrr_stream_t stream_)
{
    // checks of the page's 约束说明 section and its Torch-side checks
    if (dt != MRR_GATE_F16 && dt != MRR_GATE_BF16 && dt != MRR_GATE_F32)
        return MRR_ERR_DTYPE;
    if (group_select_mode < 0 || group_select_mode > 1 || norm_type < 0 || norm_type > 2 || renorm != 0)
        return MRR_ERR_ATTR;
    if ((input_ids == nullptr) != (tid2eid == nullptr))
        return MRR_ERR_TOPK_PAIR;
    const bool hashing = input_ids != nullptr;
    if (T < 0 || T > INT32_MAX || e < 1 || e > MRR_GATE_MAX_EXPERTS || k < 1 || k > 64 || k > e)
        return MRR_ERR_SHAPE;
    if (group_count < 1 || k_group < 1 || k_group > group_count || e % group_count)
        return MRR_ERR_SHAPE;
    if (!hashing && k > (e / group_count) * k_group)
        return MRR_ERR_SHAPE;
    if (group_select_mode == 1 && e / group_count < 2)
        return MRR_ERR_SHAPE;
    if (hashing && n_vocab < 1)
        return MRR_ERR_SHAPE;
    if (T > 0 && (!x || !y_out || !expert_idx))
        return MRR_ERR_NULL;
    if (!workspace || ((uintptr_t)workspace % 256) || workspace_bytes < (size_t)kStatusWords * 4)
        return MRR_ERR_WORKSPACE;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int device = -1, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    Params p;
    memset(&p, 0, sizeof(p));
    p.x = x;
    p.dt = (int)dt;
    p.T = (int)T;
    p.e = (int)e;
    p.k = (int)k;
    p.bias = bias;
    p.input_ids = reinterpret_cast<const long long *>(input_ids);
    p.tid2eid = tid2eid;
    p.n_vocab = n_vocab;
    p.extra_bias = additional_bias;
    p.extra_mask = additional_token_mask;
    p.k_group = (int)k_group;
    p.group_count = (int)group_count;
    p.group_size = (int)(e / group_count);
    p.rsf = routed_scaling_factor;
    p.eps = eps;
    p.select_mode = (int)group_select_mode;
    p.norm_type = (int)norm_type;
    p.y_out = y_out;
    p.expert_idx = expert_idx;
    p.norm_out = norm_out;
    p.status = static_cast<uint32_t *>(workspace);

    const int xb = dt == MRR_GATE_F32 ? 4 : 2;
    const int vpl = choose_vpl(e);
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
    const int64_t row_bytes = e * xb;
    p.vec_bytes = 0;
    for (int w = 16; w >= 4; w >>= 1)
        if (xa % w == 0 && row_bytes % w == 0) {
            p.vec_bytes = w;
            break;
        }
    p.out_vec = norm_out && reinterpret_cast<uintptr_t>(norm_out) % 16 == 0 && e % 4 == 0;
    const int gs = (int)(e / group_count);
    p.group_path = kNoGroups;
    p.lanes_per_group = 0;
    if (!hashing && group_count > 1 && k_group < group_count) {
        const int lpg = gs / vpl;
        if (gs % vpl == 0 && (lpg & (lpg - 1)) == 0) {
            p.group_path = kLaneGroups;
            p.lanes_per_group = lpg;
            while ((1 << p.lpg_shift) < lpg)
                ++p.lpg_shift;
        } else {
            p.group_path = kSmemGroups;
        }
    }
    // shared memory: bias rows, then per-warp staging for hash lookups and smem group scores
    int words = 0;
    auto take = [&words](int64_t n) {
        const int off = words;
        words += (int)((n + 3) & ~int64_t(3));
        return off;
    };
    p.sm_bias = bias ? take(e) : -1;
    p.sm_extra = (additional_bias && additional_token_mask) ? take(e) : -1;
    p.sm_rows = (hashing || p.group_path == kSmemGroups) ? take(kWarps * e) : -1;
    p.sm_gkey = p.group_path == kSmemGroups ? take(kWarps * group_count) : -1;
    p.sm_kept = p.group_path == kSmemGroups ? take(kWarps * 32) : -1;
    const size_t smem = (size_t)words * 4;
    // rank by logit where the scores keep the logits' order and nothing else decides: no bias
    // rows, no groups, no hash table, no norm_out
    const bool by_logit = !hashing &&
                          p.group_path == kNoGroups && p.sm_bias < 0 && p.sm_extra < 0 && !norm_out &&
                          k <= (dt == MRR_GATE_F32 ? 31 : 32);
    // the grouped sigmoid instance: every condition its kernel takes as fixed (see full_row)
    const bool grouped_sigmoid = !by_logit && !hashing && p.group_path == kLaneGroups && group_count == 8 &&
                                 k == kFixedK && norm_type == 1 &&
                                 p.sm_bias == 0 && p.sm_extra < 0 && !norm_out && e == 32 * (int64_t)vpl &&
                                 p.vec_bytes == 16 && (vpl == 4 || vpl == 8 || vpl == 12 || vpl == 16);
    // the fixed-shape rank-by-logit instances: e = 32 * VPL, 16-byte rows, k in {2, 4, 6, 8}
    const bool logit_fixed = by_logit && e == 32 * (int64_t)vpl && p.vec_bytes == 16 &&
                             (vpl == 4 || vpl == 8 || vpl == 12 || vpl == 16) &&
                             (k == 2 || k == 4 || k == 6 || k == 8);
    const int path = by_logit ? (logit_fixed ? kPathLogitFixed : kPathLogit)
                              : (grouped_sigmoid ? kPathGroupedSigmoid : kPathFull);
    const cudaError_t err = dt == MRR_GATE_F32    ? launch_f32(p, vpl, path, smem, sms, stream)
                            : dt == MRR_GATE_BF16 ? launch_bf16(p, vpl, path, smem, sms, stream)
                                                  : launch_f16(p, vpl, path, smem, sms, stream);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    return MRR_OK;
}
