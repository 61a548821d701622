// GB300 (sm_103a) implementation of the MoE gating top-k op behind include/mrr_gating.h.
//
// What it computes ("CANN 自定义算子详解：npu_moe_gating_top_k" article, sections 归一化公式,
// 分组排序公式, 专家选择公式, 路由权重缩放公式): per token row, normalised scores (softmax,
// sigmoid or softplus) plus a bias, a ranking of expert groups by their maximum or top-2 sum, the
// k best experts inside the k_group best groups (or a table lookup for hash routing), and the
// chosen scores scaled to sum to routed_scaling_factor.
//
// GB300 design: the op reads T*e scores once and writes T*k results, so it is bound by memory
// and latency, not arithmetic.  One warp owns one row: lane l holds experts l, l+32, ... in
// registers (coalesced loads of the row), the scores are also staged in shared memory for the
// group statistics and table lookups, and every selection is a warp-wide arg-max by shuffles
// (ties to the lower index).  A grid of a few CTAs per SM strides over the rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "mrr_gating.h"
#include "ptx.cuh"

namespace mrr_gate {

constexpr int kWarps = 4;                       // rows per CTA per iteration
constexpr int kStatusWords = 1024;              // the status region shared with mrr_v2_read_status
constexpr int kMaxGrid = kStatusWords - 2;
constexpr uint32_t kFlagBadIndex = 8u;          // an input_ids / tid2eid value out of range
constexpr int kMaxExperts = MRR_GATE_MAX_EXPERTS;

struct Params {
    const void *x;
    int dt;
    int T, e, k;
    const void *bias;
    const long long *input_ids;
    const int *tid2eid;
    long long n_vocab;
    const void *extra_bias;
    const uint8_t *extra_mask;
    int k_group, group_count, group_size;
    float rsf, eps;
    int select_mode, norm_type;
    void *y_out;
    int *expert_idx;
    float *norm_out;
    uint32_t *status;
};

__device__ __forceinline__ float load_as_float(const void *p, int dt, long long i)
{
    if (dt == MRR_GATE_F32)
        return __ldg(static_cast<const float *>(p) + i);
    if (dt == MRR_GATE_BF16)
        return __bfloat162float(__ldg(static_cast<const __nv_bfloat16 *>(p) + i));
    return __half2float(__ldg(static_cast<const __half *>(p) + i));
}

__device__ __forceinline__ void store_from_float(void *p, int dt, long long i, float v)
{
    if (dt == MRR_GATE_F32)
        static_cast<float *>(p)[i] = v;
    else if (dt == MRR_GATE_BF16)
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else
        static_cast<__half *>(p)[i] = __float2half_rn(v);
}

// warp-wide arg-max: the larger value wins, equal values go to the lower index
__device__ __forceinline__ void warp_argmax(float &v, int &j)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oj = __shfl_xor_sync(0xffffffffu, j, o);
        if (ov > v || (ov == v && oj < j)) {
            v = ov;
            j = oj;
        }
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// VPL = values per lane: the row's e <= 32 * VPL experts live in registers, lane l holding
// experts l + 32 v.
template <int VPL>
__global__ void __launch_bounds__(32 * kWarps) gating_kernel(const Params p)
{
    extern __shared__ float smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = p.e, k = p.k, G = p.group_count, gs = p.group_size;
    float *s_score = smem + warp * (2 * kMaxExperts + 32);    // [e] scores of this warp's row
    float *s_group = s_score + kMaxExperts;                    // [G] group scores
    uint32_t *s_kept = reinterpret_cast<uint32_t *>(s_group + kMaxExperts);  // [32] kept-group bits

    // no global memory touched above: wait for the previous kernel on the stream, then let the
    // next launch be scheduled (programmatic stream serialization)
    mrr::grid_dependency_wait();
    mrr::grid_launch_dependents();
    uint32_t flags = 0u;
    const int rows_per_iter = gridDim.x * kWarps;
    for (int t = blockIdx.x * kWarps + warp; t < p.T; t += rows_per_iter) {
        // ---- steps 1-2: normalise, add the row's bias
        float v[VPL];
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int j = lane + 32 * u;
            v[u] = j < e ? load_as_float(p.x, p.dt, (long long)t * e + j) : -INFINITY;
        }
        if (p.norm_type == 0) {
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < VPL; ++u)
                mx = fmaxf(mx, v[u]);
            mx = warp_max(mx);
            float sum = 0.f;
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                v[u] = (lane + 32 * u < e) ? expf(v[u] - mx) : 0.f;
                sum += v[u];
            }
            sum = warp_sum(sum);
#pragma unroll
            for (int u = 0; u < VPL; ++u)
                v[u] = v[u] / sum;
        } else if (p.norm_type == 1) {
#pragma unroll
            for (int u = 0; u < VPL; ++u)
                v[u] = 1.f / (1.f + expf(-v[u]));
        } else {
#pragma unroll
            for (int u = 0; u < VPL; ++u)
                v[u] = v[u] > 20.f ? v[u] + log1pf(expf(-v[u])) : log1pf(expf(v[u]));
        }
        const bool extra = p.extra_bias && p.extra_mask && p.extra_mask[t];
        const void *bsrc = extra ? p.extra_bias : p.bias;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int j = lane + 32 * u;
            if (j < e) {
                if (bsrc)
                    v[u] = v[u] + load_as_float(bsrc, p.dt, j);
                s_score[j] = v[u];
                if (p.norm_out)
                    p.norm_out[(long long)t * e + j] = v[u];
            } else {
                v[u] = -INFINITY;
            }
        }
        __syncwarp();

        // ---- step 3: choose the experts; lane i (and i + 32) keeps result i (k <= 64)
        float y0 = 0.f, y1 = 0.f;
        int j0 = 0, j1 = 0;
        if (p.input_ids) {
            const long long id = p.input_ids[t];
            const bool ok = id >= 0 && id < p.n_vocab;
            for (int i = lane; i < k; i += 32) {
                int j = ok ? p.tid2eid[id * k + i] : -1;
                if (j < 0 || j >= e) {
                    flags |= kFlagBadIndex;
                    j = 0;
                }
                const float y = s_score[j];
                if (i < 32) {
                    y0 = y;
                    j0 = j;
                } else {
                    y1 = y;
                    j1 = j;
                }
            }
        } else {
            // group scores: maximum, or sum of the two largest (in float32)
            for (int g = lane; g < G; g += 32) {
                float m1 = -INFINITY, m2 = -INFINITY;
                for (int j = g * gs; j < (g + 1) * gs; ++j) {
                    const float s = s_score[j];
                    if (s > m1) {
                        m2 = m1;
                        m1 = s;
                    } else if (s > m2) {
                        m2 = s;
                    }
                }
                s_group[g] = p.select_mode == 0 ? m1 : m1 + m2;
            }
            s_kept[lane] = 0u;
            __syncwarp();
            for (int r = 0; r < p.k_group; ++r) {
                float bv = -INFINITY;
                int bg = 0x7fffffff;
                for (int g = lane; g < G; g += 32) {
                    const bool kept = (s_kept[g >> 5] >> (g & 31)) & 1u;
                    const float s = s_group[g];
                    if (!kept && (s > bv || (s == bv && g < bg))) {
                        bv = s;
                        bg = g;
                    }
                }
                warp_argmax(bv, bg);
                if (lane == 0)
                    s_kept[bg >> 5] |= 1u << (bg & 31);
                __syncwarp();
            }
            // the k largest scores among the kept groups' experts, in descending order
            uint32_t taken = 0u;  // bit u: this lane's expert lane + 32u is chosen or excluded
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const int j = lane + 32 * u;
                if (j >= e || !((s_kept[(j / gs) >> 5] >> ((j / gs) & 31)) & 1u))
                    taken |= 1u << u;
            }
            for (int i = 0; i < k; ++i) {
                float bv = -INFINITY;
                int bj = 0x7fffffff;
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    if (!((taken >> u) & 1u) && v[u] > bv) {  // lane's experts rise in index
                        bv = v[u];
                        bj = lane + 32 * u;
                    }
                }
                warp_argmax(bv, bj);
                if (bj < e && (bj & 31) == lane)
                    taken |= 1u << (bj >> 5);
                if (lane == (i & 31)) {
                    if (i < 32) {
                        y0 = bv;
                        j0 = bj;
                    } else {
                        y1 = bv;
                        j1 = bj;
                    }
                }
            }
        }

        // ---- step 4: scale and write
        const float ysum = warp_sum((lane < k ? y0 : 0.f) + (lane + 32 < k ? y1 : 0.f));
        const float scale = p.rsf / (ysum + p.eps);
        if (lane < k) {
            store_from_float(p.y_out, p.dt, (long long)t * k + lane, y0 * scale);
            p.expert_idx[(long long)t * k + lane] = j0;
        }
        if (lane + 32 < k) {
            store_from_float(p.y_out, p.dt, (long long)t * k + lane + 32, y1 * scale);
            p.expert_idx[(long long)t * k + lane + 32] = j1;
        }
        __syncwarp();
    }
    // per-CTA status word (plain stores: no clearing needed between calls)
    flags = __reduce_or_sync(0xffffffffu, flags);
    __shared__ uint32_t s_flags[kWarps];
    if (lane == 0)
        s_flags[warp] = flags;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t f = 0u;
        for (int w = 0; w < kWarps; ++w)
            f |= s_flags[w];
        p.status[2 + blockIdx.x] = f;
        if (blockIdx.x == 0) {
            p.status[0] = 0u;
            p.status[1] = gridDim.x;
        }
    }
}

}  // namespace mrr_gate

using namespace mrr_gate;

namespace {

template <int VPL>
cudaError_t launch_gating(const Params &p, int grid, cudaStream_t stream)
{
    // 4 rows x (1024 scores + 1024 group scores + 32 words): 33,280 bytes, under the 48 KiB default
    const size_t smem = (size_t)kWarps * (2 * kMaxExperts + 32) * sizeof(float);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(32 * kWarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gating_kernel<VPL>, p);
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

    int64_t want = (T + kWarps - 1) / kWarps;
    int64_t cap = 4 * (int64_t)sms;
    if (cap > kMaxGrid)
        cap = kMaxGrid;
    const int grid = (int)(want < 1 ? 1 : (want > cap ? cap : want));
    const int vpl_needed = (int)((e + 31) / 32);
    cudaError_t err;
    if (vpl_needed <= 1)
        err = launch_gating<1>(p, grid, stream);
    else if (vpl_needed <= 2)
        err = launch_gating<2>(p, grid, stream);
    else if (vpl_needed <= 4)
        err = launch_gating<4>(p, grid, stream);
    else if (vpl_needed <= 8)
        err = launch_gating<8>(p, grid, stream);
    else if (vpl_needed <= 16)
        err = launch_gating<16>(p, grid, stream);
    else
        err = launch_gating<32>(p, grid, stream);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    return MRR_OK;
}
