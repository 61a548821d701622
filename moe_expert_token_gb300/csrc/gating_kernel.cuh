// The MoE gating top-k kernel behind include/mrr_gating.h, for GB300 (sm_103a).  The kernel
// template lives here; gating_f16.cu, gating_bf16.cu and gating_f32.cu instantiate it for one
// dtype each (they compile in parallel), and gating.cu holds the host entry point.
//
// What it computes ("CANN 自定义算子详解：npu_moe_gating_top_k" article, sections 归一化公式,
// 分组排序公式, 专家选择公式, 路由权重缩放公式): per token row, normalised scores (softmax,
// sigmoid or softplus) plus a bias, a ranking of expert groups by their maximum or top-2 sum, the
// k best experts inside the k_group best groups (or a table lookup for hash routing), and the
// chosen scores scaled to sum to routed_scaling_factor.
//
// GB300 design.  The op reads T*e scores once and writes T*k results; its k picks per row make it
// bound by instruction issue long before HBM, so the kernel is built to spend few warp
// instructions per row:
//  * one warp owns one row; lane l holds the contiguous run of experts [l*VPL, (l+1)*VPL) in
//    registers, read with 16-, 8- or 4-byte loads where the row alignment allows;
//  * scores become order-preserving 32-bit keys, so an arg-max over the row is a redux.sync for
//    the largest key and then the lowest lane holding it (a ballot where k is a compile-time
//    constant, else a second redux.sync over the experts);
//  * each lane caches its three best remaining candidates and rescans its run only when all are
//    used, so a pick costs a handful of instructions instead of a pass over the row; the lane
//    that gave a pick records it in shared memory, and lane i reads pick i at the end;
//  * group scores come from a shuffle butterfly over the lanes' caches when each group is an
//    aligned block of lanes, else from the row staged in shared memory;
//  * where the normalisation alone ranks the experts (no bias, no groups), the row is ranked by
//    logit and only the chosen experts are scored; a 16-bit logit's order key is packed with its
//    expert into one word, so a pick is one redux.sync;
//  * the grouped sigmoid routing shape (8 lane-aligned groups, top-8, bias) has an instance of
//    its own with those facts fixed at compile time;
//  * 8 warps per CTA, shared memory sized to the call, as many CTAs as fit on the SMs.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "mrr_gating.h"
#include "ptx.cuh"

namespace mrr_gate {

constexpr int kWarps = 8;                       // rows in flight per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kStatusWords = 1024;              // the status region shared with mrr_v2_read_status
constexpr int kMaxGrid = kStatusWords - 2;
constexpr uint32_t kFlagBadIndex = 8u;          // an input_ids / tid2eid value out of range
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kNoIndex = 0xffffffffu;
constexpr int kSmemOptIn = 100 * 1024;          // the largest call needs 78,848 bytes

enum GroupPath { kNoGroups = 0, kLaneGroups = 1, kSmemGroups = 2 };
enum KernelPath { kPathFull = 0, kPathLogit = 1, kPathGroupedSigmoid = 2, kPathLogitFixed = 3 };
constexpr int kFixedK = 8;                      // the picks of the grouped sigmoid instance

struct Params {
    const void *x;
    int dt, T, e, k;
    int vec_bytes;            // widest row load (16, 8, 4; 0 = one element at a time) x allows
    const void *bias;
    const long long *input_ids;
    const int *tid2eid;
    long long n_vocab;
    const void *extra_bias;
    const uint8_t *extra_mask;
    int k_group, group_count, group_size, group_path, lanes_per_group, lpg_shift;
    float rsf, eps;
    int select_mode, norm_type;
    int out_vec;              // norm_out rows may be written with 16-byte stores
    // dynamic shared memory, offsets in 4-byte words (-1 = not allocated)
    int sm_bias, sm_extra, sm_rows, sm_gkey, sm_kept;
    void *y_out;
    int *expert_idx;
    float *norm_out;
    uint32_t *status;
};

// Order-preserving map of a float score to a 32-bit key: a larger float gives a larger key, equal
// floats equal keys (-0 is folded into +0 first).  Every score, -inf included, maps above 0, which
// therefore marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t b = __float_as_uint(f + 0.0f);
    return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);   // negative: all bits flip
}

__device__ __forceinline__ float key_value(uint32_t key)
{
    return __uint_as_float(key ^ ((uint32_t)((int32_t)~key >> 31) | 0x80000000u));
}

__device__ __forceinline__ float load_as_float(const void *p, int dt, long long i)
{
    if (dt == MRR_GATE_F32)
        return __ldg(static_cast<const float *>(p) + i);
    if (dt == MRR_GATE_BF16)
        return __bfloat162float(__ldg(static_cast<const __nv_bfloat16 *>(p) + i));
    return __half2float(__ldg(static_cast<const __half *>(p) + i));
}

template <int DT>
__device__ __forceinline__ float bits16_to_float(uint32_t h)
{
    if (DT == MRR_GATE_BF16)
        return __uint_as_float(h << 16);
    return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
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

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// warp_sum when only lanes below kLanes (a power of two) hold nonzero values: the same additions
// in the same order, less the rounds that only add zeros; lanes below kLanes get the sum
template <int kLanes>
__device__ __forceinline__ float warp_sum_low(float v)
{
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__host__ __device__ constexpr int pow2_at_least(int k) { return k <= 1 ? 1 : 2 * pow2_at_least((k + 1) / 2); }

// this lane's run of row `row` (e experts), experts [j0, j0 + VPL), as floats; experts at or past
// e read -inf.  vec_bytes is the widest load the rows' alignment allows.
template <int VPL, int DT>
__device__ __forceinline__ void load_run(float (&v)[VPL], const void *x, long long row, int e, int j0,
                                         int vec_bytes)
{
    const int nv = e - j0;
    if (DT == MRR_GATE_F32) {
        const float *src = static_cast<const float *>(x) + row * e + j0;
        if (VPL % 4 == 0 && nv >= VPL && vec_bytes >= 16) {
#pragma unroll
            for (int c = 0; c < VPL / 4; ++c) {
                const float4 q = __ldg(reinterpret_cast<const float4 *>(src) + c);
                v[4 * c] = q.x;
                v[4 * c + 1] = q.y;
                v[4 * c + 2] = q.z;
                v[4 * c + 3] = q.w;
            }
        } else if (VPL % 2 == 0 && nv >= VPL && vec_bytes >= 8) {
#pragma unroll
            for (int c = 0; c < VPL / 2; ++c) {
                const float2 q = __ldg(reinterpret_cast<const float2 *>(src) + c);
                v[2 * c] = q.x;
                v[2 * c + 1] = q.y;
            }
        } else {
#pragma unroll
            for (int u = 0; u < VPL; ++u)
                v[u] = u < nv ? __ldg(src + u) : -INFINITY;
        }
        return;
    }
    const unsigned short *src = static_cast<const unsigned short *>(x) + row * e + j0;
    if (VPL % 8 == 0 && nv >= VPL && vec_bytes >= 16) {
#pragma unroll
        for (int c = 0; c < VPL / 8; ++c) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(src) + c);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 8; ++h)
                v[8 * c + h] = bits16_to_float<DT>(w[h >> 1] >> (16 * (h & 1)));
        }
    } else if (VPL % 4 == 0 && nv >= VPL && vec_bytes >= 8) {
#pragma unroll
        for (int c = 0; c < VPL / 4; ++c) {
            const uint2 q = __ldg(reinterpret_cast<const uint2 *>(src) + c);
            const uint32_t w[2] = {q.x, q.y};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                v[4 * c + h] = bits16_to_float<DT>(w[h >> 1] >> (16 * (h & 1)));
        }
    } else if (VPL % 2 == 0 && nv >= VPL && vec_bytes >= 4) {
#pragma unroll
        for (int c = 0; c < VPL / 2; ++c) {
            const uint32_t q = __ldg(reinterpret_cast<const unsigned int *>(src) + c);
            v[2 * c] = bits16_to_float<DT>(q);
            v[2 * c + 1] = bits16_to_float<DT>(q >> 16);
        }
    } else {
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            v[u] = u < nv ? bits16_to_float<DT>(__ldg(src + u)) : -INFINITY;
    }
}

// The two element-wise normalisations.  Both rank-by-logit rows and fully evaluated rows call
// these, so a score is the same float whichever path computed it.
//
// Sigmoid: 1 / (1 + e^-x) with e^-x = 2^(-x log2 e).  The product -x log2 e is carried in two
// floats, hi + lo (Cody and Waite's split of the constant, "Software Manual for the Elementary
// Functions", 1980: log2 e = kHi + kLo with kHi a float, and an fma recovers the rounding error of
// -x kHi exactly).  The hardware base-2 exponential (ex2.approx) takes hi and the first-order
// factor 2^lo = 1 + lo ln 2 corrects for lo.  The sum is formed at half scale, d = (1 + e^-x) / 2
// = 2^hi (1/2 + lo ln 2 / 2) + 1/2, in one fma (one rounding where 1 + 2^hi 2^lo took two), and
// sigmoid = rcp.approx(d) / 2, the halving exact.  Rounding -x log2 e to one float instead would
// cost up to |x| 2^-24 ln 2 of relative error, about 17 ulp at |x| = 25.
// lo is tiny wherever 2^hi is a normal float.  The extremes: hi is capped at 200 (2^hi is inf from
// 128 on), so for x below about -139 or x = -inf lo is large or +inf, the factor saturates to 1
// and d = inf: sigmoid 0.  For large x or x = +inf, 2^hi = 0 and the factor (a NaN at +inf, which
// the saturating fma turns into 0) stays in [0, 1], so d = 1/2: sigmoid 1.  A NaN logit gives
// hi = 200, factor 0 and d = inf * 0: the score stays NaN.  Subnormals flush: 2^hi below 2^-126
// gives d = 1/2, and a sigmoid below the smallest normal float comes out 0 or subnormal.  Over
// every float16 and bfloat16 logit the result is within a few float32 ulps of the exact sigmoid
// (tests/test_gating_gpu.py measures it).
__device__ __forceinline__ float ex2_approx_ftz(float t)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

__device__ __forceinline__ float rcp_approx_ftz(float t)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

__device__ __forceinline__ float fma_sat(float a, float b, float c)
{
    float r;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float sigmoid_score(float x)
{
    constexpr float kHi = 1.44269502162933349609375f;   // log2 e rounded to float
    constexpr float kLo = 1.9259629911266175e-8f;        // log2 e - kHi
    constexpr float kHalfLn2 = 0.3465735902799726547f;
    const float hi = fminf(-x * kHi, 200.f);
    const float lo = fmaf(-x, kLo, fmaf(-x, kHi, -hi));
    const float d = fmaf(ex2_approx_ftz(hi), fma_sat(lo, kHalfLn2, 0.5f), 0.5f);
    return 0.5f * rcp_approx_ftz(d);
}

__device__ __forceinline__ float softplus_score(float x)
{
    return x > 20.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// steps 1-2 of the page for this lane's run: normalise, then add the row's bias (from shared memory)
template <int VPL>
__device__ __forceinline__ void normalise_and_bias(float (&v)[VPL], int norm_type, int nv, const float *bias)
{
    if (norm_type == 0) {
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            mx = fmaxf(mx, v[u]);
        mx = key_value(__reduce_max_sync(kFull, order_key(mx)));
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            v[u] = expf(v[u] - mx);      // experts past e: exp(-inf) = 0
            sum += v[u];
        }
        const float r = __frcp_rn(warp_sum(sum));
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            v[u] *= r;
    } else if (norm_type == 1) {
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            v[u] = sigmoid_score(v[u]);
    } else {
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            v[u] = softplus_score(v[u]);
    }
    if (bias == nullptr)
        return;
    if (VPL % 4 == 0 && nv >= VPL) {
#pragma unroll
        for (int c = 0; c < VPL / 4; ++c) {
            const float4 b = reinterpret_cast<const float4 *>(bias)[c];
            v[4 * c] += b.x;
            v[4 * c + 1] += b.y;
            v[4 * c + 2] += b.z;
            v[4 * c + 3] += b.w;
        }
    } else {
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u < nv)
                v[u] += bias[u];
    }
}

// A lane's view of its run during the picks: its three best remaining keys (b1 >= b2 >= b3) with
// their experts, and what moves in behind b3 when one is given up: 0 when those three were all the
// lane had, else kRefill.  A lane whose b1 reads kRefill has given up its three and must look at
// its run again before the next pick.  Three rather than two: on the grouped 256-expert case the
// eight picks crowd into the kept groups' 16 lanes, and a two-key cache rescanned about 1.3 times
// per row (a top-3 cache 0.13 times).
constexpr uint32_t kRefill = 0xffffffffu;   // above every key but a NaN score's

struct LaneCands {
    uint32_t b1, b2, b3, fill;
    uint32_t u1, u2, u3;
};

// insert key (expert u) into the lane's three best; equal keys keep the earlier expert first
__device__ __forceinline__ void insert3(LaneCands &c, uint32_t key, uint32_t u)
{
    const bool over1 = key > c.b1, over2 = key > c.b2, over3 = key > c.b3;
    c.b3 = over2 ? c.b2 : (over3 ? key : c.b3);
    c.u3 = over2 ? c.u2 : (over3 ? u : c.u3);
    c.b2 = over1 ? c.b1 : (over2 ? key : c.b2);
    c.u2 = over1 ? c.u1 : (over2 ? u : c.u2);
    c.b1 = over1 ? key : c.b1;
    c.u1 = over1 ? u : c.u1;
}

// the lane's three best keys among those `live` admits (the run starts at expert j0)
template <int VPL, typename Live>
__device__ __forceinline__ void scan3(LaneCands &c, const uint32_t (&kv)[VPL], uint32_t j0, Live live)
{
    c.b1 = c.b2 = c.b3 = 0u;
    c.u1 = c.u2 = c.u3 = j0;
#pragma unroll
    for (int u = 0; u < VPL; ++u)
        insert3(c, live(kv[u], j0 + u) ? kv[u] : 0u, j0 + u);
    c.fill = c.b3 == 0u ? 0u : kRefill;
}

template <int VPL>
__device__ __forceinline__ void first_scan(LaneCands &c, const uint32_t (&kv)[VPL], uint32_t j0)
{
    scan3<VPL>(c, kv, j0, [](uint32_t, uint32_t) { return true; });
}

// A lane that has given up its three cached keys looks at its run again: the keys still there are
// those below the last key it gave up, or equal to it at a later expert (keys leave a lane in
// that order).  The last key it gave up is found among the n picks so far.  Rarely taken, so it is
// a call of its own: the run is passed by value and the pick loop keeps its registers.
template <int VPL>
struct KeyRun {
    uint32_t k[VPL];
};

template <int VPL>
__device__ __noinline__ LaneCands refill(const KeyRun<VPL> run, uint32_t j0, const uint2 *s_pick, int n)
{
    bool gave = false;
    uint32_t last_key = 0u, last_u = 0u;
    for (int p = 0; p < n; ++p) {
        const uint2 q = s_pick[p];
        if (q.y - j0 < (uint32_t)VPL) {
            gave = true;
            last_key = q.x;
            last_u = q.y;
        }
    }
    LaneCands c;
    scan3<VPL>(c, run.k, j0, [&](uint32_t key, uint32_t u) {
        return !gave || key < last_key || (key == last_key && u > last_u);
    });
    return c;
}

// The k picks: each is the largest remaining key over the warp (a redux.sync), ties to the lower
// expert.  A lane's experts all come before the next lane's and its cache keeps equal keys in
// expert order, so the pick goes to the lowest lane whose b1 is the top key: one ballot when k is
// a compile-time kK (the picks then unrolled), else a second redux.sync for the lowest expert.
// The giving lane records the pick in s_pick[i] (64 entries per warp).  Lane i returns pick i's
// key and expert in (k0, i0), pick i + 32's in (k1, i1).
template <int VPL, int kK = 0>
__device__ __forceinline__ void pick_keys(LaneCands &c, const uint32_t (&kv)[VPL], int j0, int lane, int k,
                                          uint2 *s_pick, uint32_t &k0, uint32_t &i0, uint32_t &k1, uint32_t &i1)
{
    const uint32_t below = (1u << lane) - 1u;   // the lanes below this one
    auto pick = [&](int i) {
        uint32_t top = __reduce_max_sync(kFull, c.b1);
        // a lane uses up its three cached keys after giving three picks at the earliest; before
        // that a top of kRefill is a NaN score's key, which is picked like any other
        if (i >= 3 && top == kRefill) {   // some lane has used up its cache (or a NaN score)
            __syncwarp();
            if (c.b1 == kRefill) {
                KeyRun<VPL> run;
#pragma unroll
                for (int u = 0; u < VPL; ++u)
                    run.k[u] = kv[u];
                c = refill<VPL>(run, (uint32_t)j0, s_pick, i);
            }
            top = __reduce_max_sync(kFull, c.b1);
        }
        bool give;
        if constexpr (kK > 0) {   // the lowest lane at the top key
            const bool at_top = c.b1 == top;
            const uint32_t tied = __ballot_sync(kFull, at_top);
            give = at_top && (tied & below) == 0u;
        } else {
            give = c.u1 == __reduce_min_sync(kFull, c.b1 == top ? c.u1 : kNoIndex);
        }
        if (give) {
            s_pick[i] = make_uint2(top, c.u1);
            c.b1 = c.b2;
            c.u1 = c.u2;
            c.b2 = c.b3;
            c.u2 = c.u3;
            c.b3 = c.fill;
        }
    };
    if constexpr (kK > 0) {
#pragma unroll
        for (int i = 0; i < kK; ++i)
            pick(i);
    } else {
        for (int i = 0; i < k; ++i)
            pick(i);
    }
    __syncwarp();
    const uint2 p0 = lane < k ? s_pick[lane] : make_uint2(0u, 0u);
    const uint2 p1 = lane + 32 < k ? s_pick[lane + 32] : make_uint2(0u, 0u);
    __syncwarp();   // the next row's picks overwrite s_pick
    k0 = p0.x;
    i0 = p0.y;
    k1 = p1.x;
    i1 = p1.y;
}

// CTAs per SM each width is compiled for (its register budget: 40, 48, 64 or 80 per thread).
// Measured on GB300: 5 CTAs for 12 experts per lane beat 4 by 3.6 %; 6 CTAs for 8 per lane (40
// registers) beat 5 by 2 % on the grouped 256-expert case once the picks kept no last-key state.
constexpr int min_ctas_per_sm(int vpl) { return vpl <= 8 ? 6 : (vpl <= 12 ? 5 : (vpl <= 16 ? 4 : 3)); }

// Steps 1-3 of the page for row t with every score evaluated: normalise the lane's run, add the
// bias, rank the groups, make the k picks (or look the experts up for hash routing).  Lane i
// returns pick i in (y0, i0) and pick i + 32 in (y1, i1).
//
// kFixed: the instance for the grouped sigmoid case (DeepSeek-V3's routing shape), launched only
// when e = 32 * VPL, x's rows take 16-byte loads, the bias row is given, the experts form 8
// groups (each an aligned block of 4 lanes), k = kFixedK, the normalisation is sigmoid, and there
// is no hash table, no additional bias and no norm_out.  Those are then compile-time facts: the
// same arithmetic in the same order as the general instance, with its checks and loops over them
// folded away.
template <int VPL, int DT, bool kFixed>
__device__ __forceinline__ void full_row(const Params &p, int t, int lane, int j0, int nv_rt, float *smem,
                                         float *s_row, uint32_t *s_gkey, uint32_t *s_kept, uint2 *s_pick,
                                         uint32_t &flags, float &y0, uint32_t &i0, float &y1, uint32_t &i1)
{
    const int e = kFixed ? 32 * VPL : p.e, k = kFixed ? kFixedK : p.k;
    const int nv = kFixed ? VPL : nv_rt;
    const int group_path = kFixed ? (int)kLaneGroups : p.group_path;
    // ---- steps 1-2
    float v[VPL];
    load_run<VPL, DT>(v, p.x, t, e, j0, kFixed ? 16 : p.vec_bytes);
    const bool extra = !kFixed && p.sm_extra >= 0 && p.extra_mask[t];
    const float *bias = kFixed ? smem + j0
                               : (extra ? smem + p.sm_extra + j0 : (p.sm_bias >= 0 ? smem + p.sm_bias + j0 : nullptr));
    normalise_and_bias<VPL>(v, kFixed ? 1 : p.norm_type, nv, bias);
    if (!kFixed && p.norm_out) {
        float *dst = p.norm_out + (long long)t * e + j0;
        if (VPL % 4 == 0 && nv >= VPL && p.out_vec) {
#pragma unroll
            for (int c = 0; c < VPL / 4; ++c)
                reinterpret_cast<float4 *>(dst)[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        } else {
#pragma unroll
            for (int u = 0; u < VPL; ++u)
                if (u < nv)
                    dst[u] = v[u];
        }
    }

    // ---- step 3
    y0 = y1 = 0.f;
    i0 = i1 = 0u;
    if (!kFixed && p.input_ids) {
        // hash routing: the table row, scores looked up in the staged row
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u < nv)
                s_row[j0 + u] = v[u];
        __syncwarp();
        const long long id = p.input_ids[t];
        const bool ok = id >= 0 && id < p.n_vocab;
        for (int i = lane; i < k; i += 32) {
            int j = ok ? p.tid2eid[id * k + i] : -1;
            if (j < 0 || j >= e) {
                flags |= kFlagBadIndex;
                j = 0;
            }
            if (i < 32) {
                y0 = s_row[j];
                i0 = (uint32_t)j;
            } else {
                y1 = s_row[j];
                i1 = (uint32_t)j;
            }
        }
        __syncwarp();
    } else {
    uint32_t kv[VPL];
#pragma unroll
    for (int u = 0; u < VPL; ++u)
        kv[u] = order_key(v[u]);
    if (nv < VPL) {          // experts past e are no candidates
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u >= nv)
                kv[u] = 0u;
    }

    LaneCands c;
    if (group_path == kLaneGroups) {
        // each group is an aligned block of lanes_per_group lanes (a power of two); the group's
        // two best keys come from the lanes' caches
        first_scan<VPL>(c, kv, (uint32_t)j0);
        const int lpg = kFixed ? 4 : p.lanes_per_group;
        const int g = lane >> (kFixed ? 2 : p.lpg_shift);
        const bool member = kFixed || g < p.group_count;
        uint32_t g1 = c.b1, g2 = c.b2;
        for (int o = 1; o < lpg; o <<= 1) {
            const uint32_t o1 = __shfl_xor_sync(kFull, g1, o), o2 = __shfl_xor_sync(kFull, g2, o);
            g2 = max(max(g2, o2), min(g1, o1));
            g1 = max(g1, o1);
        }
        const uint32_t gkey = p.select_mode == 0 ? g1 : order_key(key_value(g1) + key_value(g2));
        const bool leader = member && (lane & (lpg - 1)) == 0;
        bool kept = false;
        if constexpr (kFixed) {
            // 8 groups: a group's rank is the number of groups ranked above it (a higher score,
            // or an equal one at a lower group).  The group keys sit in lanes 0, 4, ..., 28; lane
            // s of a group's four compares its key with groups 2s and 2s + 1, and the four add up.
            const int s = lane & 3, ha = 2 * s, hb = 2 * s + 1;
            const uint32_t ka = __shfl_sync(kFull, gkey, 4 * ha), kb = __shfl_sync(kFull, gkey, 4 * hb);
            int above = (ka > gkey || (ka == gkey && ha < g)) ? 1 : 0;
            above += (kb > gkey || (kb == gkey && hb < g)) ? 1 : 0;
            above += __shfl_xor_sync(kFull, above, 1);
            above += __shfl_xor_sync(kFull, above, 2);
            kept = above < p.k_group;
        } else {
            for (int r = 0; r < p.k_group; ++r) {
                const bool cand = leader && !kept;
                const uint32_t top = __reduce_max_sync(kFull, cand ? gkey : 0u);
                const uint32_t win = __reduce_min_sync(kFull, cand && gkey == top ? (uint32_t)g : kNoIndex);
                kept = kept || (member && (uint32_t)g == win);
            }
        }
        if (!kept) {   // a dropped group's experts leave the candidates
            c.b1 = c.b2 = c.b3 = 0u;
            c.fill = 0u;
        }
    } else {
    if (group_path == kSmemGroups) {
        const int G = p.group_count, gs = p.group_size;
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u < nv)
                s_row[j0 + u] = v[u];
        s_kept[lane] = 0u;
        __syncwarp();
        for (int g = lane; g < G; g += 32) {
            float m1 = -INFINITY, m2 = -INFINITY;
            for (int j = g * gs; j < (g + 1) * gs; ++j) {
                const float s = s_row[j];
                m2 = fmaxf(m2, fminf(m1, s));
                m1 = fmaxf(m1, s);
            }
            s_gkey[g] = order_key(p.select_mode == 0 ? m1 : m1 + m2);
        }
        __syncwarp();
        for (int r = 0; r < p.k_group; ++r) {
            uint32_t best = 0u, bg = kNoIndex;
            for (int g = lane; g < G; g += 32) {   // g rises: the first of equal keys stays
                const uint32_t key = ((s_kept[g >> 5] >> (g & 31)) & 1u) ? 0u : s_gkey[g];
                if (key > best) {
                    best = key;
                    bg = (uint32_t)g;
                }
            }
            const uint32_t top = __reduce_max_sync(kFull, best);
            const uint32_t win = __reduce_min_sync(kFull, best == top ? bg : kNoIndex);
            if (lane == 0 && win < (uint32_t)G)
                s_kept[win >> 5] |= 1u << (win & 31);
            __syncwarp();
        }
        // experts of dropped groups leave the candidates
        int g = j0 / gs, r = j0 - g * gs;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            if (u < nv && !((s_kept[g >> 5] >> (g & 31)) & 1u))
                kv[u] = 0u;
            if (++r == gs) {
                r = 0;
                ++g;
            }
        }
        __syncwarp();
    }
    first_scan<VPL>(c, kv, (uint32_t)j0);
    }

    uint32_t k0, k1;
    pick_keys<VPL, kFixed ? kFixedK : 0>(c, kv, j0, lane, k, s_pick, k0, i0, k1, i1);
    y0 = key_value(k0);
    y1 = key_value(k1);
    }
}

// the lane's two largest packed words below `below`
template <int VPL>
__device__ __forceinline__ void packed_top2(uint32_t &c1, uint32_t &c2, const uint32_t (&pk)[VPL], uint32_t below)
{
    c1 = c2 = 0u;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const uint32_t w = pk[u] < below ? pk[u] : 0u;
        c2 = max(c2, min(c1, w));
        c1 = max(c1, w);
    }
}

// the 16-bit logit whose order key is `key`, as float
template <int DT>
__device__ __forceinline__ float logit_value(uint32_t key)
{
    const uint32_t h = key >= 0x8000u ? key - 0x8000u : 0x8000u | (0x8000u - key);
    return bits16_to_float<DT>(h);
}

// The score of one logit, computed as the full evaluation computes it.  Softmax needs the row's
// largest logit mx and the reciprocal r of the row's exp-sum.
struct LogitScorer {
    int norm_type;
    float mx, r;
    __device__ __forceinline__ float operator()(float x) const
    {
        if (norm_type == 0)
            return expf(x - mx) * r;
        return norm_type == 1 ? sigmoid_score(x) : softplus_score(x);
    }
};

// Softmax's mx and r for a row whose largest logit is mx: the lane adds exp(x - mx) over its run
// in slot order, as the full evaluation does (experts past e add nothing), then the warp sums.
template <int VPL>
__device__ __forceinline__ float softmax_rcp(const float (&x)[VPL], int nv, float mx)
{
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < VPL; ++u)
        if (u < nv)
            sum += expf(x[u] - mx);
    return __frcp_rn(warp_sum(sum));
}

// this lane's run of row `row` as 16-bit words, two experts per 32-bit word (experts past e: zero)
template <int VPL>
__device__ __forceinline__ void load_words(uint32_t (&w)[(VPL + 1) / 2], const void *x, int row, int e, int vec_bytes,
                                           int j0, int nv)
{
    constexpr int W = (VPL + 1) / 2;
    const unsigned short *src = static_cast<const unsigned short *>(x) + (long long)row * e + j0;
    if (VPL % 8 == 0 && nv >= VPL && vec_bytes >= 16) {
#pragma unroll
        for (int c = 0; c < VPL / 8; ++c) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(src) + c);
            w[4 * c] = q.x;
            w[4 * c + 1] = q.y;
            w[4 * c + 2] = q.z;
            w[4 * c + 3] = q.w;
        }
    } else if (VPL % 4 == 0 && nv >= VPL && vec_bytes >= 8) {
#pragma unroll
        for (int c = 0; c < VPL / 4; ++c) {
            const uint2 q = __ldg(reinterpret_cast<const uint2 *>(src) + c);
            w[2 * c] = q.x;
            w[2 * c + 1] = q.y;
        }
    } else if (VPL % 2 == 0 && nv >= VPL && vec_bytes >= 4) {
#pragma unroll
        for (int c = 0; c < W; ++c)
            w[c] = __ldg(reinterpret_cast<const unsigned int *>(src) + c);
    } else {
#pragma unroll
        for (int c = 0; c < W; ++c)
            w[c] = 0u;
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u < nv)
                w[u >> 1] |= (uint32_t)__ldg(src + u) << (16 * (u & 1));
    }
}

// Lane i < k holds pick i's logit as an order key (a larger logit, a larger key; keys of
// adjacent representable logits differ by 1).  The picks rank exactly as their scores would when
//  * each pick i < k - 1 scores strictly above pick i + 1, or has the same logit (then the lower
//    expert is first either way), and
//  * pick k - 1 scores strictly above the next lower logit, so no expert left out can tie with it.
// Lane k (idle otherwise) scores that next lower logit; at k = 32, lane 31 does it as well.
// Returns whether both hold (warp-uniform); lane i < k gets pick i's score in f.
template <typename ScoreOf>
__device__ __forceinline__ bool logit_rank_holds(uint32_t key, int lane, int k, ScoreOf score_of, float &f)
{
    const uint32_t key_prev = __shfl_up_sync(kFull, key, 1);
    f = score_of(lane == k ? key_prev - 1u : key);
    const float f_next = __shfl_down_sync(kFull, f, 1);
    const uint32_t key_next = __shfl_down_sync(kFull, key, 1);
    bool unsure;
    if (lane == k - 1)
        unsure = key > 1u && !((k < 32 ? f_next : score_of(key - 1u)) < f);
    else
        unsure = lane < k && key_next != key && !(f > f_next);
    return !__any_sync(kFull, unsure);
}

// Rank by logit.  Softmax, sigmoid and softplus are non-decreasing in the logit, so with no bias
// and no groups the order of the scores is the order of the logits, and only the chosen experts
// need a score (softmax still sums exp over the row).  For
// 16-bit x the lane packs each logit's 16-bit order key above (0xffff - expert): the packed words
// are distinct, and one unsigned max over the row gives the largest logit and, among equal
// logits, the lowest expert, so a pick is a single redux.sync.
//
// Float32 rounding can give different logits the same score (sigmoid saturates near 1), and the
// ranking by score then puts the lower expert first.  The row checks the conditions of
// logit_rank_holds under which the two rankings agree; where one fails it returns false and the
// caller evaluates the row in full.  Otherwise lane i < k returns pick i in (y, idx), the same
// expert, order and score as the full evaluation (for float32 functions that are monotone there).
template <int VPL, int DT, int kK>
__device__ __forceinline__ bool logit_ranked_row(const Params &p, int t, int lane, int nv,
                                                 const uint32_t (&w)[(VPL + 1) / 2], const uint32_t (&ip)[(VPL + 1) / 2],
                                                 float &y, uint32_t &idx)
{
    constexpr int W = (VPL + 1) / 2;
    const int k = kK ? kK : p.k;   // kK: the fixed-shape instance (e = 32 * VPL, 16-byte loads)
    // 16-bit order keys, two at a time: positive h -> h ^ 0x8000, negative h -> (h ^ 0xffff) + 1,
    // so -0 and +0 both map to 0x8000 and every key is >= 1; then packed with the expert
    uint32_t pk[VPL];
#pragma unroll
    for (int c = 0; c < W; ++c) {
        const uint32_t s = (w[c] >> 15) & 0x00010001u;
        const uint32_t key2 = (w[c] ^ (s * 0x7fffu) ^ 0x80008000u) + s;
        pk[2 * c] = __byte_perm(key2, ip[c], 0x1054);
        if (2 * c + 1 < VPL)
            pk[2 * c + 1] = __byte_perm(key2, ip[c], 0x3276);
    }
    if (nv < VPL) {          // experts past e are no candidates
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u >= nv)
                pk[u] = 0u;
    }

    // k picks; a lane keeps its two best remaining words and rescans below the last one it gave
    // up when both are gone
    uint32_t c1 = pk[0], c2 = 0u;
#pragma unroll
    for (int u = 1; u < VPL; ++u) {
        c2 = max(c2, min(c1, pk[u]));
        c1 = max(c1, pk[u]);
    }
    bool complete = c2 == 0u;
    uint32_t pick = 0u;
    for (int i = 0; i < k; ++i) {
        const uint32_t top = __reduce_max_sync(kFull, c1);
        pick = lane == i ? top : pick;
        bool need = false;
        uint32_t last = 0u;
        if (c1 == top) {   // this lane gave the pick (never 0: the row has e >= k candidates)
            last = c1;
            c1 = c2;
            c2 = 0u;
            need = !complete && c1 == 0u;
        }
        if (__any_sync(kFull, need) && need) {
            packed_top2<VPL>(c1, c2, pk, last);
            complete = c2 == 0u;
        }
    }

    // lane i: pick i's expert and score
    LogitScorer score{p.norm_type, 0.f, 0.f};
    if (p.norm_type == 0) {   // the run again (an L1 hit), rather than held across the picks
        uint32_t w2[(VPL + 1) / 2];
        load_words<VPL>(w2, p.x, t, kK ? 32 * VPL : p.e, kK ? 16 : p.vec_bytes, lane * VPL, nv);
        float x[VPL];
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            x[u] = bits16_to_float<DT>(w2[u >> 1] >> (16 * (u & 1)));
        score.mx = logit_value<DT>(__shfl_sync(kFull, pick, 0) >> 16);
        score.r = softmax_rcp<VPL>(x, nv, score.mx);
    }
    float f;
    if (!logit_rank_holds(pick >> 16, lane, k, [&](uint32_t key) { return score(logit_value<DT>(key)); }, f))
        return false;
    y = lane < k ? f : 0.f;
    idx = 0xffffu - (pick & 0xffffu);
    return true;
}

// Rank by logit for float32 x: the logits' 32-bit order keys go through the same cached-key picks
// as the full evaluation's scores, and only the chosen experts are scored.  The next lower float32
// logit is one ulp down and almost always scores the same, so the boundary is checked against
// the expert actually ranked next instead: the row takes k + 1 picks (k <= 31), and pick k - 1
// must score strictly above pick k (then every expert left out scores below pick k - 1).  The
// other picks are checked as for 16-bit logits.
template <int VPL, int kK>
__device__ __forceinline__ bool logit_ranked_row_f32(const Params &p, int t, int lane, int j0, int nv, uint2 *s_pick,
                                                     float &y, uint32_t &idx)
{
    const int k = kK ? kK : p.k;   // kK: the fixed-shape instance (e = 32 * VPL, 16-byte loads)
    float v[VPL];
    load_run<VPL, MRR_GATE_F32>(v, p.x, t, kK ? 32 * VPL : p.e, j0, kK ? 16 : p.vec_bytes);
    uint32_t kv[VPL];
#pragma unroll
    for (int u = 0; u < VPL; ++u)
        kv[u] = order_key(v[u]);
    if (nv < VPL) {          // experts past e are no candidates
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (u >= nv)
                kv[u] = 0u;
    }
    uint32_t key, k1, i1;
    LaneCands c;
    first_scan<VPL>(c, kv, (uint32_t)j0);
    // lane k: the first expert left out
    pick_keys<VPL, kK ? kK + 1 : 0>(c, kv, j0, lane, k + 1, s_pick, key, idx, k1, i1);
    LogitScorer score{p.norm_type, 0.f, 0.f};
    if (p.norm_type == 0) {   // the run again (an L1 hit), rather than held across the picks
        load_run<VPL, MRR_GATE_F32>(v, p.x, t, kK ? 32 * VPL : p.e, j0, kK ? 16 : p.vec_bytes);
        score.mx = key_value(__shfl_sync(kFull, key, 0));
        score.r = softmax_rcp<VPL>(v, nv, score.mx);
    }
    const float f = score(key_value(key));
    const float f_next = __shfl_down_sync(kFull, f, 1);
    const uint32_t key_next = __shfl_down_sync(kFull, key, 1);
    bool unsure;
    if (lane == k - 1)
        unsure = key_next != 0u && !(f > f_next);   // e == k: nobody is left out
    else
        unsure = lane < k && key_next != key && !(f > f_next);
    if (__any_sync(kFull, unsure))
        return false;
    y = lane < k ? f : 0.f;
    return true;
}

// VPL = experts per lane (the row's e <= 32 * VPL scores live in registers); DT = x's type;
// kPath: kPathFull evaluates every score; kPathLogit ranks by logit (no bias, no groups, no hash
// routing, no norm_out, k <= 32, or k <= 31 for float32 x), with the full evaluation as the
// fallback; kPathGroupedSigmoid is the full evaluation specialised as full_row's kFixed says;
// kPathLogitFixed ranks by logit with the row shape fixed: e = 32 * VPL, 16-byte loads, k = kK
// (the host launches it only then; the same arithmetic, with the pick loop unrolled).
//
// Register budget: min_ctas_per_sm(VPL), except for the fixed-shape float32 rank-by-logit
// instances, whose unrolled picks over 32-bit keys spilled at 48 registers (12 experts per lane):
// 4 CTAs (64 registers) measured 13.37 -> 12.17 us on 16384 x 384 float32 logits, top-6.
template <int VPL, int DT, int kPath, int kK = 0>
__global__ void __launch_bounds__(kThreads, (DT == MRR_GATE_F32 && kPath == kPathLogitFixed) ? 4 : min_ctas_per_sm(VPL))
    gating_kernel(const Params p)
{
    constexpr bool kFixedLogit = kPath == kPathLogitFixed;
    constexpr bool kByLogit = kPath == kPathLogit || kFixedLogit, kFixed = kPath == kPathGroupedSigmoid;
    extern __shared__ __align__(16) float smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = (kFixed || kFixedLogit) ? 32 * VPL : p.e;
    const int k = kFixed ? kFixedK : (kFixedLogit ? kK : p.k);
    const int j0 = lane * VPL, nv = e - j0;
#define MRR_GATE_ROW_SHAPE (kFixedLogit ? 32 * VPL : p.e), (kFixedLogit ? 16 : p.vec_bytes)

    // no global memory touched above: wait for the previous kernel on the stream, then let the
    // next launch be scheduled (programmatic stream serialization)
    mrr::grid_dependency_wait();
    mrr::grid_launch_dependents();

    // the bias rows, once per CTA, as float
    if (p.sm_bias >= 0)
        for (int j = threadIdx.x; j < e; j += kThreads)
            smem[p.sm_bias + j] = load_as_float(p.bias, DT, j);
    if (!kFixed && p.sm_extra >= 0)
        for (int j = threadIdx.x; j < e; j += kThreads)
            smem[p.sm_extra + j] = load_as_float(p.extra_bias, DT, j);
    __syncthreads();
    float *s_row = p.sm_rows >= 0 ? smem + p.sm_rows + warp * e : nullptr;
    uint32_t *s_gkey = p.sm_gkey >= 0 ? reinterpret_cast<uint32_t *>(smem) + p.sm_gkey + warp * p.group_count
                                      : nullptr;
    uint32_t *s_kept = p.sm_kept >= 0 ? reinterpret_cast<uint32_t *>(smem) + p.sm_kept + warp * 32 : nullptr;
    __shared__ uint2 s_pick_all[kWarps][64];   // each warp's picks of its current row
    uint2 *s_pick = s_pick_all[warp];

    // rank by logit: the inverted expert numbers of the lane's run, two per word
    uint32_t ip[(VPL + 1) / 2];
    if (kByLogit) {
        const uint32_t base = 0xffffu - (uint32_t)(lane * VPL);
#pragma unroll
        for (int c = 0; c < (VPL + 1) / 2; ++c)
            ip[c] = ((base - 2 * c - 1) << 16) | ((base - 2 * c) & 0xffffu);
    }

    // rank by logit: the warp's next row is loaded while it works on the current one (not at 32
    // experts per lane, where the 16 words held across the full-evaluation fallback would spill)
    constexpr int W = (VPL + 1) / 2;
    constexpr bool kAhead = kByLogit && DT != MRR_GATE_F32 && VPL < 32;
    const int stride = gridDim.x * kWarps;
    uint32_t w_next[W];
    if (kAhead && blockIdx.x * kWarps + warp < p.T)
        load_words<VPL>(w_next, p.x, blockIdx.x * kWarps + warp, MRR_GATE_ROW_SHAPE, j0, nv);

    uint32_t flags = 0u;
    for (int t = blockIdx.x * kWarps + warp; t < p.T; t += stride) {
        float y0 = 0.f, y1 = 0.f;
        uint32_t i0 = 0u, i1 = 0u;
        bool done = false;
        if constexpr (kByLogit && DT == MRR_GATE_F32) {
            done = logit_ranked_row_f32<VPL, kFixedLogit ? kK : 0>(p, t, lane, j0, nv, s_pick, y0, i0);
        } else if constexpr (kByLogit) {
            uint32_t w[W];
            if (kAhead) {
#pragma unroll
                for (int c = 0; c < W; ++c)
                    w[c] = w_next[c];
                if (t + stride < p.T)
                    load_words<VPL>(w_next, p.x, t + stride, MRR_GATE_ROW_SHAPE, j0, nv);
            } else {
                load_words<VPL>(w, p.x, t, MRR_GATE_ROW_SHAPE, j0, nv);
            }
            done = logit_ranked_row<VPL, DT, kFixedLogit ? kK : 0>(p, t, lane, nv, w, ip, y0, i0);
        }
        if (!done)
            full_row<VPL, DT, kFixed>(p, t, lane, j0, nv, smem, s_row, s_gkey, s_kept, s_pick, flags, y0, i0, y1,
                                      i1);

        // ---- step 4: scale and write
        const bool has0 = lane < k, has1 = lane + 32 < k;
        const float y_lane = (has0 ? y0 : 0.f) + (has1 ? y1 : 0.f);
        const float ysum = (kFixed || kFixedLogit) ? warp_sum_low<pow2_at_least(kFixed ? kFixedK : kK)>(y_lane)
                                                   : warp_sum(y_lane);
        const float scale = p.rsf * __frcp_rn(ysum + p.eps);
        if (has0) {
            store_from_float(p.y_out, DT, (long long)t * k + lane, y0 * scale);
            p.expert_idx[(long long)t * k + lane] = (int)i0;
        }
        if (has1) {
            store_from_float(p.y_out, DT, (long long)t * k + lane + 32, y1 * scale);
            p.expert_idx[(long long)t * k + lane + 32] = (int)i1;
        }
    }
    // per-CTA status word (plain stores: no clearing needed between calls)
    flags = __reduce_or_sync(kFull, flags);
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
#undef MRR_GATE_ROW_SHAPE
}

template <int VPL, int DT, int kPath, int kK = 0>
inline cudaError_t launch_gating_dt(const Params &p, size_t smem, int sms, cudaStream_t stream)
{
    const auto kernel = gating_kernel<VPL, DT, kPath, kK>;
    if (smem > 48 * 1024) {
        const cudaError_t err =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptIn);
        if (err != cudaSuccess)
            return err;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t want = ((int64_t)p.T + kWarps - 1) / kWarps;
    int64_t cap = (int64_t)sms * per_sm;
    if (cap > kMaxGrid)
        cap = kMaxGrid;
    const int grid = (int)(want < 1 ? 1 : (want > cap ? cap : want));
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// The fixed-shape rank-by-logit instances: e = 32 * VPL for VPL in {4, 8, 12, 16} (128 to 512
// experts) and k in {2, 4, 6, 8}.
template <int VPL, int DT>
inline cudaError_t launch_logit_fixed(const Params &p, size_t smem, int sms, cudaStream_t stream)
{
    switch (p.k) {
    case 2:
        return launch_gating_dt<VPL, DT, kPathLogitFixed, 2>(p, smem, sms, stream);
    case 4:
        return launch_gating_dt<VPL, DT, kPathLogitFixed, 4>(p, smem, sms, stream);
    case 6:
        return launch_gating_dt<VPL, DT, kPathLogitFixed, 6>(p, smem, sms, stream);
    default:
        return launch_gating_dt<VPL, DT, kPathLogitFixed, 8>(p, smem, sms, stream);
    }
}

// one dtype's launch: the VPL template instance for the row width and the kernel path.  The
// grouped sigmoid and the fixed-shape rank-by-logit instances exist for 4, 8, 12 and 16 experts
// per lane (e = 128, 256, 384, 512).
template <int DT>
inline cudaError_t launch_dtype(const Params &p, int vpl, int path, size_t smem, int sms, cudaStream_t stream)
{
#define MRR_GATE_CASE(V)                                                                       \
    case V:                                                                                    \
        return path == kPathLogit ? launch_gating_dt<V, DT, kPathLogit>(p, smem, sms, stream)  \
                                  : launch_gating_dt<V, DT, kPathFull>(p, smem, sms, stream);
#define MRR_GATE_CASE_FIXED(V)                                                                 \
    case V:                                                                                    \
        if (path == kPathGroupedSigmoid)                                                       \
            return launch_gating_dt<V, DT, kPathGroupedSigmoid>(p, smem, sms, stream);         \
        if (path == kPathLogitFixed)                                                           \
            return launch_logit_fixed<V, DT>(p, smem, sms, stream);                            \
        return path == kPathLogit ? launch_gating_dt<V, DT, kPathLogit>(p, smem, sms, stream)  \
                                  : launch_gating_dt<V, DT, kPathFull>(p, smem, sms, stream);
    switch (vpl) {
        MRR_GATE_CASE(1)
        MRR_GATE_CASE(2)
        MRR_GATE_CASE_FIXED(4)
        MRR_GATE_CASE(6)
        MRR_GATE_CASE_FIXED(8)
        MRR_GATE_CASE_FIXED(12)
        MRR_GATE_CASE_FIXED(16)
        MRR_GATE_CASE(24)
    default:
        break;
    }
    return path == kPathLogit ? launch_gating_dt<32, DT, kPathLogit>(p, smem, sms, stream)
                              : launch_gating_dt<32, DT, kPathFull>(p, smem, sms, stream);
#undef MRR_GATE_CASE
#undef MRR_GATE_CASE_FIXED
}

// defined in gating_f16.cu, gating_bf16.cu and gating_f32.cu
cudaError_t launch_f16(const Params &p, int vpl, int path, size_t smem, int sms, cudaStream_t stream);
cudaError_t launch_bf16(const Params &p, int vpl, int path, size_t smem, int sms, cudaStream_t stream);
cudaError_t launch_f32(const Params &p, int vpl, int path, size_t smem, int sms, cudaStream_t stream);

}  // namespace mrr_gate
