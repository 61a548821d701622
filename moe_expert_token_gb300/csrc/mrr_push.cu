// The push form of the fused receive, one sender's side (mrr_v2_push in include/mrr_v2.h).
//
// What it computes ("CANN ops-transformer MoeReRoutingV2" article, section 计算公式): receiver r
// lays out the rows it receives expert-major, row k of segment (i, j) at DstOffset_r(i, j) + k.
// Here sender i writes its own segments there directly.  Its rows for receiver r's local expert j
// form segment (r, j) of its send buffer, at SendOffset(r, j) = the row-major exclusive prefix of
// its send counts; the receiver's DstOffset_r(i, j) (and SrcOffset_r(i, j), for the gather index)
// arrive from the counts exchange.
//
// GB300 design: a warp takes about 8 KB of consecutive source rows at a time and moves each
// segment's share of them as one byte range, 16 bytes per lane per access where the pointers and
// sizes allow (else 8, 4 or 1), four accesses in flight per lane, with plain loads and stores --
// a receiver's buffer may be a peer GPU's memory, which the bulk copy engine is not used for.
// Every CTA scans the send counts into shared memory (at most 4096 segments) and finds a chunk's
// first segment by a binary search there.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "mrr_shape.h"
#include "mrr_v2.h"
#include "ptx.cuh"
#include "ws_layout.h"

namespace mrr_push {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSegments = 4096;  // R * E
constexpr int64_t kChunkBytes = 8192;   // token bytes a warp takes at a time (at least one row)
constexpr int kMaxGrid = mrr_ws::kStatusWords - 2;
constexpr uint32_t kFull = 0xffffffffu;

struct Payload {
    const uint8_t *src;   // this sender's rows, or null when the payload is absent
    uint8_t *const *out;  // [R] receiver buffers
    int64_t rb;           // bytes per row
};

struct Params {
    Payload tok, sc, tk;
    const void *counts;
    int count_is_i64;
    int R, E, RE;
    int64_t S;
    const int64_t *dst_off;   // [R * E]
    const int64_t *rsrc_off;  // [R * E] or null
    int32_t *const *idx_out;  // [R] or null
    const int64_t *out_rows;  // [R] or null
    uint32_t *status;
};

__device__ __forceinline__ int64_t count_at(const Params &p, int k)
{
    return p.count_is_i64 ? __ldg(static_cast<const long long *>(p.counts) + k)
                          : (int64_t)__ldg(static_cast<const int *>(p.counts) + k);
}

// Lane `lane` of a warp moves its share of `bytes` contiguous bytes, in the widest accesses the
// two addresses and the size allow.
__device__ __forceinline__ void copy_range(uint8_t *dst, const uint8_t *src, int64_t bytes, int lane)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | (uintptr_t)bytes;
    if ((a & 15u) == 0) {
        // four 16-byte loads in flight per lane before their stores
        constexpr int64_t kStep = 32 * 16;
        int64_t i = (int64_t)lane * 16;
        for (; i + 3 * kStep < bytes; i += 4 * kStep) {
            uint4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                q[u] = __ldg(reinterpret_cast<const uint4 *>(src + i + u * kStep));
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4 *>(dst + i + u * kStep) = q[u];
        }
        for (; i < bytes; i += kStep)
            *reinterpret_cast<uint4 *>(dst + i) = __ldg(reinterpret_cast<const uint4 *>(src + i));
    } else if ((a & 7u) == 0) {
        for (int64_t i = (int64_t)lane * 8; i < bytes; i += 32 * 8)
            *reinterpret_cast<uint2 *>(dst + i) = __ldg(reinterpret_cast<const uint2 *>(src + i));
    } else if ((a & 3u) == 0) {
        for (int64_t i = (int64_t)lane * 4; i < bytes; i += 32 * 4)
            *reinterpret_cast<uint32_t *>(dst + i) = __ldg(reinterpret_cast<const uint32_t *>(src + i));
    } else {
        for (int64_t i = lane; i < bytes; i += 32)
            dst[i] = __ldg(src + i);
    }
}

// Exclusive block-wide prefix of one int64 per thread; *total receives the block's sum.
__device__ __forceinline__ int64_t block_exscan64(int64_t v, int64_t *s_warp, int64_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < kWarps ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            const int64_t y = __shfl_up_sync(kFull, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < kWarps)
            s_warp[lane] = w;  // inclusive prefix of the warp sums
    }
    __syncthreads();
    *total = s_warp[kWarps - 1];
    return (warp ? s_warp[warp - 1] : 0) + x - v;
}

__global__ void __launch_bounds__(kThreads, 3) push_kernel(const Params p)
{
    __shared__ int64_t s_off[kMaxSegments + 1];  // SendOffset(g), g = r * E + j; s_off[RE] = S
    __shared__ int64_t s_warp[kWarps];
    __shared__ uint32_t s_flags;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // the counts and the tables may come from the previous kernel on the stream
    mrr::grid_dependency_wait();
    mrr::grid_launch_dependents();
    if (tid == 0)
        s_flags = 0u;

    // ---- SendOffset: thread t scans the segments [k0, k1)
    const int per = (p.RE + kThreads - 1) / kThreads;
    const int k0 = min(p.RE, tid * per), k1 = min(p.RE, k0 + per);
    uint32_t f = 0u;
    int64_t local = 0;
    for (int k = k0; k < k1; ++k) {
        const int64_t c = count_at(p, k);
        if (c <= 0)
            f |= mrr_ws::kFlagNonPos;
        else if (c > p.S)
            f |= mrr_ws::kFlagSum;
        else
            local += c;
    }
    int64_t total;
    int64_t run = block_exscan64(local, s_warp, &total);
    for (int k = k0; k < k1; ++k) {
        s_off[k] = run;
        const int64_t c = count_at(p, k);
        run += (c > 0 && c <= p.S) ? c : 0;
    }
    if (tid == 0)
        s_off[p.RE] = total;
    if (f)
        atomicOr(&s_flags, f);
    __syncthreads();
    uint32_t flags = s_flags;
    if (!flags && total != p.S)
        flags = mrr_ws::kFlagSum;

    // ---- the rows, in chunks of consecutive source rows (about 8 KB of tokens each): warp w of
    // CTA b takes chunk b * kWarps + w, then every gridDim.x * kWarps-th.  Inside a chunk the rows
    // of one segment are consecutive on both sides, so each such piece moves as one byte range.
    uint32_t dflag = 0u;
    if (!flags) {
        const int64_t rpc = p.tok.rb < kChunkBytes ? kChunkBytes / p.tok.rb : 1;  // rows per chunk
        const int64_t nchunks = (p.S + rpc - 1) / rpc;
        const int64_t step = (int64_t)gridDim.x * kWarps;
        for (int64_t c = (int64_t)blockIdx.x * kWarps + warp; c < nchunks; c += step) {
            int64_t s = c * rpc;
            const int64_t s_end = min(p.S, s + rpc);
            // the segment holding row s: the last g with SendOffset(g) <= s (counts > 0, so the
            // offsets strictly increase)
            int lo = 0, hi = p.RE;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= s)
                    lo = mid;
                else
                    hi = mid;
            }
            for (int g = lo; s < s_end; ++g) {
                const int64_t n = min(s_end, s_off[g + 1]) - s;  // rows of segment g in this chunk
                const int r = g / p.E;
                const int64_t k = s - s_off[g];
                const int64_t d = __ldg(p.dst_off + g) + k;
                uint8_t *const to = p.tok.out[r];
                uint8_t *const to_sc = p.sc.src ? p.sc.out[r] : nullptr;
                uint8_t *const to_tk = p.tk.src ? p.tk.out[r] : nullptr;
                int32_t *const to_idx = p.idx_out ? p.idx_out[r] : nullptr;
                // the rows of the piece that land inside receiver r's buffers
                int64_t m = n;
                if (!to || (p.sc.src && !to_sc) || (p.tk.src && !to_tk) || (p.idx_out && !to_idx) || d < 0)
                    m = 0;
                else if (p.out_rows)
                    m = max((int64_t)0, min(n, __ldg(p.out_rows + r) - d));
                if (m < n)
                    dflag = mrr_ws::kFlagDest;  // rows past the receiver's end are not written
                if (m > 0) {
                    copy_range(to + d * p.tok.rb, p.tok.src + s * p.tok.rb, m * p.tok.rb, lane);
                    if (p.sc.src)
                        copy_range(to_sc + d * p.sc.rb, p.sc.src + s * p.sc.rb, m * p.sc.rb, lane);
                    if (p.tk.src)
                        copy_range(to_tk + d * 4, p.tk.src + s * 4, m * 4, lane);
                    if (to_idx) {
                        const int64_t first = __ldg(p.rsrc_off + g) + k;
                        for (int64_t t = lane; t < m; t += 32)
                            to_idx[d + t] = (int32_t)(first + t);
                    }
                }
                s += n;
            }
        }
    }

    // ---- status: CTA b's flags in word 2 + b (plain stores: no clearing between calls)
    dflag = __reduce_or_sync(kFull, dflag);
    if (lane == 0 && dflag)
        atomicOr(&s_flags, dflag);
    __syncthreads();
    if (tid == 0) {
        p.status[2 + blockIdx.x] = flags | s_flags;
        if (blockIdx.x == 0) {
            p.status[0] = 0u;
            p.status[1] = gridDim.x;
        }
    }
}

}  // namespace mrr_push

extern "C" mrr_status mrr_v2_push(const void *send_tokens, const void *send_scales, const float *send_topk_w,
                                  mrr_token_dtype dt, int64_t S, int64_t H, const void *send_counts,
                                  int count_is_i64, int64_t R, int64_t E, mrr_scale_layout sl, int64_t scale_cols,
                                  const int64_t *dst_offsets, const int64_t *recv_src_offsets,
                                  void *const *out_tokens, void *const *out_scales, float *const *out_topk_w,
                                  int32_t *const *idx_out, const int64_t *out_rows, void *workspace,
                                  size_t workspace_bytes, mrr_stream_t stream_)
{
    using namespace mrr_push;
    int64_t rb = 0, sb = 0;
    const mrr_status st =
        mrr_host::check_shape(S, H, (int)dt, R, E, count_is_i64, (int)sl, scale_cols, 1, 0, &rb, &sb);
    if (st != MRR_OK)
        return st;
    if (R * E > kMaxSegments)
        return MRR_ERR_SHAPE;
    if (!workspace || workspace_bytes < (size_t)mrr_ws::kStatusBytes ||
        reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return MRR_ERR_WORKSPACE;
    if (!send_tokens || !send_counts || !dst_offsets || !out_tokens)
        return MRR_ERR_NULL;
    if ((sl != MRR_SCALE_NONE) != (send_scales != nullptr) || (send_scales != nullptr) != (out_scales != nullptr))
        return MRR_ERR_NULL;
    if ((send_topk_w != nullptr) != (out_topk_w != nullptr))
        return MRR_ERR_TOPK_PAIR;
    if ((idx_out != nullptr) != (recv_src_offsets != nullptr))
        return MRR_ERR_NULL;
    const uintptr_t ca = reinterpret_cast<uintptr_t>(send_counts);
    if (ca % (count_is_i64 ? 8 : 4) != 0 || reinterpret_cast<uintptr_t>(dst_offsets) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(recv_src_offsets) % 8 != 0 || reinterpret_cast<uintptr_t>(out_rows) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(send_topk_w) % 4 != 0)
        return MRR_ERR_ALIGN;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (S == 0) {  // the empty problem: a clean status, nothing to move
        if (cudaMemsetAsync(workspace, 0, 8, stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return MRR_ERR_CUDA;
        }
        return MRR_OK;
    }
    int device = -1, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    Params p;
    memset(&p, 0, sizeof(p));
    p.tok = {static_cast<const uint8_t *>(send_tokens), reinterpret_cast<uint8_t *const *>(out_tokens), rb};
    p.sc = {static_cast<const uint8_t *>(send_scales), reinterpret_cast<uint8_t *const *>(out_scales), sb};
    p.tk = {reinterpret_cast<const uint8_t *>(send_topk_w), reinterpret_cast<uint8_t *const *>(out_topk_w), 4};
    p.counts = send_counts;
    p.count_is_i64 = count_is_i64;
    p.R = (int)R;
    p.E = (int)E;
    p.RE = (int)(R * E);
    p.S = S;
    p.dst_off = dst_offsets;
    p.rsrc_off = recv_src_offsets;
    p.idx_out = idx_out;
    p.out_rows = out_rows;
    p.status = static_cast<uint32_t *>(workspace);
    // a warp per chunk of rows: enough CTAs to fill the SMs, never more than the rows need
    const int64_t want = (S + kWarps - 1) / kWarps;
    int64_t cap = (int64_t)sms * 3;  // three CTAs of 8 warps fit on an SM (80 registers)
    if (cap > kMaxGrid)
        cap = kMaxGrid;
    const int grid = (int)(want < cap ? want : cap);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, push_kernel, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    return MRR_OK;
}
