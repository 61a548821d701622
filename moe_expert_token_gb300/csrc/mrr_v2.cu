// GB300 (sm_103a) implementation of the MoeReRoutingV2 re-routing step behind the C ABI in
// include/mrr_v2.h.
//
// What the op computes ("CANN ops-transformer MoeReRoutingV2" article, section 计算公式):
// the count matrix counts[N,E] splits the A received rows into segments (rank i, expert j);
// segment (i,j) starts at SrcOffset(i,j) in the rank-major input (exclusive prefix of the
// counts in row-major order) and moves, order kept, to DstOffset(i,j) in the expert-major
// output (exclusive prefix in column-major order).  Token rows, scale rows and top-k weights
// share the offsets; the index output and the per-expert counts come from the same offsets.
//
// GB300 design (pure data movement, bound by HBM bandwidth; no tensor-core work exists):
//   * One kernel does everything for N*E <= 4096: each CTA scans the counts into shared
//     memory (row-major and column-major exclusive prefixes, warp-shuffle block scans) while
//     its first token chunks are already in flight, then streams its slice of the token bytes.
//   * Work is split by SOURCE bytes.  Source addresses need no offsets, so the bulk path issues
//     its first loads (and L2 prefetches of the next chunks) before the scan and hides the scan
//     behind them.  Inside a segment both sides are contiguous, so a range of source bytes maps
//     to a few contiguous runs ("pieces"), each copied as a whole.
//   * Bulk path (rows a multiple of 16 bytes): one thread per CTA drives the bulk-copy engine:
//     cp.async.bulk global->shared into a ring of `stages` chunks (completion on mbarriers),
//     then one cp.async.bulk shared->global per piece.  Each CTA takes a few static chunks,
//     then claims chunks from a counter in the workspace, so all CTAs finish together.  The
//     other warps move the scale rows, top-k weights and the index at the same time.
//   * Vector path (rows not a multiple of 16 bytes, or unaligned buffers): each warp walks the
//     pieces of its own sub-range; pieces whose source and destination alignments differ are
//     realigned in registers (funnel shifts) so that every access is 16 bytes wide.
//   * N*E > 4096: a one-CTA scan kernel writes the offsets into the workspace first; the copy
//     kernel stages them in shared memory when they fit beside its ring.
//   * Data-dependent errors (count <= 0, Sum != A) set flags in a status word in the
//     workspace; every CTA then skips its stores.  Every wait is bounded in time; a timeout
//     sets a flag, drains the copies in flight and returns (no trap, no assert).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <chrono>
#include <type_traits>

#include "mrr_shape.h"
#include "mrr_v2.h"
#include "ptx.cuh"
#include "ws_layout.h"

namespace mrr {

using mrr_ws::kHeaderBytes;   // status region + counter; offset tables follow
using mrr_ws::kStatusBytes;   // status region at the front of the workspace
using mrr_ws::kStatusWords;   // [0] flags, [1] grid, [2 + b] CTA b's flags
using mrr_ws::kTicketOffset;  // 8-byte shared chunk counter (dynamic scheduling)
using mrr_ws::padded_len;
constexpr int kMaxGrid = kStatusWords - 2;
constexpr int64_t kFusedMaxSegs = 4096;            // N*E scanned inside every CTA up to this
constexpr int64_t kSmemScanMaxSegs = 16384;        // above kFusedMaxSegs: the scan kernel scans in
                                                   // shared memory up to this (about 200 KB)
using mrr_ws::kFlagBadIndex;  // set by the gating kernel (gating.cu)
using mrr_ws::kFlagDest;      // set by the push form (mrr_push.cu)
using mrr_ws::kFlagNonPos;
using mrr_ws::kFlagSource;    // multi-source form: a per-rank pointer is null or misaligned
using mrr_ws::kFlagSum;
using mrr_ws::kFlagTimeout;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bound on any single mbarrier wait: 2 s
constexpr int kMaxStages = 8;

struct Params {
    const uint8_t *tokens;
    uint8_t *out_tokens;
    int64_t total_bytes;  // A * row_bytes
    int64_t row_bytes;
    int64_t A;
    const void *counts;
    int count_is_i64;
    int N, E, NE;
    const uint8_t *scales;
    uint8_t *out_scales;
    int64_t scale_row_bytes;
    int scale_w;          // vector width for scale rows (1..16)
    const uint8_t *topk;
    uint8_t *out_topk;
    int topk_w;           // vector width for the 4-byte weights (1..4)
    int32_t *idx;
    int idx_type;
    void *etn;
    uint32_t *status;
    uint32_t *g_row_ex;   // N*E > 4096: offsets scanned into the workspace
    uint32_t *g_dst_off;
    uint32_t *g_col_ex;   // N*E > 4096, inverse move: column-major prefix by position (padded)
    int inverse;          // 0: rank-major -> expert-major; 1: the inverse move (no index outputs)
    int etn_type;         // expert_token_num: 1 per-expert count, 0 inclusive cumsum over experts
    int chunk_bytes;
    int stages;
    int hints;            // bulk path: MRR_HINT_* bits (L2 evict-first policies)
    int sched;            // bulk path: 0 static slices, 1 static chunks then shared-counter chunks
    int static_chunks;    // bulk path, sched 1: chunks each CTA takes before using the counter
    int prefetch_chunks;  // bulk path: chunks each CTA asks L2 to prefetch during the scan
    int scan_in_smem;     // N*E > 4096: the scan kernel scans in smem (tables fit in one CTA)
    unsigned long long *ticket;  // sched 1: shared chunk counter in the workspace
    unsigned long long epoch;    // sched 1: this launch's tag for the counter (40 bits, nonzero)
    // multi-source form (forward move only): rank i's rows sit in their own buffers; tokens,
    // scales and topk above are then unused.  Each is a device array of N device pointers.
    int multi;
    int multi_bulk;                 // multi-source form on the bulk path (token sources 16-aligned)
    const uint8_t *const *src_tok;  // [N] rank i's token rows (16-byte aligned on the bulk path)
    const uint8_t *const *src_sc;   // [N] rank i's scale rows, or null without scales
    const uint8_t *const *src_tk;   // [N] rank i's top-k weights (any alignment), or null
    const long long *src_rows;      // [N] rows each rank's buffers hold, or null (not checked)
    int ptr_off;                    // byte offset of the pointer tables' copy in dynamic shared
                                    // memory (tokens, then scales, then top-k, then the rows), or
                                    // -1: read them from global memory
};

// The per-rank source tables the multi-source form reads: Params' global tables, or their copy in
// shared memory (the bulk driver looks one up whenever a load crosses into another rank).
struct Sources {
    const uint8_t *const *tok;
    const uint8_t *const *sc;
    const uint8_t *const *tk;
    const long long *rows;  // rows each rank's buffers hold, or null (not checked)
};

// ------------------------------------------------------------------------------------------------
// helpers

__device__ __forceinline__ int64_t load_count(const Params &p, int64_t k)
{
    if (p.count_is_i64)
        return (int64_t)__ldg(reinterpret_cast<const long long *>(p.counts) + k);
    return (int64_t)__ldg(reinterpret_cast<const int *>(p.counts) + k);
}

// Segment of source row s: the last q in [0, NE) with row_ex[q] <= s.  row_ex is strictly
// increasing (every count > 0) with row_ex[0] = 0 and row_ex[NE] = A.
__device__ __forceinline__ int find_seg(const uint32_t *row_ex, int NE, uint32_t s)
{
    int lo = 0, hi = NE;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (row_ex[mid] <= s)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Shared-memory index with one padding word per 32: walks with a stride that is a multiple of
// 32 words (a column of the count matrix) then spread over the banks instead of hitting one.
__device__ __forceinline__ int pad32(int k) { return k + (k >> 5); }

// The segments of one direction of the move, numbered in the order they sit in the SOURCE.
//   forward (rank-major -> expert-major): g = q = i*E + j; starts = SrcOffset (row_ex, dense),
//     destinations = DstOffset (dst_off, padded by q);
//   inverse (expert-major -> rank-major): g = pos = j*N + i; starts = DstOffset by position
//     (col_ex, padded), destinations = SrcOffset of (i, j).
// starts[NE] (at its index) is A.
struct SegMap {
    const uint32_t *row_ex;
    const uint32_t *dst_off;
    const uint32_t *col_ex;
    int NE, N, E;
    int inv;
    __device__ __forceinline__ uint32_t begin(int g) const { return inv ? col_ex[pad32(g)] : row_ex[g]; }
    // forward: DstOffset of segment g; inverse: SrcOffset of the segment at position g (the scan
    // stores it by position, so neither direction divides here)
    __device__ __forceinline__ uint32_t dest(int g) const { return dst_off[pad32(g)]; }
    // the last g with begin(g) * rb <= x: the segment holding source byte x, without a 64-bit
    // division (measured on GB300: 0.3 us less per launch at 4096 segments, neutral at 256)
    __device__ __forceinline__ int find_byte(int64_t x, int64_t rb) const
    {
        int lo = 0, hi = NE;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)begin(mid) * rb <= x)
                lo = mid;
            else
                hi = mid;
        }
        return lo;
    }
    // the last g in [0, NE) with begin(g) <= s (starts strictly increase: every count > 0)
    __device__ __forceinline__ int find(uint32_t s) const
    {
        if (!inv)
            return find_seg(row_ex, NE, s);
        int lo = 0, hi = NE;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (col_ex[pad32(mid)] <= s)
                lo = mid;
            else
                hi = mid;
        }
        return lo;
    }
};

// Destination row of source row s.
__device__ __forceinline__ int64_t dst_row(const SegMap &m, int64_t s)
{
    const int g = m.find((uint32_t)s);
    return (int64_t)m.dest(g) + (s - (int64_t)m.begin(g));
}

// Multi-source form (forward map only): the rows of rank i are rows [R(i), R(i+1)) of the
// rank-major order, R(i) = SrcOffset(i, 0) = row_ex[i*E], R(N) = A; they sit in rank i's own
// buffer from its start.  For source row s: its destination row, its rank and its row in that
// rank's buffer.
__device__ __forceinline__ int64_t dst_row_rank(const SegMap &m, int64_t s, int *rank, int64_t *local)
{
    const int g = m.find((uint32_t)s);
    const int i = g / m.E;
    *rank = i;
    *local = s - (int64_t)m.row_ex[i * m.E];
    return (int64_t)m.dest(g) + (s - (int64_t)m.begin(g));
}

// Multi-source form: the rank whose rows hold source byte x, the last i with R(i) * rb <= x
// (a binary search over the N rank starts, with no division).
__device__ __forceinline__ int rank_of_byte(const SegMap &m, int64_t x, int64_t rb)
{
    int lo = 0, hi = m.N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)m.row_ex[mid * m.E] * rb <= x)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Every rank's pointers checked by threads t0, t0 + ts, ...: tokens present and, on the bulk path,
// 16-byte aligned (the bulk copy engine's rule); scales and top-k weights present when they are
// moved (any alignment: their copies fall back to narrower accesses).  Returns kFlagSource or 0
// for this thread's share.
__device__ __forceinline__ uint32_t check_sources(const Params &p, const Sources &src, bool bulk, int t0, int ts)
{
    uint32_t f = 0u;
    for (int i = t0; i < p.N; i += ts) {
        const uintptr_t t = (uintptr_t)src.tok[i];
        if (!t || (bulk && (t & 15u)))
            f = kFlagSource;
        if (src.sc && !src.sc[i])
            f = kFlagSource;
        if (src.tk && !src.tk[i])
            f = kFlagSource;
    }
    return f;
}

// Multi-source form with capacities: rank i's rows, R(i+1) - R(i) from the scanned SrcOffset
// table, must fit the rows its buffers hold.  Threads t0, t0 + ts, ...; kFlagSource or 0.
__device__ __forceinline__ uint32_t check_capacity(const Params &p, const Sources &src, const uint32_t *row_ex,
                                                   int t0, int ts)
{
    uint32_t f = 0u;
    if (src.rows)
        for (int i = t0; i < p.N; i += ts)
            if ((long long)(row_ex[(i + 1) * p.E] - row_ex[i * p.E]) > src.rows[i])
                f = kFlagSource;
    return f;
}

// Multi-source form: warm L2 with what a launch reads first -- the counts and the per-rank
// tables -- before the programmatic dependency wait, so that their first touch (DRAM and address
// translation) overlaps the previous kernel's tail; the token stream waits on them.  Only L2 is
// asked: the loads that use the values come after the wait, and L2 holds whatever the previous
// kernel writes meanwhile.  (The single-source kernels start their token stream without the
// counts; there the same prefetch measured 0.1-0.5 us slower on C2-C5.)  Threads t0, t0 + ts, ...
__device__ __forceinline__ void prefetch_inputs_l2(const Params &p, int t0, int ts)
{
    const uint8_t *c = static_cast<const uint8_t *>(p.counts);
    const int64_t cb = (int64_t)p.NE * (p.count_is_i64 ? 8 : 4);
    const int64_t first = -(int64_t)(reinterpret_cast<uintptr_t>(c) & 127u);
    for (int64_t off = first + (int64_t)t0 * 128; off < cb; off += (int64_t)ts * 128)
        prefetch_line_l2(c + off);
    if (p.multi) {
        const void *tabs[4] = {p.src_tok, p.src_sc, p.src_tk, p.src_rows};
        const int64_t tb = (int64_t)p.N * 8;
        for (int t = 0; t < 4; ++t)
            if (tabs[t])
                for (int64_t off = (int64_t)t0 * 128; off < tb; off += (int64_t)ts * 128)
                    prefetch_line_l2(static_cast<const uint8_t *>(tabs[t]) + off);
    }
}

// Exclusive block-wide scan of one uint32 per thread (warp shuffles + one smem pass).
// Every thread of the block must call it.  *total receives the block sum.
__device__ __forceinline__ uint32_t block_exscan(uint32_t v, uint32_t *total, uint32_t *s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (blockDim.x + 31) >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < nwarps ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        s_warp[lane] = w;  // inclusive prefix of the warp totals
    }
    __syncthreads();
    const uint32_t base = warp ? s_warp[warp - 1] : 0u;
    *total = s_warp[nwarps - 1];
    __syncthreads();  // s_warp is reused by the next call
    return base + x - v;
}

// Exclusive scan over positions 0..n-1 of the block, read through in(k); out(k, prefix) receives
// each exclusive prefix, in increasing k for each thread.  Warp w owns a contiguous span; inside
// it each lane scans a run of kScanRun consecutive positions on its own, so one warp-shuffle
// scan serves 32 * kScanRun positions.  Every thread of the block must call it.
constexpr int kScanRun = 8;
template <class In, class Out>
__device__ __forceinline__ void block_scan_runs(int n, uint32_t *s_warp, In in, Out out)
{
    constexpr int kTile = 32 * kScanRun;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (blockDim.x + 31) >> 5;
    const int span = ((n + nwarps - 1) / nwarps + kTile - 1) / kTile * kTile;
    const int lo = min(n, warp * span), hi = min(n, lo + span);
    uint32_t wsum = 0u;
    for (int k = lo + lane; k < hi; k += 32)
        wsum += in(k);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    uint32_t total;
    uint32_t run = block_exscan(lane == 0 ? wsum : 0u, &total, s_warp);  // lane 0 carries the warp
    run = __shfl_sync(0xffffffffu, run, 0);
    for (int t = lo; t < hi; t += kTile) {
        const int k0 = t + lane * kScanRun;
        uint32_t x[kScanRun];
        uint32_t local = 0u;
#pragma unroll
        for (int e = 0; e < kScanRun; ++e) {
            x[e] = (k0 + e < hi) ? in(k0 + e) : 0u;
            local += x[e];
        }
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        uint32_t ex = run + incl - local;
#pragma unroll
        for (int e = 0; e < kScanRun; ++e) {
            if (k0 + e < hi)
                out(k0 + e, ex);
            ex += x[e];
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// The counts are loaded in batches: each thread has up to kCountBatch 16-byte vectors (4 int32
// or 2 int64 counts each) in flight at once.  The first batch is issued before the token stream
// starts, so these few loads do not queue behind it.
constexpr int kCountBatch = 4;
struct CountBatch {
    uint4 raw[kCountBatch];
};

template <typename CT>
__device__ __forceinline__ void issue_count_loads(const Params &p, int base, CountBatch &cb)
{
    constexpr int kPer = 16 / sizeof(CT);
    const int tid = threadIdx.x, nthr = blockDim.x, NE = p.NE;
    const CT *src = reinterpret_cast<const CT *>(p.counts);
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
#pragma unroll
    for (int b = 0; b < kCountBatch; ++b) {
        const int k0 = base + (b * nthr + tid) * kPer;
        if (vec && k0 + kPer <= NE) {
            cb.raw[b] = __ldg(reinterpret_cast<const uint4 *>(src + k0));
        } else {
            CT v[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                v[e] = (k0 + e < NE) ? __ldg(src + k0 + e) : CT(1);
            memcpy(&cb.raw[b], v, 16);
        }
    }
}

// Validate one batch and store each count twice: row-major at row_ex[q] (scanned in place
// later) and column-major at cnt_t[pad32(j*N + i)].  Returns error flags; adds valid counts.
template <typename CT>
__device__ __forceinline__ uint32_t process_counts(const Params &p, int base, const CountBatch &cb,
                                                   uint32_t *row_ex, uint32_t *cnt_t, unsigned long long *sum)
{
    constexpr int kPer = 16 / sizeof(CT);
    const int tid = threadIdx.x, nthr = blockDim.x, NE = p.NE, N = p.N, E = p.E;
    uint32_t f = 0u;
#pragma unroll
    for (int b = 0; b < kCountBatch; ++b) {
        const int k0 = base + (b * nthr + tid) * kPer;
        CT v[kPer];
        memcpy(v, &cb.raw[b], 16);
        int i = k0 / E, j = k0 - (k0 / E) * E;  // k0 = i*E + j
#pragma unroll
        for (int e = 0; e < kPer; ++e, ++j) {
            if (j == E) {
                j = 0;
                ++i;
            }
            const int k = k0 + e;
            if (k >= NE)
                break;
            const int64_t c = (int64_t)v[e];
            uint32_t u32 = 0u;
            if (c <= 0)
                f |= kFlagNonPos;
            else if (c > p.A)
                f |= kFlagSum;
            else {
                u32 = (uint32_t)c;
                *sum += (unsigned long long)c;
            }
            row_ex[k] = u32;
            cnt_t[pad32(j * N + i)] = u32;
        }
    }
    return f;
}

// Validate the counts (first batch already issued into `cb`), then build both prefixes in shared
// memory:
//   row_ex[q]          = SrcOffset of segment q = i*E + j (row-major walk), row_ex[NE] = A
//   dst_off[pad32(q)]  = DstOffset of segment q (column-major walk: expert outer, rank inner)
// *s_flags and *s_sum must be zero before the call.  Returns the error flags (uniform over the
// block); the tables are valid when it returns 0.
struct NoMid {
    __device__ void operator()() const {}
};

// `mid` (when given) is called by every thread once SrcOffset is complete and visible to the
// block, before DstOffset is scanned: the multi-source form starts its token stream there.
template <class Mid = NoMid>
__device__ uint32_t cta_scan(const Params &p, CountBatch &cb, uint32_t *row_ex, uint32_t *cnt_t,
                             uint32_t *dst_off, uint32_t *s_warp, uint32_t *s_flags, unsigned long long *s_sum,
                             Mid mid = Mid())
{
    const int tid = threadIdx.x, lane = tid & 31, nthr = blockDim.x;
    const int NE = p.NE, N = p.N, E = p.E;
    const int stride = nthr * (p.count_is_i64 ? 2 : 4) * kCountBatch;
    __syncthreads();  // *s_flags / *s_sum zeroed
    unsigned long long sum = 0ull;
    uint32_t f = 0u;
    for (int base = 0; base < NE; base += stride) {
        if (p.count_is_i64) {
            if (base)
                issue_count_loads<long long>(p, base, cb);
            f |= process_counts<long long>(p, base, cb, row_ex, cnt_t, &sum);
        } else {
            if (base)
                issue_count_loads<int>(p, base, cb);
            f |= process_counts<int>(p, base, cb, row_ex, cnt_t, &sum);
        }
    }
    f = __reduce_or_sync(0xffffffffu, f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_down_sync(0xffffffffu, sum, o);
    if (lane == 0) {
        if (f)
            atomicOr(s_flags, f);
        if (sum)
            atomicAdd(s_sum, sum);
    }
    __syncthreads();
    uint32_t flags = *s_flags;
    if (!flags && *s_sum != (unsigned long long)p.A)
        flags |= kFlagSum;
    if (flags)
        return flags;  // uniform: every thread read the same smem values

    // SrcOffset: row-major exclusive prefix, in place (each element is read before it is written)
    block_scan_runs(
        NE, s_warp, [&](int k) { return row_ex[k]; }, [&](int k, uint32_t v) { row_ex[k] = v; });
    if (tid == 0)
        row_ex[NE] = (uint32_t)p.A;
    if constexpr (!std::is_same<Mid, NoMid>::value) {
        __syncthreads();
        mid();
    }
    // DstOffset: exclusive prefix over the column-major copy, stored at pad32(q), q = i*E + j.
    // Each thread's positions come in increasing runs, so (i, j) of pos = j*N + i is stepped.
    int ci = -1, cj = 0, cpos = -2;
    block_scan_runs(
        NE, s_warp, [&](int pos) { return cnt_t[pad32(pos)]; },
        [&](int pos, uint32_t v) {
            if (pos == cpos + 1) {
                if (++ci == N) {
                    ci = 0;
                    ++cj;
                }
            } else {
                cj = pos / N;
                ci = pos - cj * N;
            }
            cpos = pos;
            if (p.inverse) {
                cnt_t[pad32(pos)] = v;                       // in place: the inverse move's source starts
                dst_off[pad32(pos)] = row_ex[ci * E + cj];   // and its destinations, by position
            } else {
                dst_off[pad32(ci * E + cj)] = v;
            }
        });
    if (p.inverse && tid == 0)
        cnt_t[pad32(NE)] = (uint32_t)p.A;
    __syncthreads();
    return 0u;
}

// expert_token_num[j], count mode  = size of expert j's block in the destination
//                                  = DstOffset(0, j+1) - DstOffset(0, j)   (A for the last one)
//                     cumsum mode = end of expert j's block = DstOffset(0, j+1) (inclusive)
__device__ __forceinline__ void write_expert_token_num(const Params &p, const uint32_t *dst_off, int t0,
                                                       int ts)
{
    for (int j = t0; j < p.E; j += ts) {
        const uint32_t next = (j + 1 < p.E) ? dst_off[pad32(j + 1)] : (uint32_t)p.A;
        const uint32_t v = p.etn_type == 0 ? next : next - dst_off[pad32(j)];
        if (p.count_is_i64)
            reinterpret_cast<long long *>(p.etn)[j] = (long long)v;
        else
            reinterpret_cast<int *>(p.etn)[j] = (int)v;
    }
}

__device__ __forceinline__ void copy_unit(uint8_t *d, const uint8_t *s, int w)
{
    switch (w) {
    case 16:
        *reinterpret_cast<uint4 *>(d) = __ldg(reinterpret_cast<const uint4 *>(s));
        break;
    case 8:
        *reinterpret_cast<uint2 *>(d) = __ldg(reinterpret_cast<const uint2 *>(s));
        break;
    case 4:
        *reinterpret_cast<uint32_t *>(d) = __ldg(reinterpret_cast<const uint32_t *>(s));
        break;
    case 2:
        *reinterpret_cast<uint16_t *>(d) = __ldg(reinterpret_cast<const uint16_t *>(s));
        break;
    default:
        *d = __ldg(s);
        break;
    }
}

template <int W>
struct Vec;
template <>
struct Vec<16> {
    static __device__ __forceinline__ uint4 ld(const uint8_t *p) { return ld_stream_v4(p); }
    static __device__ __forceinline__ void st(uint8_t *p, uint4 v) { st_v4(p, v); }
    using T = uint4;
};
template <>
struct Vec<8> {
    static __device__ __forceinline__ uint2 ld(const uint8_t *p) { return __ldg(reinterpret_cast<const uint2 *>(p)); }
    static __device__ __forceinline__ void st(uint8_t *p, uint2 v) { *reinterpret_cast<uint2 *>(p) = v; }
    using T = uint2;
};
template <>
struct Vec<4> {
    static __device__ __forceinline__ uint32_t ld(const uint8_t *p) { return __ldg(reinterpret_cast<const uint32_t *>(p)); }
    static __device__ __forceinline__ void st(uint8_t *p, uint32_t v) { *reinterpret_cast<uint32_t *>(p) = v; }
    using T = uint32_t;
};
template <>
struct Vec<2> {
    static __device__ __forceinline__ uint16_t ld(const uint8_t *p) { return __ldg(reinterpret_cast<const uint16_t *>(p)); }
    static __device__ __forceinline__ void st(uint8_t *p, uint16_t v) { *reinterpret_cast<uint16_t *>(p) = v; }
    using T = uint16_t;
};
template <>
struct Vec<1> {
    static __device__ __forceinline__ uint8_t ld(const uint8_t *p) { return __ldg(p); }
    static __device__ __forceinline__ void st(uint8_t *p, uint8_t v) { *p = v; }
    using T = uint8_t;
};

constexpr int kSideBatch = 4;  // rows (or scale vectors) per thread with their loads in flight

// W bytes from a source that may be less aligned than W (multi-source form: each rank's buffer has
// its own alignment), assembled from byte loads.
template <int W>
__device__ __forceinline__ typename Vec<W>::T ld_any(const uint8_t *p)
{
    if (((uintptr_t)p & (W - 1)) == 0)
        return Vec<W>::ld(p);
    uint8_t b[W];
#pragma unroll
    for (int i = 0; i < W; ++i)
        b[i] = __ldg(p + i);
    typename Vec<W>::T v;
    memcpy(&v, b, W);
    return v;
}

// w bytes (a power of two up to 16) with the widest unit both addresses allow.
__device__ __forceinline__ void copy_unit_any(uint8_t *d, const uint8_t *s, int w)
{
    int u = w;
    while (u > 1 && (((uintptr_t)d | (uintptr_t)s) & (uintptr_t)(u - 1)))
        u >>= 1;
    for (int k = 0; k < w; k += u)
        copy_unit(d + k, s + k, u);
}

// Scale vectors of width W (16, 8 or 4 bytes, both pointers aligned to W) for source rows
// [r_lo, r_hi): kSideBatch loads in flight per thread, then the stores.  Multi-source form: the
// source row is found in its rank's buffer, which may be less aligned than W.
template <int W, bool kMulti>
__device__ void move_scales(const Params &p, const SegMap &m, const Sources &src, int64_t r_lo, int64_t r_hi,
                            int t0, int ts)
{
    const int64_t sb = p.scale_row_bytes, vpr = sb / W;
    const int64_t items = (r_hi - r_lo) * vpr;
    for (int64_t t = t0; t < items; t += (int64_t)ts * kSideBatch) {
        typename Vec<W>::T v[kSideBatch];
        int64_t s[kSideBatch], off[kSideBatch], d[kSideBatch];
#pragma unroll
        for (int u = 0; u < kSideBatch; ++u) {
            const int64_t it = t + (int64_t)u * ts;
            if (it < items) {
                const int64_t r = it / vpr;
                s[u] = r_lo + r;
                off[u] = (it - r * vpr) * W;
                if constexpr (kMulti) {
                    int rk;
                    int64_t loc;
                    d[u] = dst_row_rank(m, s[u], &rk, &loc);
                    v[u] = ld_any<W>(src.sc[rk] + loc * sb + off[u]);
                } else {
                    v[u] = Vec<W>::ld(p.scales + s[u] * sb + off[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kSideBatch; ++u) {
            if (t + (int64_t)u * ts < items) {
                if constexpr (!kMulti)
                    d[u] = dst_row(m, s[u]);
                Vec<W>::st(p.out_scales + d[u] * sb + off[u], v[u]);
            }
        }
    }
}

// Scale rows, top-k weights and the index for this CTA's share of the SOURCE rows,
// processed by threads t0, t0 + ts, ... of the block.
template <bool kMulti>
__device__ void side_arrays(const Params &p, const SegMap &m, const Sources &src, int t0, int ts)
{
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t r_lo = b * p.A / G, r_hi = (b + 1) * p.A / G;
    const bool topk4 = kMulti ? src.tk && p.topk_w == 4 : p.topk && p.topk_w == 4;
    for (int64_t base = r_lo + t0; base < r_hi; base += (int64_t)ts * kSideBatch) {
        uint32_t w[kSideBatch];
        int64_t dd[kSideBatch], loc[kSideBatch];
        int rk[kSideBatch];
#pragma unroll
        for (int u = 0; u < kSideBatch; ++u) {
            const int64_t s = base + (int64_t)u * ts;
            if constexpr (kMulti) {
                if (s < r_hi) {
                    dd[u] = dst_row_rank(m, s, &rk[u], &loc[u]);
                    if (topk4) {
                        const uint8_t *a = src.tk[rk[u]] + loc[u] * 4;
                        w[u] = ((uintptr_t)a & 3u) ? ld_any<4>(a) : __ldg(reinterpret_cast<const uint32_t *>(a));
                    }
                }
            } else {
                if (topk4 && s < r_hi)
                    w[u] = __ldg(reinterpret_cast<const uint32_t *>(p.topk) + s);
            }
        }
#pragma unroll
        for (int u = 0; u < kSideBatch; ++u) {
            const int64_t s = base + (int64_t)u * ts;
            if (s >= r_hi)
                break;
            const int64_t d = kMulti ? dd[u] : dst_row(m, s);
            if (p.inverse) {
                // the inverse move writes no index
            } else if (p.idx_type == 0) {
                p.idx[d] = (int32_t)s;  // gather index: out[d] = in[idx[d]]
            } else {
                p.idx[s] = (int32_t)d;  // scatter index: out[idx[s]] = in[s]
            }
            if (topk4) {
                reinterpret_cast<uint32_t *>(p.out_topk)[d] = w[u];
            } else if constexpr (kMulti) {
                if (src.tk)
                    copy_unit_any(p.out_topk + d * 4, src.tk[rk[u]] + loc[u] * 4, 4);
            } else if (p.topk) {
                for (int k = 0; k < 4; k += p.topk_w)
                    copy_unit(p.out_topk + d * 4 + k, p.topk + s * 4 + k, p.topk_w);
            }
        }
    }
    if (kMulti ? !src.sc : !p.scales)
        return;
    switch (p.scale_w) {
    case 16:
        move_scales<16, kMulti>(p, m, src, r_lo, r_hi, t0, ts);
        break;
    case 8:
        move_scales<8, kMulti>(p, m, src, r_lo, r_hi, t0, ts);
        break;
    case 4:
        move_scales<4, kMulti>(p, m, src, r_lo, r_hi, t0, ts);
        break;
    default: {  // 1- or 2-byte aligned scale rows
        const int w = p.scale_w;
        const int64_t sb = p.scale_row_bytes, vpr = sb / w;
        const int64_t items = (r_hi - r_lo) * vpr;
        for (int64_t t = t0; t < items; t += ts) {
            const int64_t r = t / vpr;
            const int64_t v = t - r * vpr;
            const int64_t s = r_lo + r;
            if constexpr (kMulti) {
                int rk1;
                int64_t loc1;
                const int64_t d = dst_row_rank(m, s, &rk1, &loc1);
                copy_unit_any(p.out_scales + d * sb + v * w, src.sc[rk1] + loc1 * sb + v * w, w);
            } else {
                const int64_t d = dst_row(m, s);
                copy_unit(p.out_scales + d * sb + v * w, p.scales + s * sb + v * w, w);
            }
        }
    }
    }
}

// ------------------------------------------------------------------------------------------------
// vector path: cooperative copy of one contiguous run

// dst and src are congruent modulo W: bytes up to dst's W boundary, W-wide body, byte tail
template <int W>
__device__ __forceinline__ void copy_run(uint8_t *dst, const uint8_t *src, int64_t len, int tid, int nthr)
{
    int64_t head = (int64_t)((W - ((uintptr_t)dst & (W - 1))) & (W - 1));
    if (head > len)
        head = len;
    for (int64_t i = tid; i < head; i += nthr)
        dst[i] = __ldg(src + i);
    const int64_t nv = (len - head) / W;
    uint8_t *d = dst + head;
    const uint8_t *s = src + head;
    constexpr int U = 4;
    int64_t i = tid;
    for (; i + (int64_t)(U - 1) * nthr < nv; i += (int64_t)U * nthr) {
        typename Vec<W>::T r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            r[u] = Vec<W>::ld(s + (i + (int64_t)u * nthr) * W);
#pragma unroll
        for (int u = 0; u < U; ++u)
            Vec<W>::st(d + (i + (int64_t)u * nthr) * W, r[u]);
    }
    for (; i < nv; i += nthr)
        Vec<W>::st(d + i * W, Vec<W>::ld(s + i * W));
    for (int64_t k = head + nv * W + tid; k < len; k += nthr)
        dst[k] = __ldg(src + k);
}

// Realigning copy of nv 16-byte vectors: output vector k (16-byte aligned, at d + 16k) is bytes
// [r, r + 16) of the 32 bytes at the aligned source blocks a0 + 16k and a0 + 16k + 16, where
// r = 4*Q + shift_bits/8 (1..15).  Each output word is a funnel shift of two source words.
template <int Q>
__device__ __forceinline__ void copy_shift_run(uint8_t *d, const uint8_t *a0, int64_t nv, uint32_t shift_bits,
                                               int tid, int nthr)
{
    constexpr int U = 2;
    int64_t k = tid;
    for (; k + (int64_t)(U - 1) * nthr < nv; k += (int64_t)U * nthr) {
        uint4 x[U], y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint8_t *src = a0 + (k + (int64_t)u * nthr) * 16;
            x[u] = __ldg(reinterpret_cast<const uint4 *>(src));
            y[u] = __ldg(reinterpret_cast<const uint4 *>(src + 16));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t w[8] = {x[u].x, x[u].y, x[u].z, x[u].w, y[u].x, y[u].y, y[u].z, y[u].w};
            uint4 o;
            o.x = __funnelshift_r(w[Q], w[Q + 1], shift_bits);
            o.y = __funnelshift_r(w[Q + 1], w[Q + 2], shift_bits);
            o.z = __funnelshift_r(w[Q + 2], w[Q + 3], shift_bits);
            o.w = __funnelshift_r(w[Q + 3], w[Q + 4], shift_bits);
            st_v4(d + (k + (int64_t)u * nthr) * 16, o);
        }
    }
    for (; k < nv; k += nthr) {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(a0 + k * 16));
        const uint4 y = __ldg(reinterpret_cast<const uint4 *>(a0 + k * 16 + 16));
        const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        uint4 o;
        o.x = __funnelshift_r(w[Q], w[Q + 1], shift_bits);
        o.y = __funnelshift_r(w[Q + 1], w[Q + 2], shift_bits);
        o.z = __funnelshift_r(w[Q + 2], w[Q + 3], shift_bits);
        o.w = __funnelshift_r(w[Q + 3], w[Q + 4], shift_bits);
        st_v4(d + k * 16, o);
    }
}

// Copy len bytes whose source and destination differ in alignment.  [buf_lo, buf_hi) is the whole
// source buffer: the aligned 16-byte source blocks read must lie inside it, so the realigned
// middle is clamped to its inner aligned part and everything else moves byte by byte.
__device__ __forceinline__ void copy_realign(uint8_t *dst, const uint8_t *src, int64_t len, const uint8_t *buf_lo,
                                             const uint8_t *buf_hi, int tid, int nthr)
{
    int64_t head = (int64_t)((16 - ((uintptr_t)dst & 15u)) & 15u);   // bytes until dst is aligned
    if (head > len)
        head = len;
    const uint8_t *s1 = src + head;
    const uint32_t r = (uint32_t)((uintptr_t)s1 & 15u);             // != 0: the alignments differ
    const uint8_t *a0 = s1 - r;                                      // aligned block holding s1
    int64_t nv = (len - head) / 16;
    // first and last source blocks read: a0 and a0 + 16 * nv (the second block of the last vector)
    const uintptr_t lo_ok = ((uintptr_t)buf_lo + 15u) & ~(uintptr_t)15u, hi_ok = (uintptr_t)buf_hi & ~(uintptr_t)15u;
    int64_t skip = 0;  // vectors at the front whose first block would start before the buffer
    if ((uintptr_t)a0 < lo_ok)
        skip = (int64_t)((lo_ok - (uintptr_t)a0 + 15u) / 16u);
    if (skip > nv)
        skip = nv;
    const int64_t fit = (int64_t)hi_ok >= (int64_t)((uintptr_t)a0 + 32u)
                            ? ((int64_t)hi_ok - (int64_t)(uintptr_t)a0 - 16) / 16 : 0;  // vectors k < fit read in bounds
    if (nv > fit)
        nv = fit > skip ? fit : skip;
    // bytes before the realigned middle (the head and any skipped vectors), one by one
    const int64_t mid0 = head + skip * 16, mid1 = head + nv * 16;
    for (int64_t i = tid; i < mid0; i += nthr)
        dst[i] = __ldg(src + i);
    uint8_t *d = dst + mid0;
    const uint8_t *b0 = a0 + skip * 16;
    const uint32_t sh = 8u * (r & 3u);
    switch (r >> 2) {
    case 0: copy_shift_run<0>(d, b0, nv - skip, sh, tid, nthr); break;
    case 1: copy_shift_run<1>(d, b0, nv - skip, sh, tid, nthr); break;
    case 2: copy_shift_run<2>(d, b0, nv - skip, sh, tid, nthr); break;
    default: copy_shift_run<3>(d, b0, nv - skip, sh, tid, nthr); break;
    }
    for (int64_t i = mid1 + tid; i < len; i += nthr)
        dst[i] = __ldg(src + i);
}

__device__ __forceinline__ void copy_block(uint8_t *dst, const uint8_t *src, int64_t len, const uint8_t *buf_lo,
                                           const uint8_t *buf_hi, int tid, int nthr)
{
    const uintptr_t mis = ((uintptr_t)dst ^ (uintptr_t)src) & 15u;
    if (mis == 0)
        copy_run<16>(dst, src, len, tid, nthr);
    else if ((mis & 7u) == 0)
        copy_run<8>(dst, src, len, tid, nthr);
    else if (len >= 256)
        copy_realign(dst, src, len, buf_lo, buf_hi, tid, nthr);
    else if ((mis & 3u) == 0)
        copy_run<4>(dst, src, len, tid, nthr);
    else if ((mis & 1u) == 0)
        copy_run<2>(dst, src, len, tid, nthr);
    else
        copy_run<1>(dst, src, len, tid, nthr);
}

// Walk the pieces of source byte range [lo, hi): each piece lies inside one segment, where the
// destination is the source shifted by (DstOffset - SrcOffset) rows.  Every warp takes its own
// contiguous sub-range (in 16-byte units), so a CTA has as many pieces in flight as it has warps:
// a run of small segments is not copied one latency-bound piece at a time.  Multi-source form:
// the piece is read from its rank's buffer (segment q belongs to rank q / E).
template <bool kMulti>
__device__ void vector_copy(const Params &p, const SegMap &m, const Sources &src, int64_t lo, int64_t hi, int tid,
                            int nthr)
{
    const int nwarps = nthr >> 5, warp = tid >> 5;
    const int64_t units = (hi - lo + 15) >> 4;
    const int64_t wlo = min(hi, lo + ((warp * units / nwarps) << 4));
    const int64_t whi = (warp == nwarps - 1) ? hi : min(hi, lo + (((warp + 1) * units / nwarps) << 4));
    lo = wlo;
    hi = whi;
    tid &= 31;
    nthr = 32;
    if (lo >= hi)
        return;
    const int64_t rb = p.row_bytes;
    int q = m.find((uint32_t)(lo / rb));
    int64_t seg_end = (int64_t)m.begin(q + 1) * rb;
    int64_t delta = ((int64_t)m.dest(q) - (int64_t)m.begin(q)) * rb;
    // multi-source: rank of segment q, the rank's first byte in rank-major order, its buffer
    int rank = kMulti ? q / m.E : 0;
    int64_t rank_b0 = 0, rank_b1 = p.total_bytes;
    const uint8_t *rank_buf = p.tokens;
    if constexpr (kMulti) {
        rank_b0 = (int64_t)m.row_ex[rank * m.E] * rb;
        rank_b1 = (int64_t)m.row_ex[(rank + 1) * m.E] * rb;
        rank_buf = src.tok[rank];
    }
    for (int64_t pos = lo; pos < hi;) {
        while (pos >= seg_end) {
            ++q;
            seg_end = (int64_t)m.begin(q + 1) * rb;
            delta = ((int64_t)m.dest(q) - (int64_t)m.begin(q)) * rb;
            if constexpr (kMulti) {
                if (q == (rank + 1) * m.E) {
                    ++rank;
                    rank_b0 = rank_b1;
                    rank_b1 = (int64_t)m.row_ex[(rank + 1) * m.E] * rb;
                    rank_buf = src.tok[rank];
                }
            }
        }
        const int64_t pe = min(hi, seg_end);
        copy_block(p.out_tokens + pos + delta, rank_buf + (pos - rank_b0), pe - pos, rank_buf,
                   rank_buf + (rank_b1 - rank_b0), tid, nthr);
        pos = pe;
    }
}

// ------------------------------------------------------------------------------------------------
// bulk path: one driver thread per CTA
//
// Chunks of chunk_bytes source bytes move through a ring of `stages` shared-memory buffers.
// Scheduling (plan.sched):
//   0  static: CTA b owns an equal 16-byte-aligned slice of the token bytes;
//   1  dynamic: CTA b first takes the static_chunks chunks starting at chunk b*static_chunks,
//      then claims further chunks from a counter shared by all CTAs, so CTAs whose memory
//      traffic drains faster take more chunks and all finish together.

constexpr int kTicketBits = 24;  // shared counter: [epoch of the launch | ticket (low 24 bits)]
constexpr unsigned long long kTicketMask = (1ull << kTicketBits) - 1;
constexpr uint32_t kNoTicket = 0xFFFFFFFFu;

// First claim of this launch on the shared counter, tagged with the host's launch epoch (a
// per-process random seed plus a launch count).  The counter holds the tag of an older launch, or
// anything in a fresh workspace; the first claimant installs (epoch, 1) with a compare-and-swap
// and takes ticket 0, later claimants see the epoch and add.
// A launch replayed from a CUDA graph keeps its parameters, epoch included, so it finds its own
// tag left by the previous replay.  Every launch draws exactly last_claim + 1 values (each CTA its
// tickets + 3), and a CTA's first claim comes before all its others, so a first claim can never
// see its own launch's final count: a counter that reads (epoch, last_claim + 1) was finished by
// an earlier run of this same launch and is installed afresh.  Bounded: kNoTicket on failure.
__device__ uint32_t claim_first_ticket(unsigned long long *ticket, unsigned long long epoch, int64_t last_claim)
{
    const unsigned long long finished = (epoch << kTicketBits) | (unsigned long long)(last_claim + 1);
    unsigned long long cur = atomicAdd(ticket, 0ull);
    for (int it = 0; it < (1 << 16); ++it) {
        if ((cur >> kTicketBits) == epoch && cur != finished)
            return (uint32_t)(atomicAdd(ticket, 1ull) & kTicketMask);
        const unsigned long long prev = atomicCAS(ticket, cur, (epoch << kTicketBits) | 1ull);
        if (prev == cur)
            return 0u;
        cur = prev;
    }
    return kNoTicket;
}

struct BulkRing {
    uint64_t *bars;
    uint8_t *base;
    int64_t *stage_b0, *stage_b1;  // shared memory: byte range held by each stage
    int64_t issued;                // chunk loads issued so far (sequence numbers 0 .. issued-1)
    uint64_t policy;               // L2 evict-first policy, used when hints ask for it
    int64_t next, hi;              // static part: next byte to load and the end of the range
    int64_t dyn_first;             // first chunk id served by tickets; -1 when none (left)
    int64_t nch;                   // chunks in the whole token buffer
    uint32_t pending[2];           // the next two tickets, claimed ahead of use
    bool started;                  // the first ticket has been taken
    int64_t last_claim;            // the launch's last ticket value: tickets + 3 * grid - 1
    int64_t tk_next, tk_end;       // chunk ids of the current ticket not yet served
    int per_ticket;                // consecutive chunks per ticket (about 64 KiB per claim)
    // multi-source form: the rank whose buffer the last load read, and its byte range in
    // rank-major order (consecutive chunks mostly come from one rank: one lookup per change)
    const uint8_t *src_base;
    int64_t src_b0, src_b1;
    const uint8_t *const *src_tab;  // the token pointer table (shared memory when staged)
};

// Next chunk of this CTA as the byte range [*b0, *b1); false when the CTA has no more work.
__device__ bool next_chunk(const Params &p, BulkRing &r, volatile uint32_t *s_first, int64_t *b0, int64_t *b1,
                           uint32_t *tflag)
{
    const int64_t C = p.chunk_bytes;
    if (r.next < r.hi) {
        *b0 = r.next;
        *b1 = min(r.next + C, r.hi);
        r.next = *b1;
        return true;
    }
    if (r.dyn_first < 0)
        return false;
    if (r.tk_next >= r.tk_end) {
        uint32_t t;
        if (!r.started) {
            // the first ticket is claimed by warp 1 (off this thread's path) and handed over in smem
            const uint64_t t0 = global_timer_ns();
            while (s_first[1] == 0u) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    *tflag |= kFlagTimeout;
                    r.dyn_first = -1;
                    return false;
                }
            }
            t = s_first[0];
            r.started = true;
            // keep two claims in flight: a ticket is read two tickets after its atomic was issued
            r.pending[0] = (uint32_t)(atomicAdd(p.ticket, 1ull) & kTicketMask);
            r.pending[1] = (uint32_t)(atomicAdd(p.ticket, 1ull) & kTicketMask);
        } else {
            t = r.pending[0];
            r.pending[0] = r.pending[1];
            r.pending[1] = (uint32_t)(atomicAdd(p.ticket, 1ull) & kTicketMask);
        }
        if (t == kNoTicket || (int64_t)t > r.last_claim) {
            // no ticket, or one no launch can draw: the counter was left by a run of this launch
            // that never finished its claims (an error flagged at the time); flag it here too
            *tflag |= kFlagTimeout;
            r.dyn_first = -1;
            return false;
        }
        r.tk_next = r.dyn_first + (int64_t)t * r.per_ticket;
        r.tk_end = min(r.nch, r.tk_next + r.per_ticket);
        if (r.tk_next >= r.nch) {
            r.dyn_first = -1;
            return false;
        }
    }
    const int64_t id = r.tk_next++;
    *b0 = id * C;
    *b1 = min(*b0 + C, p.total_bytes);
    return true;
}

// Load source bytes [b0, b1) into the next ring stage.  Multi-source form: the range is split
// where it crosses from one rank's buffer into the next (rank boundaries are whole rows, so every
// piece stays 16-byte aligned); all pieces complete on the stage's one barrier.
template <bool kMulti>
__device__ __forceinline__ void bulk_issue_load(const Params &p, BulkRing &r, const SegMap &m, int64_t b0,
                                                int64_t b1)
{
    const int st = (int)(r.issued % p.stages);
    const uint32_t bytes = (uint32_t)(b1 - b0);
    const uint32_t bar = smem_addr(&r.bars[st]);
    const uint32_t dst = smem_addr(r.base + (size_t)st * p.chunk_bytes);
    r.stage_b0[st] = b0;
    r.stage_b1[st] = b1;
    mbar_arrive_expect_tx(bar, bytes);
    if constexpr (kMulti) {
        const int64_t rb = p.row_bytes;
        for (int64_t x = b0; x < b1;) {
            if (x < r.src_b0 || x >= r.src_b1) {
                const int i = rank_of_byte(m, x, rb);
                r.src_b0 = (int64_t)m.row_ex[i * m.E] * rb;
                r.src_b1 = (int64_t)m.row_ex[(i + 1) * m.E] * rb;
                r.src_base = r.src_tab[i];
            }
            const int64_t y = min(b1, r.src_b1);
            const uint32_t d = dst + (uint32_t)(x - b0), n = (uint32_t)(y - x);
            if (p.hints & MRR_HINT_LOAD_EVICT_FIRST)
                bulk_g2s_hint(d, r.src_base + (x - r.src_b0), n, bar, r.policy);
            else
                bulk_g2s(d, r.src_base + (x - r.src_b0), n, bar);
            x = y;
        }
    } else {
        if (p.hints & MRR_HINT_LOAD_EVICT_FIRST)
            bulk_g2s_hint(dst, p.tokens + b0, bytes, bar, r.policy);
        else
            bulk_g2s(dst, p.tokens + b0, bytes, bar);
    }
    ++r.issued;
}

// Ask L2 for source bytes [lo, hi) (16-byte aligned, a multiple of 16 long); the multi-source
// form splits the range where it crosses into the next rank's buffer.
template <bool kMulti>
__device__ __forceinline__ void prefetch_src(const Params &p, const SegMap &m, const Sources &src, int64_t lo,
                                             int64_t hi)
{
    if constexpr (!kMulti) {
        bulk_prefetch_l2(p.tokens + lo, (uint32_t)(hi - lo));
    } else {
        const int64_t rb = p.row_bytes;
        int i = rank_of_byte(m, lo, rb);
        for (int64_t x = lo; x < hi; ++i) {
            const int64_t b0 = (int64_t)m.row_ex[i * m.E] * rb, b1 = (int64_t)m.row_ex[(i + 1) * m.E] * rb;
            const int64_t y = min(hi, b1);
            bulk_prefetch_l2(src.tok[i] + (x - b0), (uint32_t)(y - x));
            x = y;
        }
    }
}

// kCarry: a chunk that starts where the previous one ended (a static range) takes its first
// segment from the previous chunk's last one instead of a binary search.  Measured on GB300: 65,536
// segments (tables in L2) 312.5 -> 294.4 us, 16,384: 100.9 -> 99.8, the multi-source form on C5
// 52.4 -> 51.2; on the fused single-source kernels within noise (C5 -0.2 us, C2 +0.1 us), so those
// are compiled without it.
template <bool kMulti, bool kCarry>
__device__ uint32_t bulk_driver(const Params &p, BulkRing &r, const SegMap &m, uint32_t flags,
                                volatile uint32_t *s_first)
{
    const int S = p.stages;
    const int64_t rb = p.row_bytes;
    int64_t consumed = 0;
    uint32_t tflag = 0u;
    if (!flags) {
        bool more = true;
        int64_t b0, b1;
        // stages the pre-scan prologue left empty (fewer static chunks than stages)
        while (more && r.issued < S) {
            more = next_chunk(p, r, s_first, &b0, &b1, &tflag);
            if (more)
                bulk_issue_load<kMulti>(p, r, m, b0, b1);
        }
        int64_t prev_c1 = -1;  // end of the previous chunk and the segment its last piece was in
        int prev_q = 0;
        for (int64_t n = 0; n < r.issued; ++n) {
            const int st = (int)(n % S);
            if (!mbar_wait_bounded(smem_addr(&r.bars[st]), (uint32_t)((n / S) & 1), kWaitLimitNs)) {
                tflag |= kFlagTimeout;
                break;
            }
            consumed = n + 1;
            const int64_t c0 = r.stage_b0[st], c1 = r.stage_b1[st];
            const uint32_t sbase = smem_addr(r.base + (size_t)st * p.chunk_bytes);
            // one bulk store per piece: the part of the chunk inside one segment
            int q;
            if (kCarry && c0 == prev_c1)   // consecutive (a static range): that segment or the next
                q = (int64_t)m.begin(prev_q + 1) * rb <= c0 ? prev_q + 1 : prev_q;
            else
                q = m.find_byte(c0, rb);
            for (int64_t pos = c0; pos < c1; ++q) {
                const int64_t seg_end = (int64_t)m.begin(q + 1) * rb;
                const int64_t delta = ((int64_t)m.dest(q) - (int64_t)m.begin(q)) * rb;
                const int64_t pe = min(c1, seg_end);
                if (p.hints & MRR_HINT_STORE_EVICT_FIRST)
                    bulk_s2g_hint(p.out_tokens + pos + delta, sbase + (uint32_t)(pos - c0), (uint32_t)(pe - pos),
                                  r.policy);
                else
                    bulk_s2g(p.out_tokens + pos + delta, sbase + (uint32_t)(pos - c0), (uint32_t)(pe - pos));
                pos = pe;
            }
            prev_c1 = c1;
            prev_q = q - 1;
            bulk_commit();
            // refill each stage whose previous chunk (sequence issued - S <= n - 1) has been read out
            bool waited = false;
            while (more && r.issued <= n - 1 + S) {
                more = next_chunk(p, r, s_first, &b0, &b1, &tflag);
                if (!more)
                    break;
                if (!waited) {
                    bulk_wait_read<1>();
                    waited = true;
                }
                bulk_issue_load<kMulti>(p, r, m, b0, b1);
            }
        }
    }
    // loads issued but not consumed (invalid counts or a timeout): let them land before exit
    for (int64_t c = consumed; c < r.issued; ++c)
        (void)mbar_wait_bounded(smem_addr(&r.bars[c % S]), (uint32_t)((c / S) & 1), kWaitLimitNs);
    bulk_wait_all<0>();
    return tflag;
}

// ------------------------------------------------------------------------------------------------
// kernels

// kBulk: bulk-copy ring (rows a multiple of 16 bytes) or vector path; kFused: the counts are
// scanned in every CTA (N*E <= 4096); kStage (N*E > 4096 only): the scan kernel's tables are
// copied into shared memory first instead of being read from L2; kMulti: the multi-source form
// (rank i's rows in a buffer of their own, forward move only).
template <bool kBulk, bool kFused, bool kStage, bool kMulti>
__global__ void __launch_bounds__(1024) reroute_kernel(const Params p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bars[kMaxStages];
    __shared__ int64_t stage_b0[kMaxStages], stage_b1[kMaxStages];
    __shared__ uint32_t s_warp[32];
    __shared__ uint32_t s_flags;
    __shared__ unsigned long long s_sum;
    __shared__ volatile uint32_t s_first[2];  // [0] first ticket of this CTA, [1] set once [0] is valid

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int64_t G = gridDim.x, b = blockIdx.x;

    // this CTA's slice of the source bytes, in 16-byte units (static scheduling, vector path)
    const int64_t units = (p.total_bytes + 15) >> 4;
    const int64_t lo = min(p.total_bytes, (b * units / G) << 4);
    const int64_t hi = (b == G - 1) ? p.total_bytes : min(p.total_bytes, ((b + 1) * units / G) << 4);

    BulkRing ring;
    ring.bars = bars;
    ring.base = smem;
    ring.stage_b0 = stage_b0;
    ring.stage_b1 = stage_b1;
    ring.issued = 0;
    ring.policy = 0;
    ring.pending[0] = ring.pending[1] = 0u;
    ring.tk_next = ring.tk_end = 0;
    ring.per_ticket = (int)max(1, min(64, 65536 / p.chunk_bytes));
    ring.started = false;
    ring.nch = (p.total_bytes + p.chunk_bytes - 1) / p.chunk_bytes;
    ring.src_base = nullptr;
    ring.src_b0 = ring.src_b1 = 0;
    const bool dynamic = kBulk && p.sched == 1;
    if (dynamic) {
        const int64_t span = (int64_t)p.static_chunks * p.chunk_bytes;
        ring.next = min(p.total_bytes, b * span);
        ring.hi = min(p.total_bytes, (b + 1) * span);
        ring.dyn_first = (G * span < p.total_bytes) ? G * (int64_t)p.static_chunks : -1;
        // Each CTA draws exactly its tickets + 3 values: the first ticket, the two claims kept in
        // flight, and one claim per ticket it takes, the last of which is past the end.
        const int64_t tickets = (ring.nch - ring.dyn_first + ring.per_ticket - 1) / ring.per_ticket;
        ring.last_claim = ring.dyn_first >= 0 ? tickets + 3 * G - 1 : -1;
    } else {
        ring.next = lo;
        ring.hi = hi;
        ring.dyn_first = -1;
        ring.last_claim = -1;
    }
    uint32_t *tab = reinterpret_cast<uint32_t *>(smem + (kBulk ? (size_t)p.stages * p.chunk_bytes : 0));

    SegMap m;
    m.NE = p.NE;
    m.N = p.N;
    m.E = p.E;
    m.inv = p.inverse;
    Sources src{p.src_tok, p.src_sc, p.src_tk, p.src_rows};
    ring.src_tab = p.src_tok;
    // Multi-source form: copy the per-rank pointer tables and row capacities into shared memory
    // (their loads overlap the count loads); the capacity check before the token stream and the
    // bulk driver's rank lookups then take no global round trip.  The block synchronises before
    // anything reads the copy.
    auto stage_pointers = [&]() {
        if (kMulti && p.ptr_off >= 0) {
            const uint8_t **t = reinterpret_cast<const uint8_t **>(smem + p.ptr_off);
            const int n_sc = p.src_sc ? 1 : 0, n_tk = p.src_tk ? 1 : 0;
            const uint8_t **tok = t, **sc = t + p.N, **tk = t + (1 + n_sc) * p.N;
            long long *rows = reinterpret_cast<long long *>(t + (1 + n_sc + n_tk) * p.N);
            for (int i = tid; i < p.N; i += nthr) {
                tok[i] = p.src_tok[i];
                if (p.src_sc)
                    sc[i] = p.src_sc[i];
                if (p.src_tk)
                    tk[i] = p.src_tk[i];
                if (p.src_rows)
                    rows[i] = p.src_rows[i];
            }
            src.tok = tok;
            src.sc = p.src_sc ? sc : nullptr;
            src.tk = p.src_tk ? tk : nullptr;
            src.rows = p.src_rows ? rows : nullptr;
            ring.src_tab = tok;
        }
    };

    CountBatch cb;
    if (tid == 0)
        s_first[1] = 0u;
    if (kBulk && tid == 0) {
        for (int s = 0; s < p.stages; ++s)
            mbar_init(smem_addr(&bars[s]), 1u);
        mbar_init_fence();
    }
    // Start streaming the token rows: their source addresses need no offsets (single source).
    // Thread 0 fills the ring with this CTA's first chunks; warp 1 asks L2 for the next ones.
    // The multi-source form needs the rank offsets to address its sources, so it starts only once
    // the segment map is ready and the per-rank pointers have been checked.
    auto start_token_stream = [&]() {
        if (kBulk && tid == 0) {
            if (p.hints)
                ring.policy = policy_evict_first();
            while (ring.issued < p.stages && ring.next < ring.hi) {
                const int64_t b0 = ring.next, b1 = min(ring.next + p.chunk_bytes, ring.hi);
                ring.next = b1;
                bulk_issue_load<kMulti>(p, ring, m, b0, b1);
            }
        }
        if (kBulk && p.prefetch_chunks > 0 && tid >= 32 && tid < 64) {
            // The ring holds only `stages` chunks, which land long before the offsets are ready.
            // Keep HBM busy meanwhile: warp 1 asks L2 for the next chunks, one per lane -- first
            // this CTA's own static chunks past the ring, then its share of the first chunks the
            // counter hands out.
            const int64_t C = p.chunk_bytes;
            const int64_t st0 = ring.next + (int64_t)p.stages * C;  // ring.next: this CTA's first byte
            const int64_t n_s =
                st0 < ring.hi ? min((ring.hi - st0 + C - 1) / C, (int64_t)p.prefetch_chunks) : 0;
            const int64_t n_d = ring.dyn_first >= 0 ? p.prefetch_chunks - n_s : 0;
            const int64_t d_lo = ring.dyn_first + b * n_d;
            for (int64_t i = tid - 32; i < n_s + n_d; i += 32) {
                int64_t lo, hi;
                if (i < n_s) {
                    lo = st0 + i * C;
                    hi = min(lo + C, ring.hi);
                } else {
                    const int64_t c = d_lo + (i - n_s);
                    if (c >= ring.nch)
                        break;
                    lo = c * C;
                    hi = min(lo + C, p.total_bytes);
                }
                prefetch_src<kMulti>(p, m, src, lo, hi);
            }
        }
    };
    // Behind the scan kernel (N*E > 4096) the tokens can stream before the wait below: that kernel
    // runs its own wait before it lets this one start, so whatever wrote the tokens has finished,
    // and it writes only the workspace tables, which are read after the wait.  The fused kernel may
    // follow the tokens' producer directly, so it starts them after the wait.
    if (!kFused && !kMulti)
        start_token_stream();
    if (kFused && kMulti)
        prefetch_inputs_l2(p, tid, nthr);
    // When launched behind another kernel with programmatic stream serialization, wait for it
    // here, then let the next launch be scheduled.
    grid_dependency_wait();
    grid_launch_dependents();
    if (kFused) {
        if (tid == 0) {
            s_flags = 0u;
            s_sum = 0ull;
        }
        if (p.count_is_i64)
            issue_count_loads<long long>(p, 0, cb);
        else
            issue_count_loads<int>(p, 0, cb);
        if (!kMulti)
            start_token_stream();
        stage_pointers();
    }

    uint32_t flags;
    if (kFused) {
        uint32_t *rex = tab, *cnt_t = tab + p.NE + 1, *dof = cnt_t + padded_len(p.NE);
        m.row_ex = rex;
        m.dst_off = dof;
        m.col_ex = cnt_t;
        if constexpr (kMulti) {
            // Once SrcOffset is scanned (rank i's rows start at SrcOffset(i, 0)), check every
            // rank's pointers and row count (uniform over the block), then start the token stream
            // while DstOffset is scanned.  Counts that fail validation return before this point.
            uint32_t src_flag = 0u;
            auto mid = [&]() {
                const uint32_t f = check_sources(p, src, kBulk, tid, nthr) | check_capacity(p, src, rex, tid, nthr);
                if (__syncthreads_or(f != 0u))
                    src_flag = kFlagSource;
                else
                    start_token_stream();
            };
            flags = cta_scan(p, cb, rex, cnt_t, dof, s_warp, &s_flags, &s_sum, mid) | src_flag;
        } else {
            flags = cta_scan(p, cb, rex, cnt_t, dof, s_warp, &s_flags, &s_sum);
        }
        if (b == 0) {
            if (!flags && !p.inverse)
                write_expert_token_num(p, dof, tid, nthr);
            if (tid == 0) {
                p.status[0] = flags;
                p.status[1] = (uint32_t)G;
            }
        }
    } else {
        stage_pointers();
        __syncthreads();  // s_first[1] cleared before warp 1 may set it; pointer tables staged
        // written by the scan kernel (its count checks and, multi-source, its pointer checks)
        flags = *reinterpret_cast<volatile uint32_t *>(p.status);
        m.row_ex = p.g_row_ex;
        m.dst_off = p.g_dst_off;
        m.col_ex = p.g_col_ex;
        if (kStage && !flags) {
            // Copy the two tables this direction uses from L2 into shared memory, so the driver's
            // binary searches and per-piece lookups do not pay an L2 round trip each:
            //   the starts: SrcOffset [0, NE] (forward) or the column-major starts (inverse, padded)
            //   the destinations: dst_off (padded; by segment forward, by position inverse)
            // 16-byte copies; the workspace tables are 256-byte aligned and a few words longer.
            const int n2 = (int)((padded_len(p.NE) + 3) >> 2);
            const int n1 = p.inverse ? n2 : (p.NE + 1 + 3) >> 2;
            uint32_t *first = tab, *second = tab + 4 * n1;
            const uint32_t *gfirst = p.inverse ? p.g_col_ex : p.g_row_ex;
#pragma unroll 1
            for (int k = tid; k < n1; k += nthr)
                reinterpret_cast<uint4 *>(first)[k] = reinterpret_cast<const uint4 *>(gfirst)[k];
#pragma unroll 1
            for (int k = tid; k < n2; k += nthr)
                reinterpret_cast<uint4 *>(second)[k] = reinterpret_cast<const uint4 *>(p.g_dst_off)[k];
            __syncthreads();
            m.row_ex = first;
            m.col_ex = first;
            m.dst_off = second;
        }
        if (b == 0 && tid == 0)
            p.status[1] = (uint32_t)G;
    }
    if (kMulti && !kFused && !flags)
        start_token_stream();

    uint32_t tflag = 0u;
    if (kBulk) {
        if (tid == 0) {
            tflag = bulk_driver<kMulti, !kFused || kMulti>(p, ring, m, flags, s_first);
        } else if (tid >= 32 && !flags) {
            if (tid == 32 && dynamic && ring.dyn_first >= 0) {
                s_first[0] = claim_first_ticket(p.ticket, p.epoch, ring.last_claim);
                __threadfence_block();
                s_first[1] = 1u;
            }
            side_arrays<kMulti>(p, m, src, tid - 32, nthr - 32);
        }
    } else if (!flags) {
        vector_copy<kMulti>(p, m, src, lo, hi, tid, nthr);
        side_arrays<kMulti>(p, m, src, tid, nthr);
    }
    if (tid == 0)
        p.status[2 + b] = tflag;
}

// N*E > 4096: one CTA validates the counts and writes both prefixes and expert_token_num to
// global memory, tile by tile with a running carry.
__global__ void __launch_bounds__(1024) scan_kernel(const Params p)
{
    extern __shared__ __align__(16) uint32_t sm_tab[];
    __shared__ uint32_t s_warp[32];
    __shared__ uint32_t s_flags;
    __shared__ unsigned long long s_sum;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
    const int NE = p.NE, N = p.N, E = p.E;
    if (tid == 0) {
        s_flags = 0u;
        s_sum = 0ull;
    }
    if (p.multi)
        prefetch_inputs_l2(p, tid, nthr);
    // The wait must stay ahead of launch_dependents: the copy kernel behind this one loads token
    // rows before its own wait, and only this order makes whatever wrote them finish first.
    grid_dependency_wait();
    grid_launch_dependents();
    if (p.multi) {
        // the multi-source form's per-rank pointers, checked once here for the copy kernel, which
        // reads this status word before it touches any source
        const Sources src{p.src_tok, p.src_sc, p.src_tk, p.src_rows};
        if (__syncthreads_or(check_sources(p, src, p.multi_bulk != 0, tid, nthr) != 0u)) {
            if (tid == 0)
                p.status[0] = kFlagSource;
            return;
        }
    }
    if (p.scan_in_smem) {
        // the same in-CTA scan the fused copy kernel runs, then the tables written out
        uint32_t *rex = sm_tab, *cnt_t = sm_tab + NE + 1, *dof = cnt_t + padded_len(NE);
        CountBatch cb;
        if (p.count_is_i64)
            issue_count_loads<long long>(p, 0, cb);
        else
            issue_count_loads<int>(p, 0, cb);
        uint32_t flags = cta_scan(p, cb, rex, cnt_t, dof, s_warp, &s_flags, &s_sum);
        if (p.multi && !flags &&
            __syncthreads_or(check_capacity(p, Sources{p.src_tok, p.src_sc, p.src_tk, p.src_rows}, rex, tid, nthr) != 0u))
            flags = kFlagSource;
        if (flags) {
            if (tid == 0)
                p.status[0] = flags;
            return;
        }
        for (int k = tid; k <= NE; k += nthr)
            p.g_row_ex[k] = rex[k];
        const int np = (int)padded_len(NE);
        for (int k = tid; k < np; k += nthr)
            p.g_dst_off[k] = dof[k];
        if (p.inverse)
            for (int k = tid; k < np; k += nthr)
                p.g_col_ex[k] = cnt_t[k];
        else
            write_expert_token_num(p, dof, tid, nthr);
        if (tid == 0)
            p.status[0] = 0u;
        return;
    }
    __syncthreads();
    uint32_t f = 0u;
    unsigned long long sum = 0ull;
    for (int k = tid; k < NE; k += nthr) {
        const int64_t c = load_count(p, k);
        if (c <= 0)
            f |= kFlagNonPos;
        else if (c > p.A)
            f |= kFlagSum;
        else
            sum += (unsigned long long)c;
    }
    f = __reduce_or_sync(0xffffffffu, f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_down_sync(0xffffffffu, sum, o);
    if (lane == 0) {
        if (f)
            atomicOr(&s_flags, f);
        if (sum)
            atomicAdd(&s_sum, sum);
    }
    __syncthreads();
    uint32_t flags = s_flags;
    if (!flags && s_sum != (unsigned long long)p.A)
        flags |= kFlagSum;
    if (flags) {
        if (tid == 0)
            p.status[0] = flags;
        return;
    }
    uint32_t carry = 0u, total;
    for (int base = 0; base < NE; base += nthr) {
        const int k = base + tid;
        const uint32_t v = k < NE ? (uint32_t)load_count(p, k) : 0u;
        const uint32_t ex = block_exscan(v, &total, s_warp);
        if (k < NE)
            p.g_row_ex[k] = carry + ex;
        carry += total;
    }
    if (tid == 0)
        p.g_row_ex[NE] = (uint32_t)p.A;
    __syncthreads();  // the row-major starts above, read by position below (inverse move)
    if (p.multi &&
        __syncthreads_or(check_capacity(p, Sources{p.src_tok, p.src_sc, p.src_tk, p.src_rows}, p.g_row_ex, tid, nthr) != 0u)) {
        if (tid == 0)
            p.status[0] = kFlagSource;
        return;
    }
    carry = 0u;
    for (int base = 0; base < NE; base += nthr) {
        const int pos = base + tid;
        const int q = pos < NE ? (pos % N) * E + pos / N : 0;
        const uint32_t v = pos < NE ? (uint32_t)load_count(p, q) : 0u;
        const uint32_t ex = block_exscan(v, &total, s_warp);
        if (pos < NE && !p.inverse)
            p.g_dst_off[pad32(q)] = carry + ex;
        if (pos < NE && p.inverse) {
            p.g_col_ex[pad32(pos)] = carry + ex;
            p.g_dst_off[pad32(pos)] = p.g_row_ex[q];
        }
        carry += total;
    }
    if (tid == 0 && p.inverse)
        p.g_col_ex[pad32(NE)] = (uint32_t)p.A;
    __syncthreads();  // global writes of the block visible to the whole block
    if (!p.inverse)
        write_expert_token_num(p, p.g_dst_off, tid, nthr);
    if (tid == 0)
        p.status[0] = 0u;
}

}  // namespace mrr

// ================================================================================================
// host side

using namespace mrr;

namespace {

int token_bits(int dt)
{
    switch (dt) {
    case MRR_F16:
    case MRR_BF16:
        return 16;
    case MRR_I8:
    case MRR_F8E5M2:
    case MRR_F8E4M3FN:
    case MRR_HIF8:
        return 8;
    case MRR_F4E2M1:
    case MRR_F4E1M2:
        return 4;
    default:
        return 0;
    }
}

using mrr_ws::round_up;
using mrr_ws::table_workspace_bytes;

// Shared memory of the two tables the copy kernel stages when N*E > 4096 (see reroute_kernel).
int64_t staged_table_bytes(int64_t NE)
{
    return 8 * ((padded_len(NE) + 3) & ~int64_t(3));  // two padded tables (the row-major one is shorter)
}

// Shared memory of the scan kernel's in-CTA scan (row-major counts, column-major copy, DstOffset).
int64_t scan_smem_bytes(int64_t NE)
{
    return 4 * (NE + 1 + 2 * padded_len(NE));
}

int widest_width(uintptr_t a, uintptr_t b, int64_t bytes, int cap)
{
    int w = cap;
    while (w > 1 && (((a | b) & (uintptr_t)(w - 1)) != 0 || bytes % w != 0))
        w >>= 1;
    return w;
}

// checks shared by plan and run: shapes and attributes (no pointers)
mrr_status check_shape(int64_t A, int64_t H, int dt, int64_t N, int64_t E, int count_is_i64, int sl,
                       int64_t scale_cols, int64_t etn_type, int64_t idx_type, int64_t *row_bytes,
                       int64_t *scale_row_bytes)
{
    const int bits = token_bits(dt);
    if (bits == 0 || sl < MRR_SCALE_NONE || sl > MRR_SCALE_E8M0_AK2 || (count_is_i64 != 0 && count_is_i64 != 1))
        return MRR_ERR_DTYPE;
    if (etn_type != 0 && etn_type != 1)
        return MRR_ERR_ATTR;
    if (idx_type != 0 && idx_type != 1)
        return MRR_ERR_ATTR;
    // section 约束说明: 0 < H < 16384; A = Sum(counts) with every count > 0 (so N*E <= A);
    // the index output is int32, so A <= INT32_MAX
    if (H <= 0 || H >= 16384 || (bits == 4 && (H & 1)))
        return MRR_ERR_SHAPE;
    if (A < 0 || A > INT32_MAX || N < 0 || E < 0)
        return MRR_ERR_SHAPE;
    if (N > INT32_MAX || E > INT32_MAX || (N > 0 && E > INT32_MAX / N))
        return MRR_ERR_SHAPE;
    const int64_t NE = N * E;
    if ((NE == 0) != (A == 0) || NE > A)
        return MRR_ERR_SHAPE;
    int64_t sb = 0;
    switch (sl) {
    case MRR_SCALE_NONE:
        sb = 0;
        break;
    case MRR_SCALE_F32_A:
        if (scale_cols != 1)
            return MRR_ERR_SHAPE;
        sb = 4;
        break;
    case MRR_SCALE_F32_AS:
        if (scale_cols < 1 || scale_cols > (1 << 20))
            return MRR_ERR_SHAPE;
        sb = 4 * scale_cols;
        break;
    case MRR_SCALE_E8M0_AK2:
        if (scale_cols < 2 || (scale_cols & 1) || scale_cols > (1 << 20))
            return MRR_ERR_SHAPE;
        sb = scale_cols;
        break;
    }
    *row_bytes = H * bits / 8;
    *scale_row_bytes = sb;
    return MRR_OK;
}

// pointer checks shared by run and run_plan (section 参数说明: the top-k input and output come
// as a pair; scales need an output; index and counts are read/written as their int types)
// (inverse: the move back to rank-major order, which writes no index and no counts)
mrr_status check_buffers(int64_t NE, int64_t E, int cb, int sl, const void *tokens, const void *counts,
                         const void *scales, const void *topk_w, const void *permute_tokens,
                         const void *permute_scales, const void *idx, const void *etn, const void *permute_topk_w,
                         const void *workspace, size_t workspace_bytes, int inverse = 0)
{
    if (inverse) {
        idx = nullptr;
        etn = nullptr;
    }
    if ((topk_w == nullptr) != (permute_topk_w == nullptr))
        return MRR_ERR_TOPK_PAIR;
    if (sl != MRR_SCALE_NONE && (!scales || !permute_scales))
        return MRR_ERR_NULL;
    if (sl == MRR_SCALE_NONE && scales)
        return MRR_ERR_DTYPE;
    if (!inverse && E > 0 && !etn)
        return MRR_ERR_NULL;
    if (NE > 0 && (!tokens || !counts || !permute_tokens || (!inverse && !idx)))
        return MRR_ERR_NULL;
    if (((uintptr_t)counts % cb) || ((uintptr_t)etn % cb) || ((uintptr_t)idx % 4))
        return MRR_ERR_ALIGN;
    if (!workspace || ((uintptr_t)workspace % 256) || workspace_bytes < (size_t)kHeaderBytes)
        return MRR_ERR_WORKSPACE;
    return MRR_OK;
}

// A fresh 40-bit tag for every launch: it marks the shared chunk counter as belonging to that
// launch, so stale counter values from earlier launches (or a fresh workspace) are recognised.
unsigned long long next_launch_epoch()
{
    static std::atomic<unsigned long long> counter{0};
    static const unsigned long long seed = [] {
        unsigned long long x = (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
        x ^= (unsigned long long)(uintptr_t)&counter;
        x += 0x9E3779B97F4A7C15ull;  // splitmix64 finaliser
        x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
        x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
        return x ^ (x >> 31);
    }();
    const unsigned long long mask = (1ull << (64 - kTicketBits)) - 1;
    for (;;) {
        const unsigned long long e = (seed + counter.fetch_add(1)) & mask;
        if (e)
            return e;
    }
}

constexpr int kNumKernels = 17;  // 16 copy-kernel variants, then the scan kernel
// per device: the kernel's dynamic shared memory limit has been raised (any host thread may launch;
// two first launches may both raise it, which is harmless, but the flag itself must not race)
std::atomic<bool> g_smem_attr_set[64][kNumKernels];

template <bool kBulk, bool kFused, bool kStage, bool kMulti>
int kernel_slot()
{
    return (kMulti ? 8 : 0) + (kBulk ? 4 : 0) + (kFused ? 2 : 0) + (kStage ? 1 : 0);
}

// Launch with or without programmatic stream serialization (the kernels wait for their
// predecessor before touching global memory either way).
template <typename K>
cudaError_t launch(K kern, const Params &p, int grid, int block, int smem, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_scan(const Params &p, int smem, cudaStream_t stream, int device, bool pdl)
{
    constexpr int slot = 16;
    if (smem > 48 * 1024 && device >= 0 && device < 64 &&
        !g_smem_attr_set[device][slot].load(std::memory_order_acquire)) {
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 1024);
        if (e != cudaSuccess)
            return e;
        g_smem_attr_set[device][slot].store(true, std::memory_order_release);
    }
    return launch(scan_kernel, p, 1, 1024, smem, stream, pdl);
}

template <bool kBulk, bool kFused, bool kStage, bool kMulti>
cudaError_t launch_copy(const Params &p, int grid, int block, int smem, cudaStream_t stream, int device, bool pdl)
{
    auto kern = reroute_kernel<kBulk, kFused, kStage, kMulti>;
    const int slot = kernel_slot<kBulk, kFused, kStage, kMulti>();
    if (device >= 0 && device < 64 && !g_smem_attr_set[device][slot].load(std::memory_order_acquire)) {
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 1024);
        if (e != cudaSuccess)
            return e;
        g_smem_attr_set[device][slot].store(true, std::memory_order_release);
    }
    return launch(kern, p, grid, block, smem, stream, pdl);
}

}  // namespace

namespace mrr_host {

mrr_status check_shape(int64_t A, int64_t H, int dt, int64_t N, int64_t E, int count_is_i64, int sl,
                       int64_t scale_cols, int64_t etn_type, int64_t idx_type, int64_t *row_bytes,
                       int64_t *scale_row_bytes)
{
    return ::check_shape(A, H, dt, N, E, count_is_i64, sl, scale_cols, etn_type, idx_type, row_bytes,
                         scale_row_bytes);
}

}  // namespace mrr_host

extern "C" {

const char *mrr_status_str(mrr_status s)
{
    switch (s) {
    case MRR_OK:
        return "MRR_OK";
    case MRR_ERR_NULL:
        return "MRR_ERR_NULL: a required pointer is NULL";
    case MRR_ERR_SHAPE:
        return "MRR_ERR_SHAPE: A, H, N, E or scale_cols out of range";
    case MRR_ERR_DTYPE:
        return "MRR_ERR_DTYPE: unknown token dtype, scale layout or count type";
    case MRR_ERR_ATTR:
        return "MRR_ERR_ATTR: expert_token_num_type or idx_type not in {0, 1}";
    case MRR_ERR_UNSUPPORTED:
        return "MRR_ERR_UNSUPPORTED: expert_token_num_type 0 (cumsum mode) is not supported";
    case MRR_ERR_TOPK_PAIR:
        return "MRR_ERR_TOPK_PAIR: expert_topk_weight and permute_topk_weight must be given together";
    case MRR_ERR_WORKSPACE:
        return "MRR_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MRR_ERR_CUDA:
        return "MRR_ERR_CUDA: a CUDA runtime call failed";
    case MRR_ERR_ALIGN:
        return "MRR_ERR_ALIGN: counts, index or expert_token_num pointer misaligned for its type";
    case MRR_ERR_PLAN:
        return "MRR_ERR_PLAN: the plan does not match the arguments or is out of range";
    case MRR_ERR_COUNT_NONPOS:
        return "MRR_ERR_COUNT_NONPOS: a count is <= 0";
    case MRR_ERR_COUNT_SUM:
        return "MRR_ERR_COUNT_SUM: the counts do not sum to A";
    case MRR_ERR_TIMEOUT:
        return "MRR_ERR_TIMEOUT: a bounded wait in the copy kernel gave up";
    case MRR_ERR_INDEX:
        return "MRR_ERR_INDEX: an input_ids or tid2eid value is out of range";
    case MRR_ERR_SOURCE:
        return "MRR_ERR_SOURCE: a per-rank source pointer is NULL, or not 16-byte aligned on the bulk path";
    case MRR_ERR_DEST:
        return "MRR_ERR_DEST: a receiver's buffer pointer is NULL, or a row would land past its rows";
    }
    return "unknown mrr_status";
}

}  // extern "C"

namespace {

mrr_status make_plan(int64_t A, int64_t H, mrr_token_dtype dt, int64_t N, int64_t E, int count_is_i64,
                     mrr_scale_layout sl, int64_t scale_cols, int has_topk, int64_t expert_token_num_type,
                     int64_t idx_type, int device, int direction, mrr_v2_plan_t *out)
{
    if (!out)
        return MRR_ERR_NULL;
    int64_t rb = 0, sb = 0;
    mrr_status st = check_shape(A, H, (int)dt, N, E, count_is_i64, (int)sl, scale_cols, expert_token_num_type,
                                idx_type, &rb, &sb);
    if (st != MRR_OK)
        return st;
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    const int64_t NE = N * E;
    const int64_t total = A * rb;
    mrr_v2_plan_t p;
    memset(&p, 0, sizeof(p));
    p.A = A;
    p.H = H;
    p.N = N;
    p.E = E;
    p.row_bytes = rb;
    p.scale_row_bytes = sb;
    p.count_is_i64 = count_is_i64;
    p.scale_layout = (int32_t)sl;
    p.has_topk = has_topk ? 1 : 0;
    p.idx_type = (int32_t)idx_type;
    p.fuse_scan = NE <= kFusedMaxSegs ? 1 : 0;
    p.path = (rb % 16 == 0) ? MRR_PATH_BULK : MRR_PATH_VECTOR;
    p.num_sms = sms;
    p.pdl = 1;
    p.direction = direction;
    // N*E > 4096: the copy kernel stages its two tables in shared memory when a ring of 3 x 48 KiB
    // still fits beside them (up to about 10k segments; the ring below is sized around them).
    // Measured on GB300: a smaller ring loses more than the L2 lookups cost (16384 segments:
    // 2 x 44 KiB staged 147 us per copy launch, 3 x 64 KiB reading the tables from L2 about 105).
    const int64_t stage = staged_table_bytes(NE);
    const bool can_stage = !p.fuse_scan && (p.path == MRR_PATH_BULK ? stage + 3 * 49152 <= optin - 1024
                                                                   : stage <= optin - 1024);
    const int64_t table_bytes = p.fuse_scan ? round_up(4 * (NE + 1 + 2 * padded_len(NE)), 128)
                                            : (can_stage ? stage : 0);
    if (p.path == MRR_PATH_BULK) {
        // the ring: 5 x 44 KiB or 5 x 40 KiB up to 1024 segments, else 3 x 64 KiB, 3 x 48 KiB,
        // 4 x 32 KiB, ..., the first that fits beside the tables
        // More threads when the in-CTA scan of many segments is long.
        p.block = NE > 1024 ? 512 : 256;
        // Measured on GB300: plain L2 policies beat evict-first hints on both loads and stores.
        p.hints = 0;
        p.chunk_bytes = 65536;
        p.stages = 3;
        // Up to 1024 segments a deeper ring of smaller chunks (5 x 44 KiB, else 5 x 40 KiB) keeps
        // more loads in flight per SM: measured on GB300 against 3 x 64 KiB, C2 36.99 -> 35.96 us,
        // C3 70.49 -> 69.58, C4 72.91 -> 71.75.  At 4096 segments (C5) five stages lost (51 us).
        // Above 1024 segments (the in-CTA tables take 13-50 KB) four stages of 44 KiB still fit:
        // measured on GB300 against 3 x 48 KiB / 3 x 64 KiB, 4096 segments (C5) 44.22 -> 42.99 us
        // and 2048 segments 44.90 -> 42.7 us, with 2 prefetched chunks and 8 static chunks (below).
        if (NE <= 1024 && 5 * 45056 + table_bytes <= optin - 1024) {
            p.chunk_bytes = 45056;
            p.stages = 5;
        } else if (NE <= 1024 && 5 * 40960 + table_bytes <= optin - 1024) {
            p.chunk_bytes = 40960;
            p.stages = 5;
        } else if (p.fuse_scan && 4 * 45056 + table_bytes <= optin - 1024) {
            p.chunk_bytes = 45056;
            p.stages = 4;
        }
        if ((int64_t)p.stages * p.chunk_bytes + table_bytes > optin - 1024)
            p.chunk_bytes = 49152;
        if ((int64_t)p.stages * p.chunk_bytes + table_bytes > optin - 1024) {
            p.chunk_bytes = 32768;
            p.stages = 4;
        }
        while (p.stages > 2 && (int64_t)p.stages * p.chunk_bytes + table_bytes > optin - 1024)
            --p.stages;
        while (p.chunk_bytes > 4096 && (int64_t)p.stages * p.chunk_bytes + table_bytes > optin - 1024)
            p.chunk_bytes /= 2;
        // dynamic chunk scheduling unless the counter's 24-bit ticket space could run out; with
        // the four-stage ring above 1024 segments, 8 static chunks per CTA (measured at 4096
        // segments: 6 or 8 best, 42.99 us; the default 5: 43.69; 12: 43.39; 16: 44.00)
        const bool ring4 = p.fuse_scan && NE > 1024 && p.stages == 4;
        p.static_chunks = ring4 ? 8 : p.stages + 1;
        // many segments: the in-CTA scan outlasts the ring's loads, so prefetch the next chunks
        // into L2 meanwhile (measured at 4096 segments: 4 chunks per CTA with a 3-stage ring, 2
        // with the 4-stage ring (0: 44.93 us, 1: 43.95, 2: 43.69, 3: 44.04, 6: 45.10); none
        // below 1024 segments; behind the scan kernel, N*E > 4096, 4 to 12 chunks were 0-10 %
        // slower than none)
        p.prefetch_chunks = (p.fuse_scan && NE > 1024) ? (ring4 ? 2 : 4) : 0;
        const int64_t nch = (total + p.chunk_bytes - 1) / p.chunk_bytes;
        p.sched = (nch + 3 * kMaxGrid < (int64_t)kTicketMask) ? 1 : 0;
        p.smem_bytes = (int32_t)((int64_t)p.stages * p.chunk_bytes + table_bytes);
        const int64_t want = (total + 65535) / 65536;
        p.grid = (int32_t)(want < 1 ? 1 : (want > sms ? sms : want));
        // Behind the scan kernel with the tables left in L2 (too many segments to stage), a chunk
        // claimed from the counter lands anywhere in the tables, and its binary search then misses
        // in L1 on every probe.  Static ranges walk the tables in order, so they cover about 90 %
        // of the chunks there and the counter balances the rest.  Measured on GB300 (A=32768,
        // H=7168 int8): 12,288 segments 112.0 -> 97.2 us, 16,384: 123.0 -> 102.4, 20,000 (A=40000):
        // 176.3 -> 147.2; 65,536 segments (A=131072, H=1024 bf16) 347.7 -> 312.7.
        if (!p.fuse_scan && !can_stage && p.grid > 0) {
            const int64_t per_cta = nch * 9 / 10 / p.grid;
            if (per_cta > p.static_chunks)
                p.static_chunks = (int32_t)(per_cta < (1 << 20) ? per_cta : (1 << 20));
        }
    } else {
        p.block = 512;
        p.chunk_bytes = 32768;
        p.stages = 4;
        p.smem_bytes = (int32_t)table_bytes;
        const int64_t want = (total + 65535) / 65536;
        const int64_t cap = 2 * (int64_t)sms;
        p.grid = (int32_t)(want < 1 ? 1 : (want > cap ? cap : want));
    }
    if (p.grid > kMaxGrid)
        p.grid = kMaxGrid;
    p.workspace_bytes = kHeaderBytes + (p.fuse_scan ? 0 : table_workspace_bytes(NE, direction));
    *out = p;
    return MRR_OK;
}

// The copy-kernel variant for a path, scan placement and table staging.
template <bool kMulti>
cudaError_t launch_variant(bool bulk, bool fused, bool stage, const Params &p, int grid, int block, int sm,
                           cudaStream_t stream, int device, bool pdl)
{
    if (bulk)
        return fused   ? launch_copy<true, true, false, kMulti>(p, grid, block, sm, stream, device, pdl)
               : stage ? launch_copy<true, false, true, kMulti>(p, grid, block, sm, stream, device, pdl)
                       : launch_copy<true, false, false, kMulti>(p, grid, block, sm, stream, device, pdl);
    return fused   ? launch_copy<false, true, false, kMulti>(p, grid, block, sm, stream, device, pdl)
           : stage ? launch_copy<false, false, true, kMulti>(p, grid, block, sm, stream, device, pdl)
                   : launch_copy<false, false, false, kMulti>(p, grid, block, sm, stream, device, pdl);
}

// The per-rank source tables of the multi-source form (device arrays of N device pointers).
struct MultiSrc {
    const void *const *tokens;
    const void *const *scales;
    const float *const *topk;
    const int64_t *rows;
};

// mrr_v2_run_plan, and with ms != NULL its multi-source form: tokens / scales / topk_w are then
// unused and each rank's rows come from ms's tables.
mrr_status run_plan_impl(const mrr_v2_plan_t *plan, const MultiSrc *ms, const void *tokens, mrr_token_dtype dt,
                         const void *counts, const void *scales, const float *topk_w, void *permute_tokens,
                         void *permute_scales, int32_t *permute_token_idx, void *expert_token_num,
                         float *permute_topk_w, int64_t expert_token_num_type, void *workspace,
                         size_t workspace_bytes, mrr_stream_t stream_)
{
    if (!plan)
        return MRR_ERR_NULL;
    const mrr_v2_plan_t &pl = *plan;
    int64_t rb = 0, sb = 0;
    mrr_status st = check_shape(pl.A, pl.H, (int)dt, pl.N, pl.E, pl.count_is_i64, pl.scale_layout,
                                pl.scale_layout == MRR_SCALE_E8M0_AK2 ? pl.scale_row_bytes
                                                                      : pl.scale_row_bytes / 4,
                                expert_token_num_type, pl.idx_type, &rb, &sb);
    if (st != MRR_OK)
        return st;
    if (rb != pl.row_bytes || sb != pl.scale_row_bytes)
        return MRR_ERR_PLAN;
    const int64_t A = pl.A, N = pl.N, E = pl.E, NE = N * E;
    const int cb = pl.count_is_i64 ? 8 : 4;
    if (pl.direction != 0 && pl.direction != 1)
        return MRR_ERR_PLAN;
    const int inverse = pl.direction;
    if (inverse) {
        if (ms)
            return MRR_ERR_PLAN;  // the multi-source form is the forward move only
        permute_token_idx = nullptr;
        expert_token_num = nullptr;
    }
    if (ms) {
        // the tables stand in for the buffers in the checks below; each rank's own pointers are
        // checked on the device (they live in device memory)
        tokens = ms->tokens;
        scales = ms->scales;
        topk_w = reinterpret_cast<const float *>(ms->topk);
    }

    st = check_buffers(NE, E, cb, pl.scale_layout, tokens, counts, scales, topk_w, permute_tokens, permute_scales,
                       permute_token_idx, expert_token_num, permute_topk_w, workspace, workspace_bytes, inverse);
    if (st != MRR_OK)
        return st;
    if ((topk_w != nullptr) != (pl.has_topk != 0))
        return MRR_ERR_PLAN;
    if ((int64_t)workspace_bytes < pl.workspace_bytes)
        return MRR_ERR_WORKSPACE;

    // plan fields
    const int64_t table_bytes = pl.fuse_scan ? round_up(4 * (NE + 1 + 2 * padded_len(NE)), 128) : 0;
    if (pl.fuse_scan != (NE <= kFusedMaxSegs ? 1 : 0))
        return MRR_ERR_PLAN;
    if (pl.workspace_bytes < kHeaderBytes + (pl.fuse_scan ? 0 : table_workspace_bytes(NE, inverse)))
        return MRR_ERR_PLAN;
    if (pl.grid < 1 || pl.grid > kMaxGrid || pl.block < 64 || pl.block > 1024 || pl.block % 32)
        return MRR_ERR_PLAN;
    if (pl.hints & ~(MRR_HINT_LOAD_EVICT_FIRST | MRR_HINT_STORE_EVICT_FIRST))
        return MRR_ERR_PLAN;
    if (pl.pdl != 0 && pl.pdl != 1)
        return MRR_ERR_PLAN;
    if (pl.epoch < 0 || pl.epoch >= (int64_t)(1ull << (64 - kTicketBits)))
        return MRR_ERR_PLAN;
    int path = pl.path;
    // (multi-source: the sources' alignment is checked on the device, MRR_ERR_SOURCE)
    const bool aligned16 = rb % 16 == 0 && (ms || ((uintptr_t)tokens % 16) == 0) &&
                           ((uintptr_t)permute_tokens % 16) == 0;
    if (path == MRR_PATH_AUTO)
        path = aligned16 ? MRR_PATH_BULK : MRR_PATH_VECTOR;
    if (path == MRR_PATH_BULK && !aligned16)
        path = (pl.path == MRR_PATH_BULK) ? -1 : MRR_PATH_VECTOR;
    if (path != MRR_PATH_BULK && path != MRR_PATH_VECTOR)
        return MRR_ERR_PLAN;
    int64_t smem = table_bytes;
    const int64_t stage = staged_table_bytes(NE);
    if (path == MRR_PATH_BULK) {
        if (pl.stages < 2 || pl.stages > kMaxStages || pl.chunk_bytes < 16 || pl.chunk_bytes % 16 ||
            pl.chunk_bytes > (1 << 20))
            return MRR_ERR_PLAN;
        if (pl.sched != 0 && pl.sched != 1)
            return MRR_ERR_PLAN;
        if (pl.prefetch_chunks < 0 || pl.prefetch_chunks > 64)
            return MRR_ERR_PLAN;
        if (pl.sched == 1) {
            const int64_t nch = (A * rb + pl.chunk_bytes - 1) / pl.chunk_bytes;
            if (pl.static_chunks < 1 || pl.static_chunks > (1 << 20) || nch + 3 * kMaxGrid >= (int64_t)kTicketMask)
                return MRR_ERR_PLAN;
        }
        smem += (int64_t)pl.stages * pl.chunk_bytes;
    }

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    if (smem > optin - 1024)
        return MRR_ERR_PLAN;
    // N*E > 4096: stage the copy kernel's tables when they fit beside what the plan asks for
    const bool stage_tables = !pl.fuse_scan && smem + stage <= optin - 1024;
    if (stage_tables)
        smem += stage;
    const bool scan_in_smem = !pl.fuse_scan && NE <= kSmemScanMaxSegs && scan_smem_bytes(NE) <= optin - 1024;

    uint32_t *status = reinterpret_cast<uint32_t *>(workspace);
    if (NE == 0) {
        // the empty problem: no rows; expert_token_num is all zero
        cudaError_t e = cudaSuccess;
        if (E > 0 && !inverse)
            e = cudaMemsetAsync(expert_token_num, 0, (size_t)(E * cb), stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(status, 0, 8, stream);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return MRR_ERR_CUDA;
        }
        return MRR_OK;
    }

    Params p;
    memset(&p, 0, sizeof(p));
    p.tokens = static_cast<const uint8_t *>(tokens);
    p.out_tokens = static_cast<uint8_t *>(permute_tokens);
    p.total_bytes = A * rb;
    p.row_bytes = rb;
    p.A = A;
    p.counts = counts;
    p.count_is_i64 = pl.count_is_i64;
    p.N = (int)N;
    p.E = (int)E;
    p.NE = (int)NE;
    p.scales = static_cast<const uint8_t *>(scales);
    p.out_scales = scales ? static_cast<uint8_t *>(permute_scales) : nullptr;
    p.scale_row_bytes = sb;
    // vector widths of the side arrays: both pointers aligned to them (multi-source: the output
    // alone; a less aligned rank buffer is read with narrower loads)
    const uintptr_t sc_src = ms ? (uintptr_t)permute_scales : (uintptr_t)scales;
    const uintptr_t tk_src = ms ? (uintptr_t)permute_topk_w : (uintptr_t)topk_w;
    p.scale_w = scales ? widest_width(sc_src, (uintptr_t)permute_scales, sb, 16) : 1;
    p.topk = reinterpret_cast<const uint8_t *>(topk_w);
    p.out_topk = reinterpret_cast<uint8_t *>(permute_topk_w);
    p.topk_w = topk_w ? widest_width(tk_src, (uintptr_t)permute_topk_w, 4, 4) : 4;
    p.idx = permute_token_idx;
    p.idx_type = pl.idx_type;
    p.etn = expert_token_num;
    p.inverse = inverse;
    p.etn_type = (int)expert_token_num_type;
    p.status = status;
    p.chunk_bytes = pl.chunk_bytes;
    p.stages = pl.stages;
    p.hints = pl.hints;
    p.sched = pl.sched;
    p.static_chunks = pl.static_chunks;
    p.prefetch_chunks = path == MRR_PATH_BULK ? pl.prefetch_chunks : 0;
    p.scan_in_smem = scan_in_smem ? 1 : 0;
    p.ptr_off = -1;
    if (ms) {
        // the pointer tables' and capacities' copy in shared memory, behind everything else,
        // when it fits
        const int64_t pb = 8 * N * (1 + (ms->scales ? 1 : 0) + (ms->topk ? 1 : 0) + (ms->rows ? 1 : 0));
        if (round_up(smem, 16) + pb <= optin - 1024) {
            p.ptr_off = (int)round_up(smem, 16);
            smem = p.ptr_off + pb;
        }
        p.multi = 1;
        p.multi_bulk = path == MRR_PATH_BULK ? 1 : 0;
        p.src_tok = reinterpret_cast<const uint8_t *const *>(ms->tokens);
        p.src_sc = reinterpret_cast<const uint8_t *const *>(ms->scales);
        p.src_tk = reinterpret_cast<const uint8_t *const *>(ms->topk);
        p.src_rows = reinterpret_cast<const long long *>(ms->rows);
        p.tokens = nullptr;
        p.scales = nullptr;
        p.topk = nullptr;
    }
    p.ticket = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(workspace) + kTicketOffset);
    p.epoch = (path == MRR_PATH_BULK && pl.sched == 1)
                  ? (pl.epoch ? (unsigned long long)pl.epoch : next_launch_epoch()) : 0ull;
    if (!pl.fuse_scan) {
        uint8_t *ws = static_cast<uint8_t *>(workspace) + kHeaderBytes;
        p.g_row_ex = reinterpret_cast<uint32_t *>(ws);
        p.g_dst_off = reinterpret_cast<uint32_t *>(ws + round_up(4 * (NE + 1), 256));
        if (inverse)
            p.g_col_ex = reinterpret_cast<uint32_t *>(ws + round_up(4 * (NE + 1), 256) +
                                                      round_up(4 * padded_len(NE), 256));
    }

    cudaError_t e = cudaSuccess;
    const bool pdl = pl.pdl != 0;
    if (!pl.fuse_scan)
        e = launch_scan(p, scan_in_smem ? (int)scan_smem_bytes(NE) : 0, stream, device, pdl);
    if (e == cudaSuccess) {
        const int grid = pl.grid, block = pl.block, sm = (int)smem;
        if (ms)
            e = launch_variant<true>(path == MRR_PATH_BULK, pl.fuse_scan != 0, stage_tables, p, grid, block, sm,
                                     stream, device, pdl);
        else
            e = launch_variant<false>(path == MRR_PATH_BULK, pl.fuse_scan != 0, stage_tables, p, grid, block, sm,
                                      stream, device, pdl);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    return MRR_OK;
}

}  // namespace

extern "C" {

mrr_status mrr_v2_plan(int64_t A, int64_t H, mrr_token_dtype dt, int64_t N, int64_t E, int count_is_i64,
                       mrr_scale_layout sl, int64_t scale_cols, int has_topk, int64_t expert_token_num_type,
                       int64_t idx_type, int device, mrr_v2_plan_t *out)
{
    return make_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, has_topk, expert_token_num_type, idx_type,
                     device, 0, out);
}

mrr_status mrr_v2_unroute_plan(int64_t A, int64_t H, mrr_token_dtype dt, int64_t N, int64_t E, int count_is_i64,
                               mrr_scale_layout sl, int64_t scale_cols, int has_topk, int device,
                               mrr_v2_plan_t *out)
{
    return make_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, has_topk, 1, 0, device, 1, out);
}

mrr_status mrr_v2_run_plan(const mrr_v2_plan_t *plan, const void *tokens, mrr_token_dtype dt, const void *counts,
                           const void *scales, const float *topk_w, void *permute_tokens, void *permute_scales,
                           int32_t *permute_token_idx, void *expert_token_num, float *permute_topk_w,
                           int64_t expert_token_num_type, void *workspace, size_t workspace_bytes,
                           mrr_stream_t stream)
{
    return run_plan_impl(plan, nullptr, tokens, dt, counts, scales, topk_w, permute_tokens, permute_scales,
                         permute_token_idx, expert_token_num, permute_topk_w, expert_token_num_type, workspace,
                         workspace_bytes, stream);
}

mrr_status mrr_v2_run_plan_multi(const mrr_v2_plan_t *plan, const void *const *src_tokens,
                                 const void *const *src_scales, const float *const *src_topk_w,
                                 const int64_t *src_rows, mrr_token_dtype dt, const void *counts,
                                 void *permute_tokens, void *permute_scales, int32_t *permute_token_idx,
                                 void *expert_token_num, float *permute_topk_w, int64_t expert_token_num_type,
                                 void *workspace, size_t workspace_bytes, mrr_stream_t stream)
{
    if (!src_tokens)
        return MRR_ERR_NULL;
    if ((uintptr_t)src_rows % 8)
        return MRR_ERR_ALIGN;
    const MultiSrc ms = {src_tokens, src_scales, src_topk_w, src_rows};
    return run_plan_impl(plan, &ms, nullptr, dt, counts, nullptr, nullptr, permute_tokens, permute_scales,
                         permute_token_idx, expert_token_num, permute_topk_w, expert_token_num_type, workspace,
                         workspace_bytes, stream);
}

mrr_status mrr_v2_run_multi(const void *const *src_tokens, const void *const *src_scales,
                            const float *const *src_topk_w, const int64_t *src_rows, mrr_token_dtype dt,
                            int64_t A, int64_t H,
                            const void *counts, int count_is_i64, int64_t N, int64_t E, mrr_scale_layout sl,
                            int64_t scale_cols, void *permute_tokens, void *permute_scales,
                            int32_t *permute_token_idx, void *expert_token_num, float *permute_topk_w,
                            int64_t expert_token_num_type, int64_t idx_type, void *workspace,
                            size_t workspace_bytes, mrr_stream_t stream)
{
    int64_t rb = 0, sb = 0;
    mrr_status st = check_shape(A, H, (int)dt, N, E, count_is_i64, (int)sl, scale_cols, expert_token_num_type,
                                idx_type, &rb, &sb);
    if (st != MRR_OK)
        return st;
    if (!src_tokens)
        return MRR_ERR_NULL;
    if ((uintptr_t)src_rows % 8)
        return MRR_ERR_ALIGN;
    if (sl == MRR_SCALE_NONE)
        src_scales = nullptr;  // "meaningless" output: nothing is read or written
    st = check_buffers(N * E, E, count_is_i64 ? 8 : 4, (int)sl, src_tokens, counts, src_scales, src_topk_w,
                       permute_tokens, permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
                       workspace, workspace_bytes);
    if (st != MRR_OK)
        return st;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    mrr_v2_plan_t plan;
    st = mrr_v2_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, src_topk_w != nullptr, expert_token_num_type,
                     idx_type, device, &plan);
    if (st != MRR_OK)
        return st;
    plan.path = MRR_PATH_AUTO;
    return mrr_v2_run_plan_multi(&plan, src_tokens, src_scales, src_topk_w, src_rows, dt, counts, permute_tokens,
                                 permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
                                 expert_token_num_type, workspace, workspace_bytes, stream);
}

mrr_status mrr_v2_run(const void *tokens, mrr_token_dtype dt, int64_t A, int64_t H, const void *counts,
                      int count_is_i64, int64_t N, int64_t E, const void *scales, mrr_scale_layout sl,
                      int64_t scale_cols, const float *topk_w, void *permute_tokens, void *permute_scales,
                      int32_t *permute_token_idx, void *expert_token_num, float *permute_topk_w,
                      int64_t expert_token_num_type, int64_t idx_type, void *workspace, size_t workspace_bytes,
                      mrr_stream_t stream)
{
    int64_t rb = 0, sb = 0;
    mrr_status st = check_shape(A, H, (int)dt, N, E, count_is_i64, (int)sl, scale_cols, expert_token_num_type,
                                idx_type, &rb, &sb);
    if (st != MRR_OK)
        return st;
    if (sl == MRR_SCALE_NONE)
        scales = nullptr;  // "meaningless" output: nothing is read or written
    st = check_buffers(N * E, E, count_is_i64 ? 8 : 4, (int)sl, tokens, counts, scales, topk_w, permute_tokens,
                       permute_scales, permute_token_idx, expert_token_num, permute_topk_w, workspace,
                       workspace_bytes);
    if (st != MRR_OK)
        return st;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    mrr_v2_plan_t plan;
    st = mrr_v2_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, topk_w != nullptr, expert_token_num_type,
                     idx_type, device, &plan);
    if (st != MRR_OK)
        return st;
    plan.path = MRR_PATH_AUTO;
    return mrr_v2_run_plan(&plan, tokens, dt, counts, scales, topk_w, permute_tokens, permute_scales,
                           permute_token_idx, expert_token_num, permute_topk_w, expert_token_num_type, workspace,
                           workspace_bytes, stream);
}

mrr_status mrr_v1_run(const void *tokens, mrr_token_dtype dt, int64_t A, int64_t H, const void *counts,
                      int count_is_i64, int64_t N, int64_t E, const float *per_token_scales, void *permute_tokens,
                      float *permute_per_token_scales, int32_t *permute_token_idx, void *expert_token_num,
                      int64_t expert_token_num_type, int64_t idx_type, void *workspace, size_t workspace_bytes,
                      mrr_stream_t stream)
{
    // the v1 subset ("torch_npu.npu_moe_re_routing" page, section 参数说明)
    if (dt != MRR_F16 && dt != MRR_BF16 && dt != MRR_I8)
        return MRR_ERR_DTYPE;
    if ((expert_token_num_type != 0 && expert_token_num_type != 1) || (idx_type != 0 && idx_type != 1))
        return MRR_ERR_ATTR;
    if (expert_token_num_type != 1 || idx_type != 0)
        return MRR_ERR_UNSUPPORTED;
    const bool sc = per_token_scales != nullptr;
    return mrr_v2_run(tokens, dt, A, H, counts, count_is_i64, N, E, per_token_scales,
                      sc ? MRR_SCALE_F32_A : MRR_SCALE_NONE, sc ? 1 : 0, nullptr, permute_tokens,
                      sc ? permute_per_token_scales : nullptr, permute_token_idx, expert_token_num, nullptr, 1, 0,
                      workspace, workspace_bytes, stream);
}

mrr_status mrr_v2_unroute(const void *permute_tokens, mrr_token_dtype dt, int64_t A, int64_t H, const void *counts,
                          int count_is_i64, int64_t N, int64_t E, const void *permute_scales, mrr_scale_layout sl,
                          int64_t scale_cols, const float *permute_topk_w, void *tokens, void *scales,
                          float *topk_w, void *workspace, size_t workspace_bytes, mrr_stream_t stream)
{
    int64_t rb = 0, sb = 0;
    mrr_status st = check_shape(A, H, (int)dt, N, E, count_is_i64, (int)sl, scale_cols, 1, 0, &rb, &sb);
    if (st != MRR_OK)
        return st;
    if (sl == MRR_SCALE_NONE)
        permute_scales = nullptr;
    st = check_buffers(N * E, E, count_is_i64 ? 8 : 4, (int)sl, permute_tokens, counts, permute_scales,
                       permute_topk_w, tokens, scales, nullptr, nullptr, topk_w, workspace, workspace_bytes, 1);
    if (st != MRR_OK)
        return st;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    mrr_v2_plan_t plan;
    st = mrr_v2_unroute_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, permute_topk_w != nullptr, device,
                             &plan);
    if (st != MRR_OK)
        return st;
    plan.path = MRR_PATH_AUTO;
    return mrr_v2_run_plan(&plan, permute_tokens, dt, counts, permute_scales, permute_topk_w, tokens, scales,
                           nullptr, nullptr, topk_w, 1, workspace, workspace_bytes, stream);
}

mrr_status mrr_v2_offsets_host(const void *counts, int count_is_i64, int64_t N, int64_t E, int64_t A,
                               int64_t *src_offset, int64_t *dst_offset, int64_t *expert_token_num)
{
    if (!counts && N * E > 0)
        return MRR_ERR_NULL;
    if ((count_is_i64 != 0 && count_is_i64 != 1))
        return MRR_ERR_DTYPE;
    if (N < 0 || E < 0 || A < 0 || A > INT32_MAX || (N > 0 && E > INT32_MAX / N) || N > INT32_MAX)
        return MRR_ERR_SHAPE;
    auto count = [&](int64_t i, int64_t j) -> int64_t {
        return count_is_i64 ? static_cast<const int64_t *>(counts)[i * E + j]
                            : (int64_t) static_cast<const int32_t *>(counts)[i * E + j];
    };
    // the same checks the kernels make: every count > 0 and no larger than A, Sum = A
    int64_t sum = 0;
    for (int64_t q = 0; q < N * E; ++q) {
        const int64_t c = count(q / E, q % E);
        if (c <= 0)
            return MRR_ERR_COUNT_NONPOS;
        if (c > A)
            return MRR_ERR_COUNT_SUM;
        sum += c;
        if (sum > A)
            return MRR_ERR_COUNT_SUM;
    }
    if (sum != A)
        return MRR_ERR_COUNT_SUM;
    int64_t run = 0;  // SrcOffset: rank outer, expert inner
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < E; ++j) {
            if (src_offset)
                src_offset[i * E + j] = run;
            run += count(i, j);
        }
    run = 0;  // DstOffset: expert outer, rank inner; expert j's block is its count
    for (int64_t j = 0; j < E; ++j) {
        const int64_t start = run;
        for (int64_t i = 0; i < N; ++i) {
            if (dst_offset)
                dst_offset[i * E + j] = run;
            run += count(i, j);
        }
        if (expert_token_num)
            expert_token_num[j] = run - start;
    }
    return MRR_OK;
}

mrr_status mrr_v2_read_status(const void *workspace, size_t workspace_bytes, mrr_stream_t stream_)
{
    if (!workspace)
        return MRR_ERR_NULL;
    if (workspace_bytes < (size_t)kStatusBytes)
        return MRR_ERR_WORKSPACE;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    uint32_t words[kStatusWords];
    if (cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    uint32_t flags = words[0];
    uint32_t n = words[1];
    if (n > (uint32_t)kMaxGrid)
        n = kMaxGrid;
    for (uint32_t b = 0; b < n; ++b)
        flags |= words[2 + b];
    if (flags & kFlagNonPos)
        return MRR_ERR_COUNT_NONPOS;
    if (flags & kFlagSum)
        return MRR_ERR_COUNT_SUM;
    if (flags & kFlagTimeout)
        return MRR_ERR_TIMEOUT;
    if (flags & kFlagBadIndex)
        return MRR_ERR_INDEX;
    if (flags & kFlagSource)
        return MRR_ERR_SOURCE;
    if (flags & kFlagDest)
        return MRR_ERR_DEST;
    return MRR_OK;
}

}  // extern "C"
