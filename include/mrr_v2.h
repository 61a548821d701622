/*
 * mrr_v2.h -- C ABI of the GB300 (sm_103a) MoE re-routing library.
 *
 * The op (MoeReRoutingV2) runs after the expert-parallel AlltoAll.  The A token rows a GPU
 * received arrive rank-major: one contiguous segment per (source rank i, expert j), sized by
 * the count matrix counts[N,E].  The op lays them out expert-major, moves the per-token scales
 * and top-k weights with them, and emits the permutation index and the per-expert counts.
 *
 * Definition (the "CANN ops-transformer MoeReRoutingV2" article, m.nlpx.cn/news/59074):
 *   - section 计算公式: segment (i,j) moves from SrcOffset(i,j) to DstOffset(i,j), where
 *     SrcOffset is the sum of all counts before (i,j) walking rank-outer (row-major) and
 *     DstOffset the sum of all counts before (i,j) walking expert-outer (column-major);
 *     permute_tokens[Dst+k] = tokens[Src+k], and the same for per_token_scales and
 *     expert_topk_weight, 0 <= k < counts[i,j].
 *   - section 参数说明 (parameter table) and 参数取值细节: input/output shapes and dtypes,
 *     idx_type 0 = gather index (permute_token_idx[d] = s), 1 = scatter index
 *     (permute_token_idx[s] = d); expert_token_num_type 1 = per-expert count.
 *   - section 约束说明 (constraints): Sum(counts) = A, 0 < H < 16384, every count > 0,
 *     only expert_token_num_type = 1 is supported (this library also offers 0, cumsum mode).
 *   - section 算子 IR 原型: permute_token_idx is INT32; attribute defaults
 *     expert_token_num_type = 1, idx_type = 0.
 *   - section InferShape 与 InferDtype: output shapes/dtypes follow the inputs; absent scales
 *     give a meaningless [A] float32 output, absent top-k weights an empty output.
 *
 * Conventions for every entry point:
 *   - All buffer pointers are DEVICE pointers unless stated otherwise.  The caller owns every
 *     buffer, including the workspace.  The library allocates no device memory.
 *   - Payload rows are moved as raw bytes: nothing is converted, so every output is
 *     bit-identical to its input row (NaN payloads, fp8/e8m0/hifloat8/fp4 codes included).
 *   - Inputs and outputs must not overlap.
 *   - mrr_v2_run / mrr_v2_run_plan only enqueue work on `stream` and return after host-side
 *     validation.  Errors found on the host are returned at once and nothing is enqueued.
 *     Errors that depend on the count VALUES (a count <= 0, Sum != A) are found on the GPU:
 *     the outputs are then left unspecified and mrr_v2_read_status reports the error.
 *   - Calls on different streams must use different workspaces.
 *   - The calls may be captured in a CUDA graph (stream capture) and the graph replayed: each
 *     replay moves every row again (the workspace's chunk counter recognises a finished earlier
 *     run of the same captured launch).  After a replay that reported MRR_ERR_TIMEOUT, zero the
 *     workspace's counter word (bytes 4096..4103) or use a fresh workspace before replaying.
 */
#ifndef MRR_V2_H
#define MRR_V2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle: the same type as cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st *mrr_stream_t;

typedef enum mrr_status {
    MRR_OK = 0,
    MRR_ERR_NULL = 1,          /* a required pointer is NULL                                   */
    MRR_ERR_SHAPE = 2,         /* A, H, N, E, scale_cols out of range (see mrr_v2_plan)         */
    MRR_ERR_DTYPE = 3,         /* unknown token dtype or scale layout code                     */
    MRR_ERR_ATTR = 4,          /* expert_token_num_type or idx_type not in {0, 1}              */
    MRR_ERR_UNSUPPORTED = 5,   /* an option the v1 entry point does not support                */
    MRR_ERR_TOPK_PAIR = 6,     /* exactly one of expert_topk_weight / permute_topk_weight given */
    MRR_ERR_WORKSPACE = 7,     /* workspace NULL, misaligned or smaller than workspace_bytes   */
    MRR_ERR_CUDA = 8,          /* a CUDA runtime call failed (no device, launch error, ...)    */
    MRR_ERR_ALIGN = 9,         /* counts / index / expert_token_num pointer not aligned to its type */
    MRR_ERR_PLAN = 10,         /* a plan passed to mrr_v2_run_plan is inconsistent             */
    /* found on the GPU; reported by mrr_v2_read_status */
    MRR_ERR_COUNT_NONPOS = 16, /* some counts[i,j] <= 0                                        */
    MRR_ERR_COUNT_SUM = 17,    /* Sum(counts) != A (or a single count > A)                     */
    MRR_ERR_TIMEOUT = 18,      /* a bounded wait inside the copy kernel gave up                */
    MRR_ERR_INDEX = 19,        /* gating top-k: an input_ids / tid2eid value out of range     */
    MRR_ERR_SOURCE = 20,       /* multi-source form: a per-rank source pointer is NULL, or a
                                  token source is not 16-byte aligned on the bulk path        */
    MRR_ERR_DEST = 21          /* push form: a receiver's buffer pointer is NULL, or a row
                                  would land past the rows its buffer holds                    */
} mrr_status;

/* Token element types (section 参数说明).  Only the width matters: rows move as bytes.
 * FP4 types are packed two per byte, so H must be even for them (row bytes = H / 2). */
typedef enum mrr_token_dtype {
    MRR_F16 = 0,      /* 16 bit */
    MRR_BF16 = 1,     /* 16 bit */
    MRR_I8 = 2,       /*  8 bit */
    MRR_F8E5M2 = 3,   /*  8 bit */
    MRR_F8E4M3FN = 4, /*  8 bit */
    MRR_HIF8 = 5,     /*  8 bit */
    MRR_F4E2M1 = 6,   /*  4 bit */
    MRR_F4E1M2 = 7    /*  4 bit */
} mrr_token_dtype;

/* per_token_scales layouts (section 参数说明).  scale_cols = elements per scale row. */
typedef enum mrr_scale_layout {
    MRR_SCALE_NONE = 0,     /* no scales; scale_cols ignored; permute_scales not written     */
    MRR_SCALE_F32_A = 1,    /* [A] float32;            scale_cols must be 1                  */
    MRR_SCALE_F32_AS = 2,   /* [A, S] float32;         scale_cols = S >= 1                   */
    MRR_SCALE_E8M0_AK2 = 3  /* [A, K/64, 2] e8m0 bytes; scale_cols = (K/64)*2, even, >= 2    */
} mrr_scale_layout;

/* copy paths of the token move */
#define MRR_PATH_AUTO 0    /* run picks: BULK when rows and base pointers are 16-byte aligned */
#define MRR_PATH_BULK 1    /* cp.async.bulk global->shared->global, one driver thread per CTA  */
#define MRR_PATH_VECTOR 2  /* all threads, widest aligned vector loads/stores (any alignment) */

/* bulk-path L2 cache hints (plan.hints bits) */
#define MRR_HINT_LOAD_EVICT_FIRST 1   /* token loads marked evict-first in L2  */
#define MRR_HINT_STORE_EVICT_FIRST 2  /* token stores marked evict-first in L2 */

/* Launch plan: plain data, owned by the caller.  mrr_v2_plan fills it; a caller may change the
 * tuning fields (path, grid, block, chunk_bytes, stages) and pass it to mrr_v2_run_plan, which
 * checks them again. */
typedef struct mrr_v2_plan {
    int64_t A, H, N, E;
    int64_t row_bytes;        /* bytes per token row: H * bits / 8                          */
    int64_t scale_row_bytes;  /* bytes per scale row; 0 without scales                      */
    int64_t workspace_bytes;  /* device scratch mrr_v2_run needs (>= 4352: status + counter) */
    int32_t count_is_i64;
    int32_t scale_layout;
    int32_t has_topk;
    int32_t idx_type;
    int32_t fuse_scan;        /* 1: every CTA scans the counts itself (N*E <= 4096)
                                 0: a one-CTA scan kernel writes the offsets to the workspace */
    int32_t path;             /* MRR_PATH_*                                                  */
    int32_t grid;             /* CTAs of the copy kernel (<= 1022)                            */
    int32_t block;            /* threads per CTA (multiple of 32, 64..1024)                   */
    int32_t chunk_bytes;      /* bulk path: bytes per pipeline stage (multiple of 16)         */
    int32_t stages;           /* bulk path: pipeline depth (2..8)                             */
    int32_t hints;            /* bulk path: MRR_HINT_* bits                                   */
    int32_t sched;            /* bulk path: 0 = each CTA an equal slice of the token bytes;
                                 1 = static_chunks chunks per CTA, then chunks claimed from a
                                 counter in the workspace (balances uneven CTA speeds)        */
    int32_t static_chunks;    /* bulk path, sched 1: chunks per CTA before claiming           */
    int32_t pdl;              /* 1: launch with programmatic stream serialization, so the next
                                 launch on the stream is scheduled while this one drains; the
                                 kernels wait for their predecessor before any global access */
    int32_t direction;        /* 0: rank-major -> expert-major (mrr_v2_plan);
                                 1: expert-major -> rank-major (mrr_v2_unroute_plan)          */
    int32_t smem_bytes;       /* dynamic shared memory per CTA                                */
    int32_t num_sms;          /* SMs on the device the plan was made for                      */
    int32_t prefetch_chunks;  /* bulk path: chunks each CTA asks L2 to prefetch while it scans
                                 the counts (its static chunks past the ring first, then its
                                 share of the first counter-served chunks); 0 = none, <= 64   */
    int64_t epoch;            /* bulk path, sched 1: the tag this launch writes into the
                                 workspace's chunk counter, 1 .. 2^40 - 1; 0 (what the plan
                                 functions set) draws a fresh tag for every call.  A fixed tag
                                 lets a caller (a test) plant a counter value the launch must
                                 reject: a ticket beyond the launch's last one is reported as
                                 MRR_ERR_TIMEOUT and the CTAs that drew it stop at once        */
} mrr_v2_plan_t;

/*
 * mrr_v2_plan -- host only, enqueues nothing, allocates nothing.
 *   Validates the shape/attribute arguments (the same checks mrr_v2_run makes, except for
 *   pointers) and fills *out with the launch plan and the workspace size for `device`.
 *   A: rows (0 <= A <= INT32_MAX; A = 0 only with N*E = 0, the empty problem);
 *   H: elements per token row, 0 < H < 16384, even for FP4 dtypes;
 *   N, E: count-matrix rows (ranks) and columns (experts), >= 0;
 *   count_is_i64: counts are int64 (1) or int32 (0); expert_token_num has the same type;
 *   sl, scale_cols: the scale layout and elements per scale row (see mrr_scale_layout);
 *   has_topk: expert_topk_weight / permute_topk_weight given;
 *   expert_token_num_type: 1 = per-expert count, 0 = cumsum mode (an extension: the pages list
 *   it but support only 1; here it is the inclusive prefix over experts, last entry A);
 *   idx_type 0 or 1.
 *   Returns MRR_ERR_CUDA when the device cannot be queried (e.g. no GPU).
 */
mrr_status mrr_v2_plan(int64_t A, int64_t H, mrr_token_dtype dt, int64_t N, int64_t E,
                       int count_is_i64, mrr_scale_layout sl, int64_t scale_cols, int has_topk,
                       int64_t expert_token_num_type, int64_t idx_type, int device,
                       mrr_v2_plan_t *out);

/*
 * mrr_v2_run -- enqueue one re-routing on `stream` (current device).
 *   tokens          [A, H] dt, row-major, rank-major segments            (read)
 *   counts          [N, E] int32 or int64 (count_is_i64), row = rank      (read)
 *   scales          per the layout, or NULL with MRR_SCALE_NONE          (read)
 *   topk_w          [A, 1] float32, or NULL                              (read)
 *   permute_tokens  [A, H] dt                                            (written)
 *   permute_scales  same shape as scales; may be NULL without scales     (written if scales)
 *   permute_token_idx [A] int32, gather (idx_type 0) or scatter (1) index (written)
 *   expert_token_num  [E] counts' type, tokens per expert                (written)
 *   permute_topk_w  [A, 1] float32; NULL exactly when topk_w is NULL     (written if given)
 *   workspace       >= plan.workspace_bytes device bytes, 256-byte aligned, caller-owned;
 *                   it holds the status words read by mrr_v2_read_status, the chunk counter
 *                   of the bulk path and, for N*E > 4096, the scanned offsets.  It needs no
 *                   initialisation: each call tags the counter with its own epoch.
 * Host-side errors return before anything is enqueued.  The empty problem (N*E = 0, A = 0)
 * only zero-fills expert_token_num.
 */
mrr_status mrr_v2_run(const void *tokens, mrr_token_dtype dt, int64_t A, int64_t H,
                      const void *counts, int count_is_i64, int64_t N, int64_t E,
                      const void *scales, mrr_scale_layout sl, int64_t scale_cols,
                      const float *topk_w,
                      void *permute_tokens, void *permute_scales, int32_t *permute_token_idx,
                      void *expert_token_num, float *permute_topk_w,
                      int64_t expert_token_num_type, int64_t idx_type,
                      void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v2_run_plan -- as mrr_v2_run, with the launch taken from *plan (made by mrr_v2_plan for
 * the same shapes, possibly with edited tuning fields).  The shape fields of the plan must
 * match the arguments (else MRR_ERR_PLAN).  MRR_PATH_BULK with unaligned rows or pointers
 * returns MRR_ERR_PLAN.
 */
mrr_status mrr_v2_run_plan(const mrr_v2_plan_t *plan,
                           const void *tokens, mrr_token_dtype dt, const void *counts,
                           const void *scales, const float *topk_w,
                           void *permute_tokens, void *permute_scales, int32_t *permute_token_idx,
                           void *expert_token_num, float *permute_topk_w,
                           int64_t expert_token_num_type,
                           void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v2_read_status -- synchronise `stream`, read the status words of the last run that used
 * `workspace`, and return MRR_OK or the device-detected error (MRR_ERR_COUNT_NONPOS,
 * MRR_ERR_COUNT_SUM, MRR_ERR_TIMEOUT, MRR_ERR_SOURCE), or MRR_ERR_CUDA if the copy back fails.
 * workspace_bytes must be >= 4096.
 */
mrr_status mrr_v2_read_status(const void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v1_run -- the v1 op (torch_npu.npu_moe_re_routing page: 接口原型, 参数说明, 输出说明): the
 * same move restricted to what v1 supports, with four outputs and no top-k weights.
 *   tokens            [A, H] float16 / bfloat16 / int8 only (else MRR_ERR_DTYPE)
 *   per_token_scales  [A] float32, or NULL; permute_per_token_scales [A] float32, written only
 *                     when per_token_scales is given (the page: otherwise the output is invalid)
 *   expert_token_num_type must be 1 and idx_type 0 (other values in {0, 1}:
 *   MRR_ERR_UNSUPPORTED, as the page states only these are supported).
 * Workspace: plan.workspace_bytes of mrr_v2_plan for the same shapes.  Otherwise as mrr_v2_run.
 */
mrr_status mrr_v1_run(const void *tokens, mrr_token_dtype dt, int64_t A, int64_t H, const void *counts,
                      int count_is_i64, int64_t N, int64_t E, const float *per_token_scales,
                      void *permute_tokens, float *permute_per_token_scales,
                      int32_t *permute_token_idx, void *expert_token_num,
                      int64_t expert_token_num_type, int64_t idx_type,
                      void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v2_unroute_plan -- host only: the launch plan of mrr_v2_unroute, which moves the rows
 * back (direction 1).  Same argument checks as mrr_v2_plan; no attributes (the inverse move
 * writes no index and no per-expert counts).
 */
mrr_status mrr_v2_unroute_plan(int64_t A, int64_t H, mrr_token_dtype dt, int64_t N, int64_t E,
                               int count_is_i64, mrr_scale_layout sl, int64_t scale_cols, int has_topk,
                               int device, mrr_v2_plan_t *out);

/*
 * mrr_v2_unroute -- the inverse move, for the combine side of the MoE layer: rows laid out
 * expert-major (by mrr_v2_run, or expert outputs in that order) go back to the rank-major order
 * they arrived in, so they can be returned to their source ranks.  The pages place the op before
 * the expert FFN and name finalize/combine ops after it ("CANN ops-transformer MoeReRoutingV2"
 * article, section 数据流定位); the inverse reuses the same segments and offsets (section
 * 计算公式):  tokens[SrcOffset(i,j) + k] = permute_tokens[DstOffset(i,j) + k],  and the same for
 * the scale rows and top-k weights, 0 <= k < counts[i,j].
 *   permute_tokens  [A, H] dt, expert-major                              (read)
 *   counts          [N, E] int32 or int64, the same matrix as the forward move (read)
 *   permute_scales  per the layout, or NULL with MRR_SCALE_NONE          (read)
 *   permute_topk_w  [A, 1] float32, or NULL                              (read)
 *   tokens          [A, H] dt, rank-major                                (written)
 *   scales          same shape as permute_scales; written when given
 *   topk_w          [A, 1] float32; NULL exactly when permute_topk_w is NULL
 *   workspace       >= plan.workspace_bytes of mrr_v2_unroute_plan (N*E > 4096 needs one more
 *                   offset table than the forward move)
 * Errors and status reporting are those of mrr_v2_run.  mrr_v2_run_plan also runs it, given a
 * plan with direction 1: its tokens / scales / topk_w arguments are then the expert-major
 * inputs, permute_* the rank-major outputs, and permute_token_idx / expert_token_num unused.
 */
mrr_status mrr_v2_unroute(const void *permute_tokens, mrr_token_dtype dt, int64_t A, int64_t H,
                          const void *counts, int count_is_i64, int64_t N, int64_t E,
                          const void *permute_scales, mrr_scale_layout sl, int64_t scale_cols,
                          const float *permute_topk_w, void *tokens, void *scales, float *topk_w,
                          void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v2_run_multi -- the same move with the received rows still in one buffer per source rank:
 * the receive side of the expert-parallel dispatch fused with the re-routing.  The dispatch
 * ("torch_npu.npu_moe_distribute_dispatch" page: expand_x, ep_recv_counts) delivers each peer's
 * rows, and the V2 article (section 数据流定位 / 在 MoE 网络中的角色) re-lays them out
 * expert-major.  When the rows land in per-peer receive slots (for example fixed-capacity slots,
 * or one buffer per peer), this call reads them there directly: rank i's segment (i, j) moves
 * from its slot to DstOffset(i, j), so the rank-major concatenation is never written and read
 * again.  The results equal mrr_v2_run on the concatenation of the N buffers in rank order.
 *   src_tokens   DEVICE array of N device pointers; src_tokens[i] holds rank i's rows, that is
 *                rows SrcOffset(i, 0) .. SrcOffset(i, 0) + sum_j counts[i, j] - 1 of the
 *                rank-major order, as [rows_i, H] dt from the pointer on       (read)
 *   src_scales   DEVICE array of N device pointers to rank i's scale rows in the layout `sl`
 *                (same row order), or NULL with MRR_SCALE_NONE                 (read)
 *   src_topk_w   DEVICE array of N device pointers to rank i's [rows_i] float32 top-k weights,
 *                or NULL; NULL exactly when permute_topk_w is NULL            (read)
 *   src_rows     DEVICE array [N] int64: the rows rank i's buffers hold (for example the
 *                capacity of its receive slot), or NULL.  When given, a count matrix whose row
 *                i sums to more than src_rows[i] is refused (MRR_ERR_SOURCE, nothing moved), so
 *                counts that arrive over the network can never make the kernel read past a
 *                buffer.  With NULL the counts are trusted for the buffers' extents.
 *   every other argument as mrr_v2_run: counts [N, E] in device memory, the five outputs in
 *   expert-major order, permute_token_idx numbering rows in the rank-major order, the workspace
 *   of mrr_v2_plan for the same shapes.
 * The pointer tables live in device memory, so the host cannot check them: the kernels do,
 * before they read any source, and report MRR_ERR_SOURCE through mrr_v2_read_status (nothing is
 * then moved) when a pointer is NULL, a rank's rows exceed src_rows, or, on the bulk path (row
 * bytes a multiple of 16 and a 16-byte aligned permute_tokens), a token pointer is not 16-byte
 * aligned.  Use
 * mrr_v2_run_plan_multi with MRR_PATH_VECTOR for token buffers of any alignment.  Scale and
 * top-k pointers may have any alignment.  The buffers must not overlap the outputs.
 */
mrr_status mrr_v2_run_multi(const void *const *src_tokens, const void *const *src_scales,
                            const float *const *src_topk_w, const int64_t *src_rows,
                            mrr_token_dtype dt, int64_t A, int64_t H,
                            const void *counts, int count_is_i64, int64_t N, int64_t E,
                            mrr_scale_layout sl, int64_t scale_cols,
                            void *permute_tokens, void *permute_scales, int32_t *permute_token_idx,
                            void *expert_token_num, float *permute_topk_w,
                            int64_t expert_token_num_type, int64_t idx_type,
                            void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v2_run_plan_multi -- mrr_v2_run_multi with the launch taken from *plan (mrr_v2_plan for
 * the same shapes, tuning fields possibly edited; direction must be 0).  Same argument rules.
 */
mrr_status mrr_v2_run_plan_multi(const mrr_v2_plan_t *plan, const void *const *src_tokens,
                                 const void *const *src_scales, const float *const *src_topk_w,
                                 const int64_t *src_rows, mrr_token_dtype dt, const void *counts,
                                 void *permute_tokens, void *permute_scales, int32_t *permute_token_idx,
                                 void *expert_token_num, float *permute_topk_w,
                                 int64_t expert_token_num_type,
                                 void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/*
 * mrr_v2_offsets_host -- host only, enqueues nothing: the offsets of the move for a count matrix
 * in HOST memory ("CANN ops-transformer MoeReRoutingV2" article, section 计算公式), for the
 * push form of the fused receive.  There each sender writes its segments straight into the
 * receiver's expert-major buffer, so it needs the receiver's DstOffset of its own row before any
 * row moves (the receiver computes it from the counts it received and sends row i back to
 * sender i; see moe_expert_token_gb300.ep).
 *   counts            [N, E] int32 or int64 (count_is_i64), HOST memory          (read)
 *   src_offset        [N, E] int64 or NULL: SrcOffset(i, j), rank-major prefix   (written)
 *   dst_offset        [N, E] int64 or NULL: DstOffset(i, j), expert-major prefix (written)
 *   expert_token_num  [E] int64 or NULL: tokens per expert                       (written)
 * Returns MRR_ERR_COUNT_NONPOS / MRR_ERR_COUNT_SUM for counts the kernels would refuse (a count
 * <= 0, Sum != A), writing nothing; MRR_ERR_SHAPE / MRR_ERR_DTYPE / MRR_ERR_NULL for bad
 * arguments.  N*E = 0 with A = 0 is the empty problem.
 */
mrr_status mrr_v2_offsets_host(const void *counts, int count_is_i64, int64_t N, int64_t E, int64_t A,
                               int64_t *src_offset, int64_t *dst_offset, int64_t *expert_token_num);

/*
 * mrr_v2_push -- the push form of the fused receive, one sender's side: this rank writes the rows
 * it sends straight into every receiver's expert-major buffers, so no receiver writes them
 * rank-major and reads them back.  Receiver r's count matrix ("CANN ops-transformer
 * MoeReRoutingV2" article, 参数说明: expert_token_num_per_rank; the dispatch's ep_recv_counts on
 * the "torch_npu.npu_moe_distribute_dispatch" page) has this sender's row i; the receiver
 * computes DstOffset_r(i, j) and SrcOffset_r(i, j) from it (计算公式; mrr_v2_offsets_host) and
 * returns row i to this sender.  Rows move as bytes, scales and top-k weights with them.
 *   send_tokens       [S, H] dt, this sender's rows: segment (r, j) -- the rows for receiver r's
 *                     local expert j -- at rows SendOffset(r, j), the row-major exclusive prefix of
 *                     send_counts (receiver outer)                                    (read)
 *   send_scales       [S] / [S, scale_cols] rows in the layout `sl`, or NULL with MRR_SCALE_NONE
 *   send_topk_w       [S] float32, or NULL (then out_topk_w must be NULL)              (read)
 *   send_counts       [R, E] int32 / int64 (count_is_i64) in device memory: rows this sender
 *                     sends to receiver r for expert j, each > 0, summing to S        (read)
 *   dst_offsets       [R, E] int64, device: DstOffset_r(i, j), the expert-major row in receiver
 *                     r's buffers where segment (r, j) starts                          (read)
 *   recv_src_offsets  [R, E] int64, device: SrcOffset_r(i, j), the segment's first row in receiver
 *                     r's rank-major order (for its gather index), or NULL with idx_out NULL
 *   out_tokens        DEVICE array of R device pointers: receiver r's [rows_r, H] expert-major
 *                     token buffer (this GPU's memory or a peer's)                      (written)
 *   out_scales, out_topk_w   DEVICE arrays of R pointers, or NULL when the sends have none
 *   idx_out           DEVICE array of R pointers to receiver r's int32 gather index
 *                     (permute_token_idx, idx_type 0: idx[d] = its rank-major row), or NULL
 *   out_rows          DEVICE array [R] int64: the rows receiver r's buffers hold, or NULL (not
 *                     checked); a row that would land at or past it is not written
 *   workspace         at least 4096 bytes of device memory for the status words; the device's
 *                     findings are read with mrr_v2_read_status: MRR_ERR_COUNT_NONPOS,
 *                     MRR_ERR_COUNT_SUM (nothing moved), MRR_ERR_DEST (a NULL receiver pointer
 *                     or a row past out_rows: those rows are skipped)
 * R * E must be at most 4096 (MRR_ERR_SHAPE otherwise), and S, H, dt, sl, scale_cols follow
 * mrr_v2_plan's rules with S in the place of A.  Each receiver's expert_token_num comes from its
 * own count matrix.  Enqueues one launch on `stream` and allocates nothing.  The writes use plain
 * stores of up to 16 bytes per thread, whatever memory the pointers name: no bulk copy and no
 * multicast.  Across senders the segments are disjoint, so the senders' launches need no order
 * among themselves.
 */
mrr_status mrr_v2_push(const void *send_tokens, const void *send_scales, const float *send_topk_w,
                       mrr_token_dtype dt, int64_t S, int64_t H, const void *send_counts, int count_is_i64,
                       int64_t R, int64_t E, mrr_scale_layout sl, int64_t scale_cols,
                       const int64_t *dst_offsets, const int64_t *recv_src_offsets,
                       void *const *out_tokens, void *const *out_scales, float *const *out_topk_w,
                       int32_t *const *idx_out, const int64_t *out_rows,
                       void *workspace, size_t workspace_bytes, mrr_stream_t stream);

/* mrr_status_str -- static, human-readable name of a status code (never NULL). */
const char *mrr_status_str(mrr_status s);

/* Limits of the fixed scratch used by mrr_v2_run_noalloc. */
#define MRR_NOALLOC_MAX_SEGMENTS 16384   /* largest N*E it accepts                          */
#define MRR_NOALLOC_SCRATCH_BYTES 137984 /* device bytes it holds on every GPU that loads
                                            the library, until the process exits            */

/*
 * mrr_v2_run_noalloc -- mrr_v2_run without a caller-provided workspace.  The paper has no
 * counterpart to this entry point.
 *
 * Intended for callers that cannot allocate device memory at the call site, for example:
 *   - a plugin whose host framework owns all device memory and passes it only the input and
 *     output tensors;
 *   - a serving loop whose device memory budget is fixed when it starts;
 *   - code that must not call cudaMalloc/cudaFree, which can synchronise the whole device and
 *     stall work on other streams.
 * It allocates nothing and calls no allocating routine.  Its scratch is one fixed array of
 * MRR_NOALLOC_SCRATCH_BYTES in the library's device memory, and that array holds the status
 * words and, for N*E > 4096, the two offset tables.
 *
 * The arguments and outputs are those of mrr_v2_run.  The caller still passes every input and
 * output buffer.
 *   - N*E > MRR_NOALLOC_MAX_SEGMENTS returns MRR_ERR_WORKSPACE before anything is enqueued.
 *   - wait_and_check != 0 synchronises `stream` after enqueuing and returns any error the device
 *     found, as mrr_v2_read_status does.  With 0 the call only enqueues, and device-detected
 *     count errors go unreported.
 *   - The first call on each device looks up the array's device address, with that device
 *     current.  Make that first call before any stream capture.
 *   - Every call on a device uses the same array, which keeps the last call's contents.  Each
 *     call rewrites the status words and tables it reads, so nothing needs clearing.  Calls
 *     that overlap on the GPU (e.g. on two streams at once) race on the array and may report
 *     wrong statuses or move rows wrongly: serialise them.
 */
mrr_status mrr_v2_run_noalloc(const void *tokens, mrr_token_dtype dt, int64_t A, int64_t H,
                              const void *counts, int count_is_i64, int64_t N, int64_t E,
                              const void *scales, mrr_scale_layout sl, int64_t scale_cols,
                              const float *topk_w,
                              void *permute_tokens, void *permute_scales, int32_t *permute_token_idx,
                              void *expert_token_num, float *permute_topk_w,
                              int64_t expert_token_num_type, int64_t idx_type,
                              int wait_and_check, mrr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MRR_V2_H */
