// mrr_v2_run_noalloc: the re-routing op for callers that cannot allocate device memory.
//
// mrr_v2_run needs a caller-provided device workspace (status words, and for N*E > 4096 the two
// offset tables).  Some callers cannot provide one: a plugin that a host framework hands only
// its input and output tensors, a serving loop whose device memory budget is fixed at start-up,
// or code that must avoid cudaMalloc/cudaFree because those calls can synchronise the device
// and stall every other stream.  This entry point takes its scratch from a fixed array in the
// library's own device memory instead, and calls no allocator at all.
//
// The array below is a module-scope __device__ variable: every GPU that loads the library holds
// its MRR_NOALLOC_SCRATCH_BYTES until the process exits.  Its name, used in host code, is only a
// host-side stand-in for the symbol, not a device address, so the host never hands it to a
// kernel.  The device address is looked up once per device with cudaGetSymbolAddress, with that
// device current, and that address is what the kernels receive.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mrr_v2.h"
#include "ws_layout.h"

namespace {

// mrr_v2_run's own workspace layout (status words, chunk counter, and the two forward-direction
// offset tables above 4096 segments) at the largest N*E this entry point accepts
static_assert(mrr_ws::kHeaderBytes + mrr_ws::table_workspace_bytes(MRR_NOALLOC_MAX_SEGMENTS, 0) <=
                  MRR_NOALLOC_SCRATCH_BYTES,
              "the fixed scratch must hold the status words and both offset tables");

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MRR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Once per device, with that device current: look up the array's device address.
mrr_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return MRR_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return MRR_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MRR_OK;
}

}  // namespace

extern "C" mrr_status mrr_v2_run_noalloc(const void *tokens, mrr_token_dtype dt, int64_t A, int64_t H,
                                         const void *counts, int count_is_i64, int64_t N, int64_t E,
                                         const void *scales, mrr_scale_layout sl, int64_t scale_cols,
                                         const float *topk_w, void *permute_tokens, void *permute_scales,
                                         int32_t *permute_token_idx, void *expert_token_num,
                                         float *permute_topk_w, int64_t expert_token_num_type, int64_t idx_type,
                                         int wait_and_check, mrr_stream_t stream)
{
    // N*E beyond what the fixed tables hold: refuse before touching the GPU
    if (N > 0 && E > 0 && N > MRR_NOALLOC_MAX_SEGMENTS / E)
        return MRR_ERR_WORKSPACE;
    void *scratch = nullptr;
    mrr_status st = scratch_for_current_device(&scratch);
    if (st != MRR_OK)
        return st;
    st = mrr_v2_run(tokens, dt, A, H, counts, count_is_i64, N, E, scales, sl, scale_cols, topk_w, permute_tokens,
                    permute_scales, permute_token_idx, expert_token_num, permute_topk_w, expert_token_num_type,
                    idx_type, scratch, (size_t)MRR_NOALLOC_SCRATCH_BYTES, stream);
    if (st != MRR_OK || !wait_and_check)
        return st;
    return mrr_v2_read_status(scratch, (size_t)MRR_NOALLOC_SCRATCH_BYTES, stream);
}
