// The gating top-k kernel instances for f16 x (one translation unit per dtype, so the three
// compile in parallel).
#include "gating_kernel.cuh"

namespace mrr_gate {

cudaError_t launch_f16(const Params &p, int vpl, int path, size_t smem, int sms, cudaStream_t stream)
{
    return launch_dtype<MRR_GATE_F16>(p, vpl, path, smem, sms, stream);
}

}  // namespace mrr_gate
