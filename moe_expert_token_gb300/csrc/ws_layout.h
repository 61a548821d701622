// Layout of the caller-owned workspace of the re-routing op, shared by every translation unit
// that sizes or addresses one (mrr_v2.cu, mrr_v2_noalloc.cu, mrr_push.cu).
//
//   bytes 0 .. 4095       status words: [0] count-error flags, [1] grid size, [2 + b] CTA b's flags
//   bytes 4096 .. 4351    the bulk path's chunk counter (one 64-bit word, the rest padding)
//   bytes 4352 ..         only when N*E exceeds the fused-scan limit: the SrcOffset table
//                         (N*E + 1 uint32) and the DstOffset table (padded, see padded_len), and
//                         for the inverse move a third table of the column-major starts, each
//                         rounded up to 256 bytes
#ifndef MRR_WS_LAYOUT_H
#define MRR_WS_LAYOUT_H

#include <stdint.h>

namespace mrr_ws {

constexpr int kStatusBytes = 4096;
constexpr int kStatusWords = kStatusBytes / 4;
constexpr int kTicketOffset = kStatusBytes;
constexpr int kHeaderBytes = kStatusBytes + 256;

// The flags kernels leave in the status words; mrr_v2_read_status maps them to status codes.
constexpr uint32_t kFlagNonPos = 1u;    // a count <= 0
constexpr uint32_t kFlagSum = 2u;       // the counts do not sum to the rows given
constexpr uint32_t kFlagTimeout = 4u;   // a bounded wait gave up
constexpr uint32_t kFlagBadIndex = 8u;  // gating: an input_ids / tid2eid value out of range
constexpr uint32_t kFlagSource = 16u;   // multi-source form: a per-rank source is missing or too small
constexpr uint32_t kFlagDest = 32u;     // push form: a receiver's buffer is missing or too small

// Length of a table indexed with one padding word per 32 entries (plus one end entry).
__host__ __device__ constexpr int64_t padded_len(int64_t n) { return n + (n >> 5) + 1; }

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Workspace bytes of the offset tables behind the header (N*E above the fused-scan limit).
__host__ __device__ constexpr int64_t table_workspace_bytes(int64_t NE, int inverse)
{
    return round_up(4 * (NE + 1), 256) + round_up(4 * padded_len(NE), 256) +
           (inverse ? round_up(4 * padded_len(NE), 256) : 0);
}

}  // namespace mrr_ws

#endif  // MRR_WS_LAYOUT_H
