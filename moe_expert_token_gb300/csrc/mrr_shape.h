// The shape and attribute rules of the re-routing op's entry points (the checks of mrr_v2_plan),
// shared by the translation units that take such a problem (mrr_v2.cu, mrr_push.cu).
#ifndef MRR_SHAPE_H
#define MRR_SHAPE_H

#include <stdint.h>

#include "mrr_v2.h"

namespace mrr_host {

// A rows of H elements of token dtype dt, counts [N, E], scale layout sl with scale_cols, and the
// two attributes: MRR_OK with the token and scale row sizes in bytes, or the status the entry
// points return for these arguments.  No pointers are checked.
mrr_status check_shape(int64_t A, int64_t H, int dt, int64_t N, int64_t E, int count_is_i64, int sl,
                       int64_t scale_cols, int64_t etn_type, int64_t idx_type, int64_t *row_bytes,
                       int64_t *scale_row_bytes);

}  // namespace mrr_host

#endif  // MRR_SHAPE_H
