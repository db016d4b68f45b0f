// Arguments of the persistent chunk-streaming kernels that the host
// dispatcher fills in (lrscan_abi.cu) and the kernels read
// (stream_kernels.cuh).
#pragma once

#include <stdint.h>
#include <vector_types.h>

namespace lrscan {

// Publication workspace of one call of the persistent chunk-streaming kernels
// (ticket counter zeroed, maps and leaving states filled with all-ones words
// before the launch; maps and leaving states then written by the kernel).
// Chunks are indexed in ticket order within each lane group (the backward
// takes the latest chunk first).
struct StreamArgs {
    unsigned int *ticket;  // next chunk ticket
    float2 *agg;           // [ng * nc][DT] chunk maps (P, Q), lane-thread order
    float *incl;           // [ng * nc][DT] state leaving the chunk, lane-thread order
    int nc;                // chunks per lane group
    int ndt;               // lane tiles per batch row
    int ng;                // lane groups: B * ndt
};

}  // namespace lrscan
