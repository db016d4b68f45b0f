// Carried state and segment resets of one call, as the kernels receive them
// (triton_training_scan.py, _samu_tiled_serial_forward / _backward: initial
// state, per-token segment positions, gradient at the final state, gradient
// of the initial state).  Every pointer may be null; all are device pointers
// already offset to the first batch row of the launch.
#pragma once

#include <stdint.h>

namespace lrscan {

struct StateArgs {
    const float *h0;         // [B, D] fp32 state before step 0 (null: zeros)
    const int32_t *seg;      // [B, T] segment positions; 0 starts a segment (null: none)
    const float *grad_last;  // [B, D] fp32 gradient arriving at the final state (null: zeros)
    float *grad_h0;          // [B, D] fp32 gradient of h0 (backward; null: not written)
    const void *a;           // the decays [B, T, D] (backward: grad_h0 = a'_0 * g_0)
};

// Carried state of a complex scan: h0 and grad_last in, grad_h0 out (re and
// im fp32 [B, D] each), segment positions int32 [B, T]; all null: none.  The
// tiled backward also reads the decay planes ar / ai [B, T, D] for
// grad_h0 = conj(a'_0) * g_0.
struct CStateArgs {
    const float *h0_r, *h0_i;
    const int32_t *seg;
    const float *gl_r, *gl_i;
    float *gh0_r, *gh0_i;
    const void *ar, *ai;
};

}  // namespace lrscan
