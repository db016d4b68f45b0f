"""GB300-native differentiable diagonal linear-recurrence scan.

    h_t = a_t * h_{t-1} + b_t          (forward, h_{-1} = 0)
    g_t = grad_out_t + a_{t+1} g_{t+1} (backward; grad_b = g, grad_a = g * h_{t-1})

its state-carrying form (initial state h0, segment resets, gradients of the
final and initial states: ``scan_state``), the complex scan on re/im planes
(``complex_scan``; with carried complex state ``complex_scan_state``), the scan with decays generated in the kernel from
per-token and per-lane parameters (``gated_scan``), and the pieces of a sequence split across devices
(``lrscan_summary``, ``lrscan_compose_maps``, module ``tsplit``), and calls on
host buffers that pipeline the copies with the kernels (``lrscan_fwd_host``,
``lrscan_bwd_host``, ``lrscan_fwd_bwd_host``).

The compute path is liblrscan.so (hand-written sm_103a CUDA kernels behind a C
ABI, ``include/lrscan.h``); ``lrscan`` is its Python binding.  Importing this
package does not load the library; the first call does, and fails loudly if
it has not been built.
"""
from .lrscan import (  # noqa: F401
    ComplexScan,
    ComplexScanState,
    GatedScan,
    LinearRecurrenceScan,
    LinearRecurrenceScanState,
    LrscanError,
    LrscanUnavailable,
    complex_scan,
    complex_scan_state,
    gated_scan,
    lrscan_bwd_gated,
    lrscan_cbwd,
    lrscan_cbwd_state,
    lrscan_cfwd,
    lrscan_cfwd_state,
    lrscan_compose_maps,
    lrscan_bwd,
    lrscan_bwd_host,
    lrscan_bwd_state,
    lrscan_fwd,
    lrscan_fwd_bwd_host,
    lrscan_fwd_gated,
    lrscan_fwd_host,
    lrscan_fwd_state,
    lrscan_gated_workspace_bytes,
    lrscan_num_variants,
    lrscan_plan,
    lrscan_plan_complex,
    lrscan_plan_gated,
    lrscan_selftest_wait_timeout,
    lrscan_set_wait_timeout_ns,
    lrscan_summary,
    lrscan_sync_check,
    lrscan_workspace_bytes,
    scan,
    scan_state,
)
