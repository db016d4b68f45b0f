/*
 * lrscan -- differentiable diagonal linear-recurrence scan on NVIDIA GB300
 * (sm_103a).  C ABI of liblrscan.so.
 *
 * The operation (triton_training_scan.py, _real_forward / _real_backward;
 * same definition in the scan's design notes): for every batch row b and
 * channel lane d of contiguous [B, T, D] tensors (D fastest; element
 * (b, t, d) at offset (b*T + t)*D + d),
 *
 *   forward   h_{-1} = 0,  h_t = a_t * h_{t-1} + b_t            t = 0..T-1
 *             out[b,t,d] = h_t (in the storage dtype), last[b,d] = h_{T-1} (fp32)
 *
 *   backward  with the loss L = sum_t grad_out_t * h_t and h read back from out:
 *             g_{T-1} = grad_out_{T-1},  g_t = grad_out_t + a_{t+1} * g_{t+1}
 *             grad_b[b,t,d] = g_t,  grad_a[b,t,d] = g_t * out[b,t-1,d]  (0 at t=0)
 *
 * State and accumulation are fp32 whatever the storage dtype; each
 * recurrence step is one fused multiply-add (one rounding); stores to bf16
 * round to nearest even.  The sequential paths reproduce that order
 * exactly; the chunked and windowed paths reassociate the recurrence through
 * affine maps h -> P*h + Q (triton_training_scan.py, _real_chunk_summary,
 * _real_chunk_prefix, _real_chunk_replay and the _real_reverse_* mirror) and
 * agree to rounding.
 *
 * Common rules for every entry point below:
 *   - All tensor pointers are caller-owned DEVICE pointers (cudaMalloc,
 *     torch, ...) on the calling thread's current CUDA device, contiguous
 *     [B, T, D]; `last` is contiguous [B, D] fp32.  The library never frees
 *     or keeps them after the call's kernels finish.
 *   - Outputs must not overlap inputs or each other (undefined otherwise).
 *   - B, T, D >= 0.  An empty problem is valid: nothing is written, except
 *     that T == 0 with B*D > 0 sets last to 0 (h_{-1}).  Pointers may be NULL
 *     when the problem is empty; otherwise every pointer but `last` (forward,
 *     optional) must be non-NULL.
 *   - Calls are asynchronous on the selected stream (see lrscan_set_stream).
 *     A return of LRSCAN_OK means the kernels were launched; errors found on
 *     the device (a bounded wait that gave up) are reported by the next call
 *     to lrscan_sync_check().
 *   - Any pointer alignment and any D are accepted.  Rows that are 16-byte
 *     aligned (D*sizeof(storage) % 16 == 0 and 16-byte aligned base
 *     pointers) take the bulk-copy (TMA) paths; others take plain-load
 *     kernels.
 *   - Return value: LRSCAN_OK (0) or one of the negative codes below.
 */
#ifndef LRSCAN_H
#define LRSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LRSCAN_VERSION 1

/* error codes */
#define LRSCAN_OK            0
#define LRSCAN_EINVAL       (-1)  /* NULL required pointer, negative size, byte size overflow, bad option */
#define LRSCAN_EDTYPE       (-2)  /* dtype is not LRSCAN_F32 or LRSCAN_BF16 */
#define LRSCAN_ECUDA        (-3)  /* a CUDA runtime call or kernel launch failed */
#define LRSCAN_ENOMEM       (-4)  /* a workspace or staging buffer could not be allocated, or a caller workspace is too small */
#define LRSCAN_ETIMEOUT     (-5)  /* a bounded device wait gave up (reported by lrscan_sync_check) */
#define LRSCAN_ENODEVICE    (-6)  /* no usable sm_103 device is current */

/* storage dtypes: applies to a, b, out, grad_out, grad_a, grad_b (last is always fp32) */
#define LRSCAN_F32   0
#define LRSCAN_BF16  1

/* execution paths (lrscan_opts.path) */
#define LRSCAN_PATH_AUTO    0  /* occupancy rule picks one of the below */
#define LRSCAN_PATH_SEQ     1  /* register-resident sequential-in-T, bulk-copied time tiles */
#define LRSCAN_PATH_CHUNK   2  /* three phases: chunk summary -> warp-shuffle prefix -> replay */
#define LRSCAN_PATH_WINDOW  3  /* single pass: time windows in shared memory, split in time inside the CTA */
#define LRSCAN_PATH_PLAIN   4  /* sequential, plain loads; any alignment */
#define LRSCAN_PATH_STREAM  5  /* single pass over time chunks (triton_training_scan.py, _real_chunk_summary /
                                  _real_chunk_prefix / _real_chunk_replay fused): one persistent CTA per SM takes
                                  chunks of 256 to 1024 steps in ticket order; its summary warps publish each
                                  chunk's map, a scan warp finds the entering state by looking back over the
                                  published maps and leaving states, and its replay warps run the chunk again
                                  while its tiles are still in L2.  Bulk-copy path (16-byte aligned rows); carries
                                  state and resets (lrscan_fwd_state / lrscan_bwd_state, lrscan_cfwd_state /
                                  lrscan_cbwd_state); needs workspace_bytes of device scratch like the
                                  chunked path; agrees with the sequential definition to rounding, and two calls
                                  may differ in the last bits (which published states a look-back composes depends
                                  on timing).  tile_variant: fp32 1 = 32-lane tiles (forward 512-step chunks,
                                  backward 256), 2 = 32-lane tiles, 256-step chunks; bf16 1 = 32-lane tiles,
                                  eight summary and eight replay warps (forward 1024, backward 512), 2 = 64-lane
                                  tiles (512), 3 = 64-lane tiles (256).  Auto takes it for few lanes and at least
                                  32 chunks of 512 steps per lane group: fp32 variant 2 for a forward from eight
                                  lane groups, else 1; bf16 variant 2 for a forward from four 64-lane groups or
                                  with carried state, else 1 */

typedef struct lrscan_opts {
    int path;               /* LRSCAN_PATH_*; 0 = auto */
    int chunk_len;          /* chunked path: 16, 32, 64, 128, 256 or 512; 0 = 64, or for long sequences on few lanes (grouped prefix) 512 forward and 128 backward */
    void *workspace;        /* chunked and streaming paths: optional caller-owned device workspace ... */
    size_t workspace_bytes; /* ... of at least lrscan_workspace_bytes() bytes; NULL = library-owned */
    int tile_variant;       /* >= 1 forces one kernel tile variant of the path (lrscan_plan lists them); 0 = auto.
                               Chunked path: 1 = flat prefix (one warp per lane walks all chunk maps),
                               2 = grouped prefix (group maps, their prefix, per-group rescan) */
} lrscan_opts;

/* What the dispatcher chose (filled by lrscan_plan). */
typedef struct lrscan_plan_info {
    int path;               /* LRSCAN_PATH_* actually taken */
    int tile_variant;       /* variant id within the path */
    int lanes_per_cta;      /* channel lanes one CTA owns */
    int rows_per_window;    /* time steps per shared-memory window (SEQ/WINDOW/STREAM) or chunk length (CHUNK) */
    int subchunks;          /* time splits inside a window (WINDOW), 1 otherwise */
    int stages;             /* shared-memory pipeline depth */
    int ctas;               /* CTAs of the main kernel */
    int threads_per_cta;
    int smem_bytes;         /* dynamic shared memory per CTA */
    int kernels;            /* kernel launches per call */
    size_t workspace_bytes; /* device workspace the call needs */
    char name[64];          /* variant name */
    int exact;              /* 1: every result is bit-identical to the sequential
                               definition (its fused multiply-add order); 0: the
                               path re-associates through affine maps (agrees to
                               rounding) or uses a fast exponential */
} lrscan_plan_info;

/*
 * Forward scan.  a, b: [B,T,D] inputs; out: [B,T,D] output (every h_t);
 * last: [B,D] fp32 final state h_{T-1}, or NULL to skip it.
 * Runs on the thread's current stream (lrscan_set_stream).
 */
int lrscan_fwd(const void *a, const void *b, void *out, float *last,
               int64_t B, int64_t T, int64_t D, int dtype);

/*
 * Backward scan.  a: [B,T,D] forward decays; out: [B,T,D] forward output
 * (h_{t-1} is read from it); grad_out: [B,T,D] dL/dout; grad_a, grad_b:
 * [B,T,D] outputs dL/da, dL/db.  b is not needed.  No gradient flows into
 * `last` or into an initial state (there is none).
 */
int lrscan_bwd(const void *a, const void *out, const void *grad_out,
               void *grad_a, void *grad_b,
               int64_t B, int64_t T, int64_t D, int dtype);

/* As above with an explicit stream (cudaStream_t; NULL = the thread's
 * current stream) and options (NULL = defaults).
 *
 * CUDA graphs: the device calls (lrscan_fwd / _bwd and their _ex, _state,
 * complex and generated-decay forms, lrscan_summary, lrscan_compose_maps)
 * enqueue kernels and stream-ordered copies only, so they can be captured
 * into a graph and replayed, provided that
 *   - one call has run on the device before the capture begins (it looks up
 *     the device's properties and the tensor-map encoder), and
 *   - the library-owned workspace of the stream (chunked path, generated-
 *     decay backward) already has the size the captured call needs: a call
 *     of that size has run on that stream outside capture, or opts->workspace
 *     is passed.  A captured call that would have to grow it returns
 *     LRSCAN_ENOMEM before it enqueues anything (the capture stays valid).
 * The captured kernels read and write the pointers given at capture time.
 * The host-buffer calls, lrscan_sync_check and lrscan_selftest_wait_timeout
 * synchronize and cannot be captured. */
int lrscan_fwd_ex(const void *a, const void *b, void *out, float *last,
                  int64_t B, int64_t T, int64_t D, int dtype,
                  void *stream, const lrscan_opts *opts);
int lrscan_bwd_ex(const void *a, const void *out, const void *grad_out,
                  void *grad_a, void *grad_b,
                  int64_t B, int64_t T, int64_t D, int dtype,
                  void *stream, const lrscan_opts *opts);

/*
 * The same operations with host buffers: every [B,T,D] operand and `last`
 * is a host pointer (page-locked memory moves at full link speed; pageable
 * memory works through the driver's staging; device pointers are accepted
 * too).  The call copies the inputs to device memory in chunks of
 * ceil(B / 8) whole batch rows (fewer when one slot of a chunk's planes
 * would pass 1 GiB, but at least one row), runs the device path on each chunk
 * (lrscan_fwd_ex / lrscan_bwd_ex with `opts`), copies the results back, and
 * returns when every host output is written.  Copies in, kernels and copies
 * out run on three library-owned streams, so one chunk's kernels overlap the
 * next chunk's copy in and the previous chunk's copy out.  Device staging is
 * library-owned (up to three slots of one chunk's planes, kept for later
 * calls).  Calls on one device run one at a time.
 *
 *   lrscan_fwd_host      a, b in; out, last out (last may be NULL).
 *   lrscan_bwd_host      a, out, grad_out in; grad_a, grad_b out.
 *   lrscan_fwd_bwd_host  a, b, grad_out in; out, last, grad_a, grad_b out:
 *                        the forward then the backward of the same inputs,
 *                        out staying on the device in between.
 *
 * Errors: as the device calls (a chunk's error stops the call after the
 * copies already issued have drained), plus LRSCAN_ENOMEM when the staging
 * cannot be allocated and LRSCAN_ECUDA for a failed copy.  A kernel's
 * recorded error (LRSCAN_ETIMEOUT) is returned, and cleared, before the call
 * returns.  T == 0 writes zeros to `last` and touches no device.
 */
int lrscan_fwd_host(const void *a, const void *b, void *out, float *last,
                    int64_t B, int64_t T, int64_t D, int dtype, const lrscan_opts *opts);
int lrscan_bwd_host(const void *a, const void *out, const void *grad_out,
                    void *grad_a, void *grad_b,
                    int64_t B, int64_t T, int64_t D, int dtype, const lrscan_opts *opts);
int lrscan_fwd_bwd_host(const void *a, const void *b, const void *grad_out,
                        void *out, float *last, void *grad_a, void *grad_b,
                        int64_t B, int64_t T, int64_t D, int dtype, const lrscan_opts *opts);

/*
 * Carried state and segment resets.  The state-carrying serial scans of
 * triton_training_scan.py (_samu_tiled_serial_forward and
 * _samu_tiled_serial_backward: initial state, per-token segment positions,
 * gradient at the final state, gradient of the initial state) applied to this
 * scan; with it a sequence split across calls (prefill, then decode, as the
 * state-carrying recurrences of the KDN page's recurrence.py do) continues
 * exactly, and packed sequences restart at their first token.
 *
 *   forward   h_{-1} = h0;  a'_t = 0 where segment_pos[b,t] == 0, else a_t;
 *             h_t = a'_t * h_{t-1} + b_t;  last = h_{T-1}
 *   backward  with L = sum_t grad_out_t * h_t + sum grad_last * last:
 *             g_T = grad_last, entering step T-1 through a'_T = 1,
 *             g_t = grad_out_t + a'_{t+1} * g_{t+1}   (one rounding),
 *             grad_b_t = g_t,
 *             grad_a_t = +0 where step t starts a segment (a_t is unused
 *                        there), else g_t * out_{t-1} with out_{-1} = h0,
 *             grad_h0  = a'_0 * g_0   (grad_last when T == 0).
 *
 * Every member may be NULL (zeros / no resets / not written); the forward
 * reads only h0 and segment_pos.  h0, grad_last and grad_h0 are fp32 [B, D]
 * whatever the storage dtype (the state precision: `last` of one call can be
 * the next call's h0); segment_pos is int32 [B, T], one position per token,
 * shared by all D channels.  All are caller-owned device pointers, 4-byte
 * aligned (else LRSCAN_EINVAL); grad_h0 must not overlap any input.
 */
typedef struct lrscan_state {
    const float *h0;            /* [B, D] fp32: state before step 0 */
    const int32_t *segment_pos; /* [B, T] int32: 0 marks the first step of a segment */
    const float *grad_last;     /* backward: [B, D] fp32 gradient arriving at `last` */
    float *grad_h0;             /* backward: [B, D] fp32 output, gradient of h0 */
} lrscan_state;

/* lrscan_fwd_ex / lrscan_bwd_ex with carried state (state NULL: the plain
 * scan).  Same paths, options, streams and errors; with T == 0 the forward
 * copies h0 (or zeros) into last and the backward grad_last (or zeros) into
 * grad_h0. */
int lrscan_fwd_state(const void *a, const void *b, void *out, float *last,
                     const lrscan_state *state,
                     int64_t B, int64_t T, int64_t D, int dtype,
                     void *stream, const lrscan_opts *opts);
int lrscan_bwd_state(const void *a, const void *out, const void *grad_out,
                     void *grad_a, void *grad_b, const lrscan_state *state,
                     int64_t B, int64_t T, int64_t D, int dtype,
                     void *stream, const lrscan_opts *opts);

/*
 * Complex diagonal scan on separate real / imaginary planes
 * (triton_training_scan.py, _complex_forward / _complex_backward and
 * complex_scan_with_last).  Per lane, with a_t = ar + i*ai, b_t = br + i*bi:
 *
 *   forward   h_{-1} = 0,  h_t = a_t * h_{t-1} + b_t
 *             out_r / out_i = Re / Im h_t (storage dtype); last_r / last_i =
 *             Re / Im h_{T-1} (fp32; either may be NULL)
 *   backward  loss L = sum_t (grad_out_r * Re h_t + grad_out_i * Im h_t):
 *             g_{T-1} = grad_out_{T-1},  g_t = grad_out_t + conj(a_{t+1}) * g_{t+1},
 *             grad_b = g,  grad_a = g * conj(h_{t-1})  (h_{-1} = 0; h read from out)
 *
 * Each component is two nested fused multiply-adds:
 *   Re h = fma(ar, Re h, fma(-ai, Im h, br)),  Im h = fma(ai, Re h, fma(ar, Im h, bi))
 *   Re g = fma(ar', Re g, fma(ai', Im g, go_r)), Im g = fma(ar', Im g, fma(-ai', Re g, go_i))
 *   grad_ar = fma(Re g, Re p, Im g * Im p),  grad_ai = fma(Im g, Re p, -(Re g * Im p))
 * (a' = a_{t+1}, p = h_{t-1}); both paths use this order and agree bit for bit.
 * All planes are caller-owned device [B, T, D] tensors of one storage dtype;
 * paths: tiled (LRSCAN_PATH_SEQ or LRSCAN_PATH_WINDOW: one table of
 * sequential and windowed tiles, 16-byte aligned rows of every plane),
 * LRSCAN_PATH_CHUNK (three phases over time chunks of opts->chunk_len steps,
 * 16 ... 512, default 64 fp32 / 128 bf16: complex chunk maps, their prefix -- flat, or grouped
 * when a lane has many chunks; tile_variant 1 / 2 forces flat / grouped --
 * and the replay; any alignment), LRSCAN_PATH_STREAM (the persistent
 * chunk-streaming kernels of the real scan on the re / im planes: complex
 * chunk maps and states published as self-validating words; fp32 forward
 * 256-step chunks, backward 128; bf16 512 and 256; aligned rows, no carried
 * state; one tile variant) or LRSCAN_PATH_PLAIN (any alignment).  Auto takes,
 * when the lanes fill fewer than 0.45 lane tiles of 32 per SM (aligned rows;
 * else 32 warps per SM) and T >= 16 chunks, the streaming path (aligned rows,
 * no carried state, no chunk_len asked for, T >= 32 * 512), else the chunked
 * path; with more lanes a tiled variant when the rows are aligned, else the
 * plain kernels.
 * The sequential tiles and the plain kernels keep the order above and agree
 * with it bit for bit; the windowed tiles, the chunked and the streaming
 * paths (complex affine maps) agree to rounding.  The chunked and streaming
 * paths need lrscan_plan_complex(...).workspace_bytes of device scratch:
 * library-owned per (device, stream), or opts->workspace.  Moves 6 elements
 * per (t, d) forward and 10 backward (the chunked path re-reads its inputs:
 * 10 and 16).
 * Other rules as lrscan_fwd_ex.
 */
int lrscan_cfwd(const void *ar, const void *ai, const void *br, const void *bi,
                void *out_r, void *out_i, float *last_r, float *last_i,
                int64_t B, int64_t T, int64_t D, int dtype,
                void *stream, const lrscan_opts *opts);
int lrscan_cbwd(const void *ar, const void *ai, const void *out_r, const void *out_i,
                const void *grad_out_r, const void *grad_out_i,
                void *grad_ar, void *grad_ai, void *grad_br, void *grad_bi,
                int64_t B, int64_t T, int64_t D, int dtype,
                void *stream, const lrscan_opts *opts);
/* lrscan_plan for the complex scan (tile variants listed by tile_variant 1..) */
int lrscan_plan_complex(int64_t B, int64_t T, int64_t D, int dtype, int dir, int aligned16,
                        const lrscan_opts *opts, lrscan_plan_info *info);
/* The plan of a complex call with carried state or resets
 * (lrscan_cfwd_state / lrscan_cbwd_state): the same choice as
 * lrscan_plan_complex, except that unaligned rows take the chunked path (the
 * plain kernels carry no state). */
int lrscan_plan_complex_state(int64_t B, int64_t T, int64_t D, int dtype, int dir, int aligned16,
                              const lrscan_opts *opts, lrscan_plan_info *info);

/*
 * Complex scan with carried state and segment resets
 * (triton_training_scan.py, _samu_tiled_serial_forward /
 * _samu_tiled_serial_backward: the page's state-carrying scan is complex).
 * The rules of lrscan_state, with complex states and conjugate transitions:
 *   forward   h_{-1} = h0 (0 when absent); a'_t = 0 where segment_pos is 0;
 *             h_t = a'_t * h_{t-1} + b_t; last = h_{T-1}
 *   backward  grad_last enters step T-1 through a'_T = 1;
 *             g_t = grad_out_t + conj(a'_{t+1}) * g_{t+1};  grad_b = g;
 *             grad_a_t = +0 where step t starts a segment, else
 *             g_t * conj(h_{t-1}) with h_{-1} = h0;
 *             grad_h0 = conj(a'_0) * g_0 (+0 when step 0 starts a segment)
 * Every member may be NULL (all NULL: the plain complex scan); fp32 / int32
 * device pointers, 4-byte aligned.  These calls run on the tiled kernels
 * (opts: LRSCAN_PATH_AUTO, or LRSCAN_PATH_SEQ / LRSCAN_PATH_WINDOW with
 * tile_variant as lrscan_plan_complex_state reports) when every plane's rows
 * are 16-byte aligned and the lanes fill the GPU, else on the chunked path
 * (LRSCAN_PATH_CHUNK: chunk_len, tile_variant 1 / 2 for the flat / grouped
 * prefix, workspace as lrscan_plan_complex_state reports; any row
 * alignment).  LRSCAN_PATH_PLAIN is refused (LRSCAN_EINVAL).  With T == 0
 * the forward copies h0 (or zeros) into last and the backward grad_last (or
 * zeros) into grad_h0.  The sequential tiles reproduce the sequential
 * definition bit for bit (lrscan_plan_info.exact); the windowed tiles and
 * the chunked path agree with it to rounding.
 */
typedef struct lrscan_cstate {
    const float *h0_r, *h0_i;         /* [B, D] fp32 each: state before step 0 */
    const int32_t *segment_pos;       /* [B, T] int32: 0 marks the first step of a segment */
    const float *grad_last_r, *grad_last_i;  /* backward: [B, D] fp32 gradient arriving at last */
    float *grad_h0_r, *grad_h0_i;     /* backward: [B, D] fp32 outputs, gradient of h0 */
} lrscan_cstate;
int lrscan_cfwd_state(const void *ar, const void *ai, const void *br, const void *bi,
                      void *out_r, void *out_i, float *last_r, float *last_i,
                      const lrscan_cstate *state, int64_t B, int64_t T, int64_t D, int dtype,
                      void *stream, const lrscan_opts *opts);
int lrscan_cbwd_state(const void *ar, const void *ai, const void *out_r, const void *out_i,
                      const void *grad_out_r, const void *grad_out_i,
                      void *grad_ar, void *grad_ai, void *grad_br, void *grad_bi,
                      const lrscan_cstate *state, int64_t B, int64_t T, int64_t D, int dtype,
                      void *stream, const lrscan_opts *opts);

/*
 * Scan with a generated decay (triton_training_scan.py, _samu_forward and
 * _samu_precompute_decay, the radius part of the page's transition): the
 * decay of lane d at token t is rebuilt in the kernel instead of being read,
 *
 *   a_{b,t,d} = exp(-exp(nu_log[d]) * exp(eta[b,t])),   h_t = a_t * h_{t-1} + b_t,
 *
 * eta fp32 [B, T] (one value per token, shared by all lanes), nu_log fp32 [D]
 * (one per lane).  Forward moves 2 elements per (t, d) (b in, out out) instead
 * of 3.  Backward, for L = sum_t grad_out_t * h_t (out read back for h_{t-1}),
 * writes grad_b [B, T, D] (storage dtype) and the parameter gradients
 *   grad_eta[b,t]  = sum_d q,   grad_nu_log[d] = sum_{b,t} q,
 *   q = grad_a * a * log a,  grad_a = g_t * out_{t-1},  log a = -exp(nu_log) exp(eta),
 * both fp32, summed in a fixed order (deterministic); it moves 3 elements per
 * (t, d).  Exponentials are fast approximations (e^x = 2^(x log2 e) with the
 * ex2.approx instruction: relative error of a few 1e-7; a decay below 2^-126
 * is taken as 0), so results agree with an exact evaluation to rounding, not
 * bit for bit.
 * The backward needs lrscan_gated_workspace_bytes(B, T, D) bytes of scratch:
 * library-owned per (device, stream), or opts->workspace.  Paths:
 * LRSCAN_PATH_SEQ (tiled, 16-byte aligned rows) or LRSCAN_PATH_PLAIN; auto
 * picks seq when it can.  Tiled kernels (tile_variant, named by
 * lrscan_plan_gated): from eight 16-lane slices per SM one warp per slice
 * (time split between its thread groups, no CTA barrier), else windowed tiles
 * (time split inside the CTA).  With T == 0 the forward sets last to 0 and the
 * backward sets grad_nu_log to 0.
 */
int lrscan_fwd_gated(const float *eta, const float *nu_log, const void *b, void *out, float *last,
                     int64_t B, int64_t T, int64_t D, int dtype,
                     void *stream, const lrscan_opts *opts);
int lrscan_bwd_gated(const float *eta, const float *nu_log, const void *out, const void *grad_out,
                     void *grad_b, float *grad_eta, float *grad_nu_log,
                     int64_t B, int64_t T, int64_t D, int dtype,
                     void *stream, const lrscan_opts *opts);
size_t lrscan_gated_workspace_bytes(int64_t B, int64_t T, int64_t D);
int lrscan_plan_gated(int64_t B, int64_t T, int64_t D, int dtype, int dir, int aligned16,
                      const lrscan_opts *opts, lrscan_plan_info *info);

/*
 * Whole-sequence affine summary of every lane (the chunk summary of
 * triton_training_scan.py, _real_chunk_summary and its reverse mirror, with
 * one chunk spanning all T steps).  With a'_t = 0 where segment_pos[b,t] == 0
 * (segment_pos may be NULL), P = prod_t a'_t and
 *   dir 0 (forward):  x = b;         h_{T-1} = P * h0 + Q,       Q = h_{T-1} from h0 = 0
 *   dir 1 (backward): x = grad_out;  grad_h0 = P * grad_last + Q, Q = grad_h0 from grad_last = 0
 * P and Q are caller-owned fp32 [B, D] device outputs.  This is the local
 * step of a sequence split across devices: each device summarizes its time
 * segment, the maps are exchanged and composed in order, and each device
 * then scans its segment with lrscan_fwd_state / lrscan_bwd_state from the
 * composed h0 / grad_last.  T == 0 gives the identity map (P = 1, Q = 0).
 * Reads a and x once (2 elements per (t, d)); one thread per lane.
 */
int lrscan_summary(const void *a, const void *x, float *P, float *Q,
                   const int32_t *segment_pos, int64_t B, int64_t T, int64_t D,
                   int dtype, int dir, void *stream);

/*
 * Composition of per-segment maps, the exchange step's arithmetic for a
 * sequence split across devices (the serial prefix over chunk maps of
 * triton_training_scan.py, _real_chunk_prefix, with one chunk per segment).
 * maps: fp32 [W][2][B][D] device array, maps[r][0] = P_r and maps[r][1] = Q_r
 * of segment r (lrscan_summary); init: fp32 [B, D] or NULL (zeros); out: fp32
 * [B, D].  out = the fold of h -> fma(P_r, h, Q_r) over
 *   dir 0: r = 0, 1, ..., rank-1   (state entering segment `rank`, init = h0)
 *   dir 1: r = W-1, ..., rank+1    (adjoint entering segment `rank` from the
 *                                   later ones, init = grad_last)
 * applied to init.  0 <= rank < W.
 */
int lrscan_compose_maps(const float *maps, int64_t W, int64_t rank, const float *init,
                        float *out, int64_t B, int64_t D, int dir, void *stream);

/* Sets the calling thread's stream (a cudaStream_t; NULL = legacy default
 * stream) used by lrscan_fwd / lrscan_bwd and by _ex calls given NULL. */
int lrscan_set_stream(void *stream);

/* Device bytes the chunked path needs for this shape: two fp32 [B, ceil(T/C), D]
 * buffers, plus two fp32 [B, ceil(T/C/512), D] buffers for the grouped prefix
 * (each rounded up to 256 bytes; the value covers both prefix variants);
 * chunk_len 0 means 64.  Other paths need none. */
size_t lrscan_workspace_bytes(int64_t B, int64_t T, int64_t D, int chunk_len);

/* Host-only: what a call with these arguments would run (no launch, no
 * device memory touched beyond reading device attributes).  dir: 0 forward,
 * 1 backward.  aligned16: whether the call's pointers are 16-byte aligned. */
int lrscan_plan(int64_t B, int64_t T, int64_t D, int dtype, int dir, int aligned16,
                const lrscan_opts *opts, lrscan_plan_info *info);
/* lrscan_plan for a call with carried state or resets (lrscan_fwd_state,
 * lrscan_bwd_state, the _ex calls given a state): the bf16 backward's
 * automatic choice differs there. */
int lrscan_plan_state(int64_t B, int64_t T, int64_t D, int dtype, int dir, int aligned16,
                      const lrscan_opts *opts, lrscan_plan_info *info);

/* Number of tile variants of a path (for sweeps); names via lrscan_plan. */
int lrscan_num_variants(int path, int dtype, int dir);

/* Waits for the thread's current stream, then returns and clears the first
 * error any kernel of this library recorded on the current device since the
 * last check (LRSCAN_ETIMEOUT for a wait that gave up), else the stream's
 * CUDA error as LRSCAN_ECUDA, else LRSCAN_OK. */
int lrscan_sync_check(void);

/* Limit on every bounded device-side wait, in nanoseconds (default 1e9; at
 * least 1e6, else LRSCAN_EINVAL: the kernels also bound their drains of their
 * own bulk copies with it).  Applies to launches made after the call, on every
 * device. */
int lrscan_set_wait_timeout_ns(uint64_t ns);

/* Self-test of the bounded wait: launches one CTA that waits, with the given
 * limit, on a shared-memory barrier that nothing will ever complete.  The
 * wait must give up, record LRSCAN_ETIMEOUT and return; this call
 * synchronizes and returns what lrscan_sync_check() reports (so
 * LRSCAN_ETIMEOUT is the expected, healthy result). */
int lrscan_selftest_wait_timeout(uint64_t timeout_ns);

/* Human-readable text for an error code (static storage). */
const char *lrscan_strerror(int code);

/* Detail of the calling thread's last failed call (why an argument was
 * rejected, which launch failed); empty after a successful call.  Valid
 * until the thread's next call into the library. */
const char *lrscan_last_error(void);

int lrscan_version(void);

/*
 * Chunked forward scan that allocates nothing.
 *
 * No counterpart in the paper: this entry point exists for callers that
 * cannot call cudaMalloc while they run (code inside an allocator or
 * memory-pool callback, where a nested allocation would re-enter the
 * allocator; latency-critical loops that ban allocation because cudaMalloc
 * may synchronize the device; hosts that only hand the library pre-sized
 * buffers).  It runs the three chunked phases of LRSCAN_PATH_CHUNK with the
 * arguments of lrscan_fwd_ex(..., path = chunk, chunk_len), but its scratch
 * (the chunk summaries P and Q) lives in one fixed device array of
 * LRSCAN_NOALLOC_SCRATCH_BYTES that the library owns.
 *   - It always uses the flat chunk prefix (one warp per lane walks all the
 *     lane's chunk maps).  Where the regular chunked call picks the grouped
 *     prefix (many chunks per lane, few lanes) the two compose the maps in a
 *     different order, so their results can differ by rounding (both stay
 *     within the scan's tolerances of the sequential definition), and long
 *     sequences on few lanes run slower here.
 *   - Every GPU that loads the library holds that array until the process
 *     exits.
 *   - A problem needs 2 * B * ceil(T / chunk_len) * D * 4 bytes of it (each
 *     half rounded up to 256 bytes); larger problems are rejected with
 *     LRSCAN_ENOMEM (see lrscan_last_error) before anything is launched.
 *   - All calls on a device share the array: calls whose kernels overlap on
 *     the GPU (different streams, no ordering between them) race and produce
 *     wrong results.  Calls on one stream are safe.  Nothing has to be cleared
 *     between calls: each call writes all the scratch it reads.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current).  With CUDA's lazy module
 *     loading that lookup may load the library's device code and reserve the
 *     array's memory at that moment.  So make one warm-up call on each device
 *     outside any allocator callback, before any stream capture begins.
 *   - a, b, out, last, sizes and dtype as in lrscan_fwd; chunk_len 16, 32 or
 *     64 (0 means 64); stream is a cudaStream_t (NULL = legacy default stream).
 */
#define LRSCAN_NOALLOC_SCRATCH_BYTES (32u << 20)
int lrscan_fwd_chunk_noalloc(const void *a, const void *b, void *out, float *last,
                             int64_t B, int64_t T, int64_t D, int dtype,
                             int chunk_len, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LRSCAN_H */
