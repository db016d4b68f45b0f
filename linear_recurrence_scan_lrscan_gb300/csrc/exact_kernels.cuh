// Exact windowed scan, pipelined (xwp tiles).
//
// The same result as the sequential scan, bit for bit, with the time split
// of the windowed tiles.  A CTA owns one batch row and DT lanes; each window
// of W = S * L rows is split into S sub-chunks of L rows.  Three roles:
//
//   replay threads (s, g), S * G of them: copy their L rows of the window
//     into registers, release the stage at once, and after the window's
//     barrier replay their rows from the sub-chunk's entry state with the
//     sequential step, writing the results into a shared-memory stage that
//     a bulk tensor store writes back;
//   walker threads, DT of them (DT / 32 warps): each walks one lane through
//     all W rows of the window straight from the shared-memory stage with
//     the sequential step itself, recording the state that enters every
//     sub-chunk (so the entries, and every replayed value, are the
//     sequential definition's own);
//   walker thread 0 also keeps the stage ring full (bulk tensor copies
//     completed on mbarriers; a stage is refilled once the replay warps and
//     the walker warps have released it) and issues the output stores.
//
// One named barrier per window: it publishes the window's entries (written
// into one of two buffers) and tells the store issuer that the previous
// window's replay is staged.  The walk of window k + 1 then runs while the
// replay threads replay window k, so the serial walk overlaps the rest of
// the window's work; output staging has three buffers, so the store of
// window k-2 only has to finish reading before the next barrier.
//
// Backward windows run last-to-first, with the decay tile one row late
// (a_{t+1}) and the out tile one row early (h_{t-1}) as in the windowed
// backward.  EXT instantiations carry h0 / grad_last / grad_h0 and segment
// resets with the rules of the windowed kernels.
#pragma once

#include "window_kernels.cuh"

namespace lrscan {

// Entry states [2][S][DT] (by window parity) at the scan area, then the
// walker warps' per-sub-chunk reset masks [DT / 32][SMAX].
template <class C>
__device__ __forceinline__ float *xwp_entries(const WinSmem &sm, int par) {
    return reinterpret_cast<float *>(sm.base + sm.scan_off) + par * sm.S * C::DT;
}
template <class C>
__device__ __forceinline__ uint32_t *xwp_masks(const WinSmem &sm, int walker_warp) {
    return reinterpret_cast<uint32_t *>(sm.base + sm.scan_off + 2 * sm.S * C::DT * 4) + walker_warp * C::SMAX;
}

// Reset masks of one window for the walker warps: bit j of word s is row
// s * L + j (rows from `row0` of the sequence, position `shift` later: 0
// forward, 1 backward), from the positions prefetched in `pos` (lane l holds
// rows l, l + 32, ...).  Written by lanes s < S of the warp.
template <class C, int NM>
__device__ __forceinline__ void xwp_write_masks(uint32_t *mk, const int32_t (&pos)[NM], int S, int lane) {
    constexpr int L = C::L;
    uint32_t w[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) w[m] = __ballot_sync(0xffffffffu, pos[m] == 0);
    if (lane < S) {
        const int r = lane * L;
        uint32_t word = 0;
#pragma unroll
        for (int m = 0; m < NM; ++m) word = (r >> 5) == m ? w[m] : word;
        mk[lane] = (word >> (r & 31)) & (L == 32 ? 0xffffffffu : ((1u << L) - 1u));
    }
    __syncwarp();
}

// Bounded wait for every copy the producer issued that no consumer waited
// for (after an abort), so none lands after the CTA exits.
__device__ __forceinline__ void xwp_drain(const WinSmem &sm, int consumed, int issued, const WaitCtx &wc) {
    for (int k = consumed; k < issued; ++k) {
        const uint32_t fb = sm.full_bar(k % sm.nstage);
        const uint32_t par = (k / sm.nstage) & 1;
        const uint64_t start = global_timer_ns();
        while (!mbar_try_wait(fb, par)) {
            if (global_timer_ns() - start > wc.timeout_ns) {
                record_error(wc, kErrTimeout, kSiteDrain);
                break;
            }
        }
    }
}

// ============================================================================
// Forward
// ============================================================================
template <class C, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
xwp_fwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_out, float *__restrict__ last,
               const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns,
               const __grid_constant__ StateArgs sx) {
    static_assert(!C::SEQ && !C::PT && C::EX && C::NIN == 2, "pipelined exact forward: exact windowed shape");
    static_assert(C::DT % 32 == 0, "walker threads are whole warps");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    constexpr int NM = (C::SMAX * L + 31) / 32;  // position words per walker lane
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;   // replay threads
    const int NW = NT + DT;  // + walker threads; all take part in the window barrier
    win_init<C>(sm, NW / 32, S);
    pdl_trigger();
    pdl_wait();  // inputs may come from the previous kernel in the stream
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D, W = sm.W, nwin = sm.nwin, nstage = sm.nstage;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const bool walker = tid >= NT;
    const bool producer = tid == NT;
    const CUtensorMap *const imaps[2] = {&tm_a, &tm_b};
    const CUtensorMap *const omaps[1] = {&tm_out};
    const OutStage<1, St, 3> ost = make_out_stage<1, St, 3>(smem_raw, geom);
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};

    // producer prologue: the first windows into the ring
    int issued = 0;
    if (producer) {
        for (int i = 0; i < 2; ++i) prefetch_tensormap(imaps[i]);
        for (int k = 0; k < nwin && k < nstage; ++k) {
            const uint32_t fb = sm.full_bar(k);
            mbar_arrive_expect_tx(fb, sm.stage_bytes);
            for (int i = 0; i < 2; ++i) tma_load_3d(smem_addr(sm.tile<C>(k, i)), imaps[i], d0, k * W, brow, fb);
            issued = k + 1;
        }
    }

    // replay thread (s, lg): lanes d .. d + V - 1, rows s*L .. s*L + L - 1
    const int s = walker ? 0 : tid / G;
    const int lg = walker ? 0 : tid - s * G;
    const int d = d0 + lg * V;
    const bool lane_ok = !walker && d < D;
    // walker thread wi walks scan index wi (channel lane_channel(d0, wi))
    const int wi = tid - NT;
    float carry = 0.0f;
    float h[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h[v] = 0.0f;
    // EXT positions, one window ahead: replay warps' rows (one ballot per
    // window) and the walker lanes' rows l, l + 32, ...
    const int wrow = walker ? 0 : ((tid & ~31) / G) * L;
    int32_t pos_next = 1;
    int32_t wpos[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) wpos[m] = 1;
    if constexpr (EXT) {
        static_assert((G >= 32 ? 1 : 32 / G) * L <= 32, "one ballot covers a replay warp's rows");
        if (walker) {
            if (sx.h0 != nullptr) {
                const int ch = lane_channel<C>(d0, wi);
                carry = ch < D ? sx.h0[static_cast<size_t>(brow) * D + ch] : 0.0f;
            }
#pragma unroll
            for (int m = 0; m < NM; ++m) wpos[m] = (32 * m + lane < W) ? seg.at(32 * m + lane) : 1;
        } else {
            pos_next = seg.at(wrow + lane);
        }
    }

    bool failed = false;
    int k = 0;
    for (; k < nwin; ++k) {
        const int stage = k % nstage;
        const uint32_t par = (k / nstage) & 1;
        const int rbase = k * W + s * L;
        const int n = min(max(T - rbase, 0), L);
        uint32_t rbits = 0;
        if constexpr (EXT) {
            if (!walker) {
                rbits = __ballot_sync(0xffffffffu, pos_next == 0) >> (s * L - wrow);
                pos_next = seg.at((k + 1) * W + wrow + lane);
            } else {
                xwp_write_masks<C, NM>(xwp_masks<C>(sm, wi / 32), wpos, S, lane);
#pragma unroll
                for (int m = 0; m < NM; ++m) wpos[m] = (32 * m + lane < W) ? seg.at((k + 1) * W + 32 * m + lane) : 1;
            }
        }
        const bool ok = mbar_wait(sm.full_bar(stage), par, wc, kSiteConsumerFull);
        float xa[L][V], xb[L][V];
        if (!walker) {
            if (ok) {
                const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;
                const St *tb = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    unpack_lanes<St, V>(ta + j * DT, xa[j]);
                    unpack_lanes<St, V>(tb + j * DT, xb[j]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
            if (EXT && rbits != 0) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
#pragma unroll
                    for (int v = 0; v < V; ++v) xa[j][v] = ((rbits >> j) & 1u) ? 0.0f : xa[j][v];
                }
            }
            if (n < L) {
                // steps past T become exact identity steps (a = 1, b = 0)
#pragma unroll
                for (int j = 0; j < L; ++j) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        xa[j][v] = j < n ? xa[j][v] : 1.0f;
                        xb[j][v] = j < n ? xb[j][v] : 0.0f;
                    }
                }
            }
        } else if (ok) {
            carry = exact_walk<C, false, EXT, false>(sm.tile<C>(stage, 0), sm.tile<C>(stage, 1),
                                                     xwp_entries<C>(sm, k & 1), xwp_masks<C>(sm, wi / 32), S, wi,
                                                     T - k * W, carry);
        }
        // entries of window k published; replay of window k-1 staged and fenced
        if (bar_sync_or(1, NW, !ok)) { failed = true; break; }
        if (walker) {
            if (lane == 0) mbar_arrive(sm.empty_bar(stage));  // the walk has read the stage
            if (producer) {
                if (k > 0) {
                    ost.store(omaps, k - 1, d0, (k - 1) * W, brow);
                    bulk_wait_read<1>();  // the store of k-2 is done with its buffer
                }
                const int kn = k + nstage;
                if (kn < nwin) {
                    // every warp has released this stage: refill it with window kn
                    if (mbar_wait(sm.empty_bar(stage), par, wc, kSiteProducerEmpty)) {
                        const uint32_t fb = sm.full_bar(stage);
                        mbar_arrive_expect_tx(fb, sm.stage_bytes);
                        for (int i = 0; i < 2; ++i)
                            tma_load_3d(smem_addr(sm.tile<C>(stage, i)), imaps[i], d0, kn * W, brow, fb);
                        issued = kn + 1;
                    }
                }
            }
        } else {
            const float *entry = xwp_entries<C>(sm, k & 1);
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = entry[s * DT + v * G + lg];
            St *op = ost.plane(k, 0) + (s * L) * DT + lg * V;
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
                store_lanes<St, V>(op + j * DT, h);
            }
            fence_proxy_async_smem();
            // the thread whose sub-chunk holds step T-1 owns the final state
            if (last != nullptr && lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
                for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
            }
        }
    }
    // the last window's tile (not after an abort), then every store and
    // every issued copy complete before the CTA's shared memory goes away
    const bool aborted = bar_sync_or(1, NW, failed);
    if (producer) {
        if (!aborted && nwin > 0) ost.store(omaps, nwin - 1, d0, (nwin - 1) * W, brow);
        bulk_wait<0>();
        xwp_drain(sm, aborted ? k : nwin, issued, wc);
    }
}

// ============================================================================
// Backward
// ============================================================================
template <class C, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
xwp_bwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_out,
               const __grid_constant__ CUtensorMap tm_go, const __grid_constant__ CUtensorMap tm_ga,
               const __grid_constant__ CUtensorMap tm_gb, const __grid_constant__ WinGeom geom, DevStatus *status,
               uint64_t timeout_ns, const __grid_constant__ StateArgs sx) {
    static_assert(!C::SEQ && !C::PT && C::EX && C::NIN == 3, "pipelined exact backward: exact windowed shape");
    static_assert(C::DT % 32 == 0, "walker threads are whole warps");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    constexpr int NM = (C::SMAX * L + 31) / 32;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    const int NW = NT + DT;
    win_init<C>(sm, NW / 32, S);
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D, W = sm.W, nwin = sm.nwin, nstage = sm.nstage;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const bool walker = tid >= NT;
    const bool producer = tid == NT;
    const CUtensorMap *const imaps[3] = {&tm_a, &tm_out, &tm_go};
    const CUtensorMap *const omaps[2] = {&tm_ga, &tm_gb};
    const OutStage<2, St, 3> ost = make_out_stage<2, St, 3>(smem_raw, geom);  // planes grad_a, grad_b
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    // time row of input tile i of processed window kw: a one step later, out
    // one step earlier, grad_out as is
    auto row_of = [nwin, W](int kw, int i) { return (nwin - 1 - kw) * W + (i == 0 ? 1 : (i == 1 ? -1 : 0)); };

    int issued = 0;
    if (producer) {
        for (int i = 0; i < 3; ++i) prefetch_tensormap(imaps[i]);
        for (int k = 0; k < nwin && k < nstage; ++k) {
            const uint32_t fb = sm.full_bar(k);
            mbar_arrive_expect_tx(fb, sm.stage_bytes);
            for (int i = 0; i < 3; ++i) tma_load_3d(smem_addr(sm.tile<C>(k, i)), imaps[i], d0, row_of(k, i), brow, fb);
            issued = k + 1;
        }
    }

    const int s = walker ? 0 : tid / G;
    const int lg = walker ? 0 : tid - s * G;
    const int d = d0 + lg * V;
    const bool lane_ok = !walker && d < D;
    const int wi = tid - NT;
    float carry = 0.0f;  // walker: adjoint entering the window from above
    float g[V];
#pragma unroll
    for (int v = 0; v < V; ++v) g[v] = 0.0f;
    float h0v[V];  // h_{-1}
#pragma unroll
    for (int v = 0; v < V; ++v) h0v[v] = 0.0f;
    const int wrow = walker ? 0 : ((tid & ~31) / G) * L;
    int32_t pos0_next = 1, pos1_next = 1;
    int32_t wpos[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) wpos[m] = 1;
    if constexpr (EXT) {
        static_assert((G >= 32 ? 1 : 32 / G) * L <= 32, "one ballot covers a replay warp's rows");
        const int wb0 = (nwin - 1) * W;
        if (walker) {
            if (sx.grad_last != nullptr) {
                const int ch = lane_channel<C>(d0, wi);
                carry = ch < D ? sx.grad_last[static_cast<size_t>(brow) * D + ch] : 0.0f;
            }
            // the walker masks a'_{t+1}: positions of rows + 1
#pragma unroll
            for (int m = 0; m < NM; ++m) wpos[m] = (32 * m + lane < W) ? seg.at(wb0 + 32 * m + lane + 1) : 1;
        } else {
            if (sx.h0 != nullptr && lane_ok) {
#pragma unroll
                for (int v = 0; v < V; ++v) h0v[v] = sx.h0[static_cast<size_t>(brow) * D + d + v];
            }
            pos0_next = seg.at(wb0 + wrow + lane);
            pos1_next = seg.at(wb0 + wrow + lane + 1);
        }
    }

    bool failed = false;
    int k = 0;
    for (; k < nwin; ++k) {
        const int stage = k % nstage;
        const uint32_t par = (k / nstage) & 1;
        const int wbase = (nwin - 1 - k) * W;
        const int rbase = wbase + s * L;
        const int n = min(max(T - rbase, 0), L);
        uint32_t r0bits = 0, r1bits = 0;
        if constexpr (EXT) {
            if (!walker) {
                r0bits = __ballot_sync(0xffffffffu, pos0_next == 0) >> (s * L - wrow);
                r1bits = __ballot_sync(0xffffffffu, pos1_next == 0) >> (s * L - wrow);
                const int wb = wbase - W + wrow + lane;
                pos0_next = seg.at(wb);
                pos1_next = seg.at(wb + 1);
            } else {
                xwp_write_masks<C, NM>(xwp_masks<C>(sm, wi / 32), wpos, S, lane);
#pragma unroll
                for (int m = 0; m < NM; ++m)
                    wpos[m] = (32 * m + lane < W) ? seg.at(wbase - W + 32 * m + lane + 1) : 1;
            }
        }
        const bool ok = mbar_wait(sm.full_bar(stage), par, wc, kSiteConsumerFull);
        float xa[L][V], xh[L][V], xg[L][V];
        if (!walker) {
            if (ok) {
                const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;  // a_{t+1}
                const St *th = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;  // h_{t-1}
                const St *tg = sm.tile<C>(stage, 2) + (s * L) * DT + lg * V;  // grad_out_t
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    unpack_lanes<St, V>(ta + j * DT, xa[j]);
                    unpack_lanes<St, V>(th + j * DT, xh[j]);
                    unpack_lanes<St, V>(tg + j * DT, xg[j]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
            // rows from na on take a' = 1: steps past T (identity steps) and,
            // with the carried state, step T-1 (grad_last enters through a'_T = 1)
            int na = n;
            if constexpr (EXT) {
                if (n > 0 && rbase + n == T) na = n - 1;
                if (r1bits != 0) {
#pragma unroll
                    for (int j = 0; j < L; ++j) {
#pragma unroll
                        for (int v = 0; v < V; ++v) xa[j][v] = ((r1bits >> j) & 1u) ? 0.0f : xa[j][v];
                    }
                }
                if (rbase == 0) {
#pragma unroll
                    for (int v = 0; v < V; ++v) xh[0][v] = h0v[v];
                }
            }
            if (na < L) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        xa[j][v] = j < na ? xa[j][v] : 1.0f;
                        xg[j][v] = j < n ? xg[j][v] : 0.0f;
                    }
                }
            }
        } else if (ok) {
            carry = exact_walk<C, true, EXT, EXT>(sm.tile<C>(stage, 0), sm.tile<C>(stage, 2),
                                                  xwp_entries<C>(sm, k & 1), xwp_masks<C>(sm, wi / 32), S, wi,
                                                  T - wbase, carry);
        }
        if (bar_sync_or(1, NW, !ok)) { failed = true; break; }
        if (walker) {
            if (lane == 0) mbar_arrive(sm.empty_bar(stage));
            if (producer) {
                if (k > 0) {
                    ost.store(omaps, k - 1, d0, wbase + W, brow);
                    bulk_wait_read<1>();
                }
                const int kn = k + nstage;
                if (kn < nwin) {
                    if (mbar_wait(sm.empty_bar(stage), par, wc, kSiteProducerEmpty)) {
                        const uint32_t fb = sm.full_bar(stage);
                        mbar_arrive_expect_tx(fb, sm.stage_bytes);
                        for (int i = 0; i < 3; ++i)
                            tma_load_3d(smem_addr(sm.tile<C>(stage, i)), imaps[i], d0, row_of(kn, i), brow, fb);
                        issued = kn + 1;
                    }
                }
            }
        } else {
            const float *entry = xwp_entries<C>(sm, k & 1);
#pragma unroll
            for (int v = 0; v < V; ++v) g[v] = entry[s * DT + v * G + lg];
            St *sga = ost.plane(k, 0) + (s * L) * DT + lg * V;
            St *sgb = ost.plane(k, 1) + (s * L) * DT + lg * V;
            if (EXT && r0bits != 0) bwd_rows<C, true, true>(xa, xh, xg, g, n, lane_ok, sgb, sga, D, r0bits);
            else bwd_rows<C, false, true>(xa, xh, xg, g, n, lane_ok, sgb, sga, D, 0u);
            fence_proxy_async_smem();
            if constexpr (EXT) {
                if (rbase == 0 && sx.grad_h0 != nullptr && lane_ok) store_grad_h0<C>(sx, seg, row0, brow, d, D, g);
            }
        }
    }
    const bool aborted = bar_sync_or(1, NW, failed);
    if (producer) {
        if (!aborted && nwin > 0) ost.store(omaps, nwin - 1, d0, 0, brow);
        bulk_wait<0>();
        xwp_drain(sm, aborted ? k : nwin, issued, wc);
    }
}

}  // namespace lrscan
