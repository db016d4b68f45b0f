// Exact windowed scan in wavefront order (wfx tiles).
//
// A CTA owns one batch row and DT lanes; each window of W = S * L rows is
// split into S sub-chunks of L rows, one warp per sub-chunk (32 lane groups
// of V lanes).  Every warp copies its rows of the window into registers as
// soon as the stage lands and releases the stage at once; the recurrence
// itself runs as one chain per lane through the warps in order: warp s takes
// the state leaving warp s - 1 (the previous window's last warp for warp 0),
// runs its L rows with the sequential step, writes them into a shared-memory
// output stage, and hands its state to the next warp (shared memory plus an
// mbarrier per warp, waits bounded).  The warp that ends a window issues its
// bulk tensor store.  Each lane's values are the sequential definition's own
// fused multiply-adds in order, so every result is bit-identical to the
// sequential scan; unlike the exact windowed tiles there is no separate walk
// and no replay: the chain is the only serial part, and the loads, the
// conversions and the stores of the other warps overlap it.
//
// Backward windows run last-to-first and sub-chunks last-to-first, with the
// decay tile one row late (a_{t+1}) and the out tile one row early
// (h_{t-1}); EXT instantiations carry h0 / grad_last / grad_h0 and segment
// resets with the rules of the windowed kernels.
#pragma once

#include "window_kernels.cuh"

namespace lrscan {

enum WavefrontSite : int { kSiteHandoff = 7 };

template <class C, bool BWD, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
wfx_kernel(const __grid_constant__ CUtensorMap tm_0, const __grid_constant__ CUtensorMap tm_1,
           const __grid_constant__ CUtensorMap tm_2, const __grid_constant__ CUtensorMap tm_3,
           const __grid_constant__ CUtensorMap tm_4, float *__restrict__ last, const __grid_constant__ WinGeom geom,
           DevStatus *status, uint64_t timeout_ns, const __grid_constant__ StateArgs sx) {
    static_assert(!C::SEQ && !C::PT && C::EX, "wavefront tile: exact windowed shape");
    static_assert(C::G == 32, "one warp per sub-chunk row of lanes");
    static_assert(C::NIN == (BWD ? 3 : 2), "forward tiles a, b; backward a, out, grad_out");
    static_assert(C::L <= 32, "one ballot covers a sub-chunk's rows");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT;
    constexpr int NP = BWD ? 2 : 1;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * 32;
    float *xfer = reinterpret_cast<float *>(smem_raw + geom.scan_off);  // [S][DT] state handed to warp s
    auto hb = [&](int q) { return smem_addr(smem_raw + geom.scan_off + S * DT * 4 + q * 8); };
    // staged[k & 1]: the other warps' output rows of window k are written
    auto staged = [&](int q) { return smem_addr(smem_raw + geom.scan_off + S * DT * 4 + S * 8 + q * 8); };
    if (threadIdx.x == 0) {
        for (int q = 0; q < S; ++q) mbar_init(hb(q), 32);
        for (int q = 0; q < 2; ++q) mbar_init(staged(q), (S - 1) * 32);
    }
    win_init<C>(sm, S, S);  // full / empty barriers, abort flag; syncs the CTA
    pdl_trigger();
    pdl_wait();  // inputs may come from the previous kernel in the stream
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D, W = sm.W, nwin = sm.nwin;

    if (static_cast<int>(threadIdx.x) >= NT) {  // producer warp
        if (static_cast<int>(threadIdx.x) == NT) {
            if constexpr (BWD) {
                // a one step later, out one step earlier, grad_out as is
                const CUtensorMap *const maps[3] = {&tm_0, &tm_1, &tm_2};
                win_producer<C>(sm, maps, d0, brow,
                                [W, nwin](int k, int i) { return (nwin - 1 - k) * W + (i == 0 ? 1 : (i == 1 ? -1 : 0)); },
                                wc);
            } else {
                const CUtensorMap *const maps[2] = {&tm_0, &tm_1};
                win_producer<C>(sm, maps, d0, brow, [W](int k, int) { return k * W; }, wc);
            }
        }
        return;
    }

    const int s = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int d = d0 + lane * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    // chain order: forward sub-chunks 0 .. S-1, backward S-1 .. 0
    const bool first = BWD ? s == S - 1 : s == 0;   // starts a window's chain
    const bool closer = BWD ? s == 0 : s == S - 1;  // ends it and stores the window
    const int succ = BWD ? (s + S - 1) % S : (s + 1) % S;
    const OutStage<NP, St, 3> ost = make_out_stage<NP, St, 3>(smem_raw, geom);
    const CUtensorMap *omaps[NP];
    if constexpr (BWD) {
        omaps[0] = &tm_3;
        omaps[1] = &tm_4;
    } else {
        omaps[0] = &tm_2;
    }
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    float h[V];  // forward state / backward adjoint
#pragma unroll
    for (int v = 0; v < V; ++v) h[v] = 0.0f;
    float h0v[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h0v[v] = 0.0f;
    if constexpr (EXT) {
        if (lane_ok) {
            const size_t hs = static_cast<size_t>(brow) * D + d;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (BWD) {
                    if (first && sx.grad_last != nullptr) h[v] = sx.grad_last[hs + v];
                    if (sx.h0 != nullptr) h0v[v] = sx.h0[hs + v];
                } else if (first && sx.h0 != nullptr) {
                    h[v] = sx.h0[hs + v];
                }
            }
        }
    }
    // EXT positions of this warp's rows, one window ahead (lane l: row l,
    // backward also row l + 1)
    auto wbase_of = [&](int k) { return BWD ? (nwin - 1 - k) * W : k * W; };
    int32_t pos0 = 1, pos1 = 1;
    if constexpr (EXT) {
        const int r = wbase_of(0) + s * L + lane;
        pos0 = lane < L ? seg.at(r) : 1;
        if (BWD) pos1 = lane < L ? seg.at(r + 1) : 1;
    }

    bool failed = false;
    int stage = 0, use = 0;
    for (int k = 0; k < nwin; ++k) {
        const int wbase = wbase_of(k);
        const int rbase = wbase + s * L;
        const int n = min(max(T - rbase, 0), L);
        uint32_t r0bits = 0, r1bits = 0;
        if constexpr (EXT) {
            r0bits = __ballot_sync(0xffffffffu, pos0 == 0);
            if (BWD) r1bits = __ballot_sync(0xffffffffu, pos1 == 0);
            if (k + 1 < nwin) {
                const int r = wbase_of(k + 1) + s * L + lane;
                pos0 = lane < L ? seg.at(r) : 1;
                if (BWD) pos1 = lane < L ? seg.at(r + 1) : 1;
            }
        }
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) { failed = true; break; }
        float xa[L][V], xb[L][V], xh[BWD ? L : 1][V];
        {
            const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lane * V;
            const St *tb = sm.tile<C>(stage, C::NIN - 1) + (s * L) * DT + lane * V;
#pragma unroll
            for (int j = 0; j < L; ++j) {
                unpack_lanes<St, V>(ta + j * DT, xa[j]);
                unpack_lanes<St, V>(tb + j * DT, xb[j]);
            }
            if constexpr (BWD) {
                const St *th = sm.tile<C>(stage, 1) + (s * L) * DT + lane * V;
#pragma unroll
                for (int j = 0; j < L; ++j) unpack_lanes<St, V>(th + j * DT, xh[j]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
        // decays and addends as the sequential definition takes them: a' = 0
        // at a reset (backward: a'_{t+1} where step t+1 starts a segment),
        // step T-1 of the backward with carried state takes a'_T = 1, and
        // rows past T are identity steps
        int na = n;
        if constexpr (EXT && BWD) {
            if (n > 0 && rbase + n == T) na = n - 1;
        }
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const bool z = EXT && (((BWD ? r1bits : r0bits) >> j) & 1u);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                xa[j][v] = j < na ? (z ? 0.0f : xa[j][v]) : 1.0f;
                xb[j][v] = j < n ? xb[j][v] : 0.0f;
            }
        }
        if constexpr (EXT && BWD) {
            if (rbase == 0) {
#pragma unroll
                for (int v = 0; v < V; ++v) xh[0][v] = h0v[v];  // h_{-1} = h0
            }
        }
        // the state entering this sub-chunk
        if (!(first && k == 0)) {
            const uint32_t par = (first ? k - 1 : k) & 1;
            ok = mbar_wait(hb(s), par, wc, kSiteHandoff);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { failed = true; break; }
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = xfer[s * DT + lane * V + v];
        }
        // the chain through this sub-chunk's rows: the fused multiply-adds
        // alone, so that the state moves on before the conversions and stores
        float hr[L][V];
#pragma unroll
        for (int q = 0; q < L; ++q) {
            const int j = BWD ? L - 1 - q : q;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
                hr[j][v] = h[v];
            }
        }
        if (closer) {
            // the store of window k-2 has finished reading the buffer window
            // k+1 takes (the latest store, of k-1, may still be reading)
            __syncwarp();
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
        }
        // hand the state to the next sub-chunk in chain order
        if (!(closer && k + 1 == nwin)) {
#pragma unroll
            for (int v = 0; v < V; ++v) xfer[succ * DT + lane * V + v] = h[v];
            mbar_arrive(hb(succ));
        }
        // this sub-chunk's outputs into the window's stage
        St *o0 = ost.plane(k, 0) + (s * L) * DT + lane * V;
#pragma unroll
        for (int j = 0; j < L; ++j) {
            if constexpr (BWD) {
                float ga[V];
                const bool z = EXT && ((r0bits >> j) & 1u);  // a_t unused at a segment start
#pragma unroll
                for (int v = 0; v < V; ++v) ga[v] = z ? 0.0f : __fmul_rn(hr[j][v], xh[j][v]);
                store_lanes<St, V>(o0 + j * DT, ga);
                store_lanes<St, V>(ost.plane(k, 1) + (s * L + j) * DT + lane * V, hr[j]);
            } else {
                store_lanes<St, V>(o0 + j * DT, hr[j]);
                if (last != nullptr && lane_ok && j == n - 1 && rbase + n == T) {
#pragma unroll
                    for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = hr[j][v];
                }
            }
        }
        if constexpr (EXT && BWD) {
            if (rbase == 0 && sx.grad_h0 != nullptr && lane_ok) store_grad_h0<C>(sx, seg, row0, brow, d, D, h);
        }
        fence_proxy_async_smem();  // the staged rows, for the closing warp's bulk store
        if (!closer) {
            mbar_arrive(staged(k & 1));
        } else {
            ok = mbar_wait(staged(k & 1), (k >> 1) & 1, wc, kSiteHandoff);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { failed = true; break; }
            __syncwarp();
            if (lane == 0) ost.store(omaps, k, d0, wbase, brow);
            __syncwarp();
        }
    }
    if (closer && lane == 0) bulk_wait<0>();
    (void)failed;
}

}  // namespace lrscan
