// Time-tiled scan kernels: a CTA owns one batch row and DT channel lanes and
// walks the whole sequence in windows of W = S*L time steps.  A producer warp
// streams the windows' input tiles into a ring of NSTAGE shared-memory stages
// with 3-D bulk tensor copies (TMA) completed on mbarriers; consumer threads
// keep the recurrence state in fp32 registers.
//
//  S == 1  ("seq"): each consumer thread owns V lanes and runs the recurrence
//          straight through every window, one fused multiply-add per step --
//          bit-identical to the sequential definition.
//  S  > 1  ("window"): the W rows of a window are split into S sub-chunks of
//          L steps.  Thread (s, lane group) summarizes its sub-chunk as the
//          affine map h -> P*h + Q (triton_training_scan.py,
//          _real_chunk_summary), the sub-chunk entry states follow from the
//          window's carried state through the maps of the earlier sub-chunks
//          (_real_chunk_prefix, here inside one CTA), and every thread
//          replays its sub-chunk (_real_chunk_replay).  One pass over HBM:
//          3 elements per (t, d) forward, 5 backward.
//
// Backward windows run last-to-first.  The decay tile is loaded one row late
// (a_{t+1}) and the out tile one row early (h_{t-1}), so the tensor copy's zero
// fill supplies a_T = 0 and h_{-1} = 0 at the sequence ends; the reverse
// recurrence g_t = fma(a_{t+1}, g_{t+1}, grad_out_t) then has the same shape
// as the forward one.
#pragma once

#include "scan_common.cuh"

namespace lrscan {

template <typename St_, int DT_, int V_, int S_, int L_, int NSTAGE_, int NIN_>
struct WinShape {
    using St = St_;
    static constexpr int DT = DT_;        // lanes per CTA
    static constexpr int V = V_;          // lanes per thread
    static constexpr int S = S_;          // sub-chunks per window
    static constexpr int L = L_;          // steps per sub-chunk
    static constexpr int NSTAGE = NSTAGE_;
    static constexpr int NIN = NIN_;      // input tiles per window (2 fwd, 3 bwd)
    static constexpr int G = DT / V;      // lane groups per row
    static constexpr int NT = S * G;      // consumer threads
    static constexpr int NWARP_C = NT / 32;
    static constexpr int THREADS = NT + 32;  // + one producer warp
    static constexpr int W = S * L;       // rows per window
    static constexpr int TILE_BYTES = W * DT * (int)sizeof(St);
    static constexpr int STAGE_BYTES = NIN * TILE_BYTES;
    static constexpr int TILES_BYTES = NSTAGE * STAGE_BYTES;
    static constexpr int BAR_OFF = TILES_BYTES;
    static constexpr int SCAN_OFF = BAR_OFF + 2 * NSTAGE * 8;
    static constexpr int SCAN_BYTES = (S > 1) ? (2 * 2 * S * DT + 2 * DT) * 4 : 0;
    static constexpr int FLAG_OFF = SCAN_OFF + SCAN_BYTES;
    static constexpr int SMEM_BYTES = FLAG_OFF + 16;

    static_assert(DT % V == 0, "lane tile must split into lane groups");
    static_assert(NT % 32 == 0, "consumers must be whole warps");
    static_assert(TILE_BYTES % 128 == 0, "tiles must stay 128-byte aligned");
    static_assert((DT * (int)sizeof(St)) % 16 == 0, "tensor-copy rows are multiples of 16 bytes");
    static_assert(DT <= 256 && W <= 256, "tensor-copy box limit");
    static_assert(S == 1 || L <= 16, "window sub-chunks are held in registers");
};

struct WinSmem {
    unsigned char *base;
    template <class C> __device__ __forceinline__ typename C::St *tile(int stage, int which) const {
        return reinterpret_cast<typename C::St *>(base + stage * C::STAGE_BYTES + which * C::TILE_BYTES);
    }
    template <class C> __device__ __forceinline__ uint32_t full_bar(int stage) const {
        return smem_addr(base + C::BAR_OFF + stage * 8);
    }
    template <class C> __device__ __forceinline__ uint32_t empty_bar(int stage) const {
        return smem_addr(base + C::BAR_OFF + (C::NSTAGE + stage) * 8);
    }
    // P,Q exchange buffers [parity][S][DT] and carried state [parity][DT]
    template <class C> __device__ __forceinline__ float *sP(int par) const {
        return reinterpret_cast<float *>(base + C::SCAN_OFF) + par * C::S * C::DT;
    }
    template <class C> __device__ __forceinline__ float *sQ(int par) const {
        return reinterpret_cast<float *>(base + C::SCAN_OFF) + (2 + par) * C::S * C::DT;
    }
    template <class C> __device__ __forceinline__ float *sCarry(int par) const {
        return reinterpret_cast<float *>(base + C::SCAN_OFF) + 4 * C::S * C::DT + par * C::DT;
    }
    template <class C> __device__ __forceinline__ volatile int *abort_flag() const {
        return reinterpret_cast<volatile int *>(base + C::FLAG_OFF);
    }
};

// Producer: one elected lane streams `nwin` windows into the stage ring, in
// processing order.  `row_of(k, i)` gives the time coordinate of input tile i
// of the k-th processed window.  Before returning (normally or on abort) it
// waits, bounded, for every copy it issued, so none lands after the CTA exits.
template <class C, class RowOf>
__device__ __forceinline__ void win_producer(const WinSmem &sm, const CUtensorMap *const (&maps)[C::NIN],
                                             int nwin, int x0, int z, RowOf row_of, const WaitCtx &wc) {
    for (int i = 0; i < C::NIN; ++i) prefetch_tensormap(maps[i]);
    int issued = 0;
    for (int k = 0; k < nwin; ++k) {
        const int stage = k % C::NSTAGE;
        const int use = k / C::NSTAGE;
        if (use > 0 && !mbar_wait(sm.empty_bar<C>(stage), (use - 1) & 1, wc, kSiteProducerEmpty)) break;
        const uint32_t fb = sm.full_bar<C>(stage);
        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
#pragma unroll
        for (int i = 0; i < C::NIN; ++i)
            tma_load_3d(smem_addr(sm.tile<C>(stage, i)), maps[i], x0, row_of(k, i), z, fb);
        issued = k + 1;
    }
    // Drain: the most recent fill of each stage must have landed.
    const int first = issued > C::NSTAGE ? issued - C::NSTAGE : 0;
    for (int k = first; k < issued; ++k) {
        const int stage = k % C::NSTAGE;
        const uint32_t fb = sm.full_bar<C>(stage);
        if (mbar_try_wait(fb, (k / C::NSTAGE) & 1)) continue;
        // A bounded wait that ignores the abort flag: copies in flight always land.
        const uint64_t start = global_timer_ns();
        while (!mbar_try_wait(fb, (k / C::NSTAGE) & 1)) {
            if (global_timer_ns() - start > wc.timeout_ns) {
                record_error(wc, kErrTimeout, kSiteDrain);
                break;
            }
        }
    }
}

template <class C>
__device__ __forceinline__ void win_init(const WinSmem &sm) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(sm.full_bar<C>(s), 1);
            mbar_init(sm.empty_bar<C>(s), C::NWARP_C);
        }
        *sm.abort_flag<C>() = 0;
        fence_mbar_init();
    }
    if constexpr (C::S > 1) {
        // carried state starts at zero (h_{-1} = 0 forward, g_T = 0 backward)
        for (int i = threadIdx.x; i < 2 * C::DT; i += blockDim.x) sm.sCarry<C>(0)[i] = 0.0f;
    }
    __syncthreads();
}

// ============================================================================
// Forward
// ============================================================================
template <class C>
__global__ void __launch_bounds__(C::THREADS)
win_fwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               typename C::St *__restrict__ out, float *__restrict__ last, int T, int D, int nwin,
               DevStatus *status, uint64_t timeout_ns) {
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, S = C::S, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm{smem_raw};
    win_init<C>(sm);
    const WaitCtx wc{status, sm.abort_flag<C>(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == C::NWARP_C) {  // producer warp
        if (lane == 0) {
            const CUtensorMap *const maps[2] = {&tm_a, &tm_b};
            win_producer<C>(sm, maps, nwin, d0, brow, [](int k, int) { return k * C::W; }, wc);
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    float h[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h[v] = 0.0f;
    bool failed = false;

    for (int k = 0; k < nwin; ++k) {
        const int stage = k % C::NSTAGE;
        const int t0 = k * C::W;
        const int rbase = t0 + s * L;
        const int n = min(max(T - rbase, 0), L);
        const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;
        const St *tb = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;
        St *op = out + (row0 + rbase) * D + d;
        bool ok = mbar_wait(sm.full_bar<C>(stage), (k / C::NSTAGE) & 1, wc, kSiteConsumerFull);

        if constexpr (S == 1) {
            if (!ok) { failed = true; break; }
            if (n == L) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    float x[V], y[V];
                    unpack_lanes<St, V>(ta + j * DT, x);
                    unpack_lanes<St, V>(tb + j * DT, y);
#pragma unroll
                    for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(x[v], h[v], y[v]);
                    if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
                }
            } else {
                for (int j = 0; j < n; ++j) {
                    float x[V], y[V];
                    unpack_lanes<St, V>(ta + j * DT, x);
                    unpack_lanes<St, V>(tb + j * DT, y);
#pragma unroll
                    for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(x[v], h[v], y[v]);
                    if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty_bar<C>(stage));
        } else {
            float xa[L][V], xb[L][V];
            if (ok) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    unpack_lanes<St, V>(ta + j * DT, xa[j]);
                    unpack_lanes<St, V>(tb + j * DT, xb[j]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar<C>(stage));
            // sub-chunk summary h -> P*h + Q (empty tail sub-chunks are the identity map)
            float P[V], Q[V];
#pragma unroll
            for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
            for (int j = 0; j < L; ++j) {
                if (j < n) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        P[v] = __fmul_rn(xa[j][v], P[v]);
                        Q[v] = __fmaf_rn(xa[j][v], Q[v], xb[j][v]);
                    }
                }
            }
            const int par = k & 1;
            float *sp = sm.sP<C>(par), *sq = sm.sQ<C>(par);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                sp[s * DT + lg * V + v] = P[v];
                sq[s * DT + lg * V + v] = Q[v];
            }
            if (bar_sync_or(1, C::NT, !ok)) { failed = true; break; }
            // entry state of this sub-chunk: the window's carried state pushed
            // through the maps of sub-chunks 0..s-1, in order
            const float *carry = sm.sCarry<C>(par);
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = carry[lg * V + v];
#pragma unroll
            for (int sp_i = 0; sp_i < S - 1; ++sp_i) {
                if (sp_i < s) {
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        h[v] = __fmaf_rn(sp[sp_i * DT + lg * V + v], h[v], sq[sp_i * DT + lg * V + v]);
                }
            }
            // replay
#pragma unroll
            for (int j = 0; j < L; ++j) {
                if (j < n) {
#pragma unroll
                    for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
                    if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
                }
            }
            if (s == S - 1) {
                float *nc = sm.sCarry<C>(par ^ 1);
#pragma unroll
                for (int v = 0; v < V; ++v) nc[lg * V + v] = h[v];
            }
            // the thread whose sub-chunk holds step T-1 owns the final state
            if (last != nullptr && lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
                for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
            }
        }
    }
    if constexpr (S == 1) {
        if (!failed && last != nullptr && lane_ok) {
#pragma unroll
            for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
        }
    }
}

// ============================================================================
// Backward
// ============================================================================
template <class C>
__global__ void __launch_bounds__(C::THREADS)
win_bwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_out,
               const __grid_constant__ CUtensorMap tm_go, typename C::St *__restrict__ grad_a,
               typename C::St *__restrict__ grad_b, int T, int D, int nwin, DevStatus *status,
               uint64_t timeout_ns) {
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, S = C::S, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm{smem_raw};
    win_init<C>(sm);
    const WaitCtx wc{status, sm.abort_flag<C>(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == C::NWARP_C) {
        if (lane == 0) {
            const CUtensorMap *const maps[3] = {&tm_a, &tm_out, &tm_go};
            // tile 0: a shifted one step later; tile 1: out one step earlier; tile 2: grad_out
            win_producer<C>(sm, maps, nwin, d0, brow,
                            [nwin](int k, int i) { return (nwin - 1 - k) * C::W + (i == 0 ? 1 : (i == 1 ? -1 : 0)); },
                            wc);
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    float g[V];
#pragma unroll
    for (int v = 0; v < V; ++v) g[v] = 0.0f;

    for (int k = 0; k < nwin; ++k) {
        const int stage = k % C::NSTAGE;
        const int t0 = (nwin - 1 - k) * C::W;
        const int rbase = t0 + s * L;
        const int n = min(max(T - rbase, 0), L);
        const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;  // a_{t+1}
        const St *th = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;  // h_{t-1}
        const St *tg = sm.tile<C>(stage, 2) + (s * L) * DT + lg * V;  // grad_out_t
        const size_t gofs = (row0 + rbase) * D + d;
        bool ok = mbar_wait(sm.full_bar<C>(stage), (k / C::NSTAGE) & 1, wc, kSiteConsumerFull);

        if constexpr (S == 1) {
            if (!ok) break;
            if (n == L) {
#pragma unroll
                for (int j = L - 1; j >= 0; --j) {
                    float x[V], hp[V], go[V], ga[V];
                    unpack_lanes<St, V>(ta + j * DT, x);
                    unpack_lanes<St, V>(th + j * DT, hp);
                    unpack_lanes<St, V>(tg + j * DT, go);
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        g[v] = __fmaf_rn(x[v], g[v], go[v]);
                        ga[v] = __fmul_rn(g[v], hp[v]);
                    }
                    if (lane_ok) {
                        store_lanes<St, V>(grad_b + gofs + static_cast<size_t>(j) * D, g);
                        store_lanes<St, V>(grad_a + gofs + static_cast<size_t>(j) * D, ga);
                    }
                }
            } else {
                for (int j = n - 1; j >= 0; --j) {
                    float x[V], hp[V], go[V], ga[V];
                    unpack_lanes<St, V>(ta + j * DT, x);
                    unpack_lanes<St, V>(th + j * DT, hp);
                    unpack_lanes<St, V>(tg + j * DT, go);
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        g[v] = __fmaf_rn(x[v], g[v], go[v]);
                        ga[v] = __fmul_rn(g[v], hp[v]);
                    }
                    if (lane_ok) {
                        store_lanes<St, V>(grad_b + gofs + static_cast<size_t>(j) * D, g);
                        store_lanes<St, V>(grad_a + gofs + static_cast<size_t>(j) * D, ga);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty_bar<C>(stage));
        } else {
            float xa[L][V], xh[L][V], xg[L][V];
            if (ok) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    unpack_lanes<St, V>(ta + j * DT, xa[j]);
                    unpack_lanes<St, V>(th + j * DT, xh[j]);
                    unpack_lanes<St, V>(tg + j * DT, xg[j]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar<C>(stage));
            // reverse sub-chunk summary: g at the sub-chunk's first step as
            // P * (g just after the sub-chunk) + Q
            float P[V], Q[V];
#pragma unroll
            for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
            for (int j = L - 1; j >= 0; --j) {
                if (j < n) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        P[v] = __fmul_rn(xa[j][v], P[v]);
                        Q[v] = __fmaf_rn(xa[j][v], Q[v], xg[j][v]);
                    }
                }
            }
            const int par = k & 1;
            float *sp = sm.sP<C>(par), *sq = sm.sQ<C>(par);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                sp[s * DT + lg * V + v] = P[v];
                sq[s * DT + lg * V + v] = Q[v];
            }
            if (bar_sync_or(1, C::NT, !ok)) break;
            const float *carry = sm.sCarry<C>(par);
#pragma unroll
            for (int v = 0; v < V; ++v) g[v] = carry[lg * V + v];
            // push the carried adjoint through sub-chunks S-1 .. s+1
#pragma unroll
            for (int i = S - 1; i > 0; --i) {
                if (i > s) {
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        g[v] = __fmaf_rn(sp[i * DT + lg * V + v], g[v], sq[i * DT + lg * V + v]);
                }
            }
#pragma unroll
            for (int j = L - 1; j >= 0; --j) {
                if (j < n) {
                    float ga[V];
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        g[v] = __fmaf_rn(xa[j][v], g[v], xg[j][v]);
                        ga[v] = __fmul_rn(g[v], xh[j][v]);
                    }
                    if (lane_ok) {
                        store_lanes<St, V>(grad_b + gofs + static_cast<size_t>(j) * D, g);
                        store_lanes<St, V>(grad_a + gofs + static_cast<size_t>(j) * D, ga);
                    }
                }
            }
            if (s == 0) {
                float *nc = sm.sCarry<C>(par ^ 1);
#pragma unroll
                for (int v = 0; v < V; ++v) nc[lg * V + v] = g[v];
            }
        }
    }
}

}  // namespace lrscan
