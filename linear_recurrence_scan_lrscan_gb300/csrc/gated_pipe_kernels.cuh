// Generated-decay forward with warp roles (triton_training_scan.py,
// _samu_forward with the decay of _samu_precompute_decay rebuilt in the
// kernel, as in gated_kernels.cuh): one CTA per (batch row, 32-lane tile)
// takes all T steps in windows of W rows, one lane per thread.  The windowed
// tiles walk their windows one after another with two CTA barriers each; here
// no warp waits on a CTA barrier:
//   producer warp   streams the b tiles into a ring of NST stages (bulk
//                   tensor copies, NST windows ahead);
//   NS summary      summary warp s takes windows s, s + NS, ...: builds the
//   warps           window's decays (a = 2^(-nu2 E_t), E_t = exp(eta_t), one
//                   exponential per row shared by shuffles), keeps them in the
//                   window's slot, reduces the window to its map
//                   h -> P h + Q and publishes it;
//   scan warp       carries the state through the window maps in order (one
//                   fma per lane and window) and publishes the state entering
//                   each window;
//   NR replay       replay warp r takes windows r, r + NR, ...: replays the
//   warps           window from its entering state with the slot's decays,
//                   writes each out_t over b_t in the stage and sends the
//                   window out with a bulk tensor store.
// Summaries run up to NM windows ahead of the replays (NM window slots of
// decays, map and entering state), so the scan warp never waits on a replay.
// A replay warp frees its window's slot at once and its stage when it starts
// its window after next, once the store that read it is done (one store of
// the warp stays in flight).  Every wait is
// bounded (LRSCAN_ETIMEOUT in the status word; the kernel returns).  The
// window maps re-associate the recurrence: results agree with the sequential
// definition to rounding.
#pragma once

#include "gated_kernels.cuh"

namespace lrscan {

// Compiled shape: storage type, rows per window, summary warps, replay
// warps, ring stages, window slots, CTAs per SM the registers must allow.  32
// lanes per CTA, one per thread.
template <class St_, int W_, int NS_, int NR_, int NST_, int NM_, int MINB_>
struct GPipeShape {
    using St = St_;
    static constexpr int DT = 32, W = W_, NS = NS_, NR = NR_, NST = NST_, NM = NM_, MINB = MINB_;
    static constexpr int THREADS = (NS + NR + 2) * 32;
    static_assert(W <= 32 && W % 8 == 0, "one exponential per row and lane of a warp");
    static_assert(NM <= NST, "a window's tile has landed before its slot comes round again");
    static_assert(NST > 2 * NR, "a stage is released when its replay warp starts its window after next");
};

// Shared-memory layout, host and device.
struct GPipeGeom {
    int tile_bytes;   // one window of b (and then out): W * 32 * elem
    int dec_off;      // window decays [NM][W][32] float
    int bar_off;      // full[NST], stage_free[NST], map_full[NM], entry_full[NM], slot_free[NM]
    int map_off;      // window maps [NM][32] float2
    int entry_off;    // entering states [NM][32] float
    int flag_off;     // abort flag
    int smem_bytes;
};

template <class C>
__host__ __device__ inline GPipeGeom make_gpipe_geom() {
    GPipeGeom g{};
    g.tile_bytes = C::W * C::DT * static_cast<int>(sizeof(typename C::St));
    g.dec_off = C::NST * g.tile_bytes;
    g.bar_off = g.dec_off + C::NM * C::W * C::DT * 4;
    g.map_off = g.bar_off + (2 * C::NST + 3 * C::NM) * 8;
    g.entry_off = g.map_off + C::NM * C::DT * 8;
    g.flag_off = g.entry_off + C::NM * C::DT * 4;
    g.smem_bytes = g.flag_off + 16;
    return g;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
gpipe_fwd_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_out,
                 const float *__restrict__ eta, const float *__restrict__ nu_log, float *__restrict__ last, int T,
                 int D, DevStatus *status, uint64_t timeout_ns) {
    using St = typename C::St;
    constexpr int DT = C::DT, W = C::W, NS = C::NS, NR = C::NR, NST = C::NST, NM = C::NM;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const GPipeGeom geo = make_gpipe_geom<C>();
    auto tile = [&](int st) { return reinterpret_cast<St *>(smem_raw + st * geo.tile_bytes); };
    auto decays = [&](int m) { return reinterpret_cast<float *>(smem_raw + geo.dec_off) + m * W * DT; };
    auto bar = [&](int i) { return smem_addr(smem_raw + geo.bar_off + 8 * i); };
    auto full = [&](int st) { return bar(st); };
    auto stage_free = [&](int st) { return bar(NST + st); };
    auto map_full = [&](int m) { return bar(2 * NST + m); };
    auto entry_full = [&](int m) { return bar(2 * NST + NM + m); };
    auto slot_free = [&](int m) { return bar(2 * NST + 2 * NM + m); };
    float2 *wmap = reinterpret_cast<float2 *>(smem_raw + geo.map_off);
    float *went = reinterpret_cast<float *>(smem_raw + geo.entry_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + geo.flag_off);
    if (threadIdx.x == 0) {
        for (int st = 0; st < NST; ++st) {
            mbar_init(full(st), 1);
            mbar_init(stage_free(st), 1);
        }
        for (int m = 0; m < NM; ++m) {
            mbar_init(map_full(m), 1);
            mbar_init(entry_full(m), 1);
            mbar_init(slot_free(m), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, abort_flag, timeout_ns};
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int nwin = (T + W - 1) / W;
    auto warp_ok = [&](uint32_t b, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(b, par, wc, site));
    };
    // window k: stage k % NST (phase k / NST), slot k % NM (phase k / NM)
    auto spar = [&](int k) { return static_cast<uint32_t>((k / NST) & 1); };
    auto mpar = [&](int k) { return static_cast<uint32_t>((k / NM) & 1); };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane != 0) return;
        int issued = 0;
        for (int k = 0; k < nwin; ++k) {
            const int st = k % NST;
            if (k >= NST && !mbar_wait(stage_free(st), spar(k - NST), wc, kSiteProducerEmpty)) break;
            mbar_arrive_expect_tx(full(st), geo.tile_bytes);
            tma_load_3d(smem_addr(tile(st)), &tm_b, d0, k * W, brow, full(st));
            issued = k + 1;
        }
        // every copy landed before this thread leaves (a warp that aborted may
        // not have waited for its tile): the newest copy of each stage, bounded
        // and blind to the abort flag
        for (int k = (issued > NST ? issued - NST : 0); k < issued; ++k) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(full(k % NST), spar(k))) {
                if (global_timer_ns() - t0 > wc.timeout_ns) {
                    record_error(wc, kErrTimeout, kSiteDrain);
                    break;
                }
            }
        }
        return;
    }

    if (warp == 1) {
        // -------------------------------------------------------------- scan
        float carry = 0.0f;  // h_{-1} = 0
        for (int k = 0; k < nwin; ++k) {
            const int m = k % NM;
            if (!warp_ok(map_full(m), mpar(k), kSiteConsumerFull)) return;
            const float2 pq = wmap[m * DT + lane];
            went[m * DT + lane] = carry;
            carry = __fmaf_rn(pq.x, carry, pq.y);
            __syncwarp();
            if (lane == 0) mbar_arrive(entry_full(m));
        }
        return;
    }

    const int d = d0 + lane;
    const bool lane_ok = d < D;
    if (warp < 2 + NS) {
        // ------------------------------------------------------ summary warps
        const int sw = warp - 2;
        const float nnu2 = lane_ok ? -rate2(nu_log, d) : -0.0f;  // the decay exponent is (-nu2) E
        const float *eta_row = eta + static_cast<size_t>(brow) * T;
        float ev_next = eta_at(eta_row, sw * W + lane, T);  // eta of row `lane` of this warp's next window
        for (int k = sw; k < nwin; k += NS) {
            const float ev = ev_next;
            ev_next = eta_at(eta_row, (k + NS) * W + lane, T);
            const float e_mine = exp_approx(ev);  // E of row `lane` (lanes < W)
            const int st = k % NST, m = k % NM;
            const int nrows = min(T - k * W, W);
            float xa[W];
#pragma unroll
            for (int j = 0; j < W; ++j) {
                xa[j] = ex2_approx(__fmul_rn(nnu2, __shfl_sync(0xffffffffu, e_mine, j)));
                if (j >= nrows) xa[j] = 1.0f;  // steps past T: identity
            }
            // the slot is free once the replay of window k - NM has read it
            if (k >= NM && !warp_ok(slot_free(m), mpar(k - NM), kSiteProducerEmpty)) return;
            if (!warp_ok(full(st), spar(k), kSiteConsumerFull)) return;
            const St *tb = tile(st);
            float *dec = decays(m);
            float P = 1.0f, Q = 0.0f;
#pragma unroll
            for (int j = 0; j < W; ++j) {
                float x[1];
                unpack_lanes<St, 1>(tb + j * DT + lane, x);
                const float bj = j < nrows ? x[0] : 0.0f;
                P = __fmul_rn(xa[j], P);
                Q = __fmaf_rn(xa[j], Q, bj);
                dec[j * DT + lane] = xa[j];
            }
            wmap[m * DT + lane] = make_float2(P, Q);
            __syncwarp();
            if (lane == 0) mbar_arrive(map_full(m));
        }
        return;
    }

    // ------------------------------------------------------------ replay warps
    const int rw = warp - 2 - NS;
    int prev_st = -1, prev2_st = -1;  // stages of this warp's last two windows
    for (int k = rw; k < nwin; k += NR) {
        if (prev2_st >= 0) {
            if (lane == 0) {
                bulk_wait_read<1>();  // the out of the window before last left its stage
                mbar_arrive(stage_free(prev2_st));
            }
            __syncwarp();
        }
        prev2_st = prev_st;
        prev_st = -1;
        const int st = k % NST, m = k % NM;
        const int rbase = k * W;
        const int nrows = min(T - rbase, W);
        if (!warp_ok(entry_full(m), mpar(k), kSiteConsumerFull)) break;
        // the tile's phase completed before its summary (this window's map is
        // out); the wait orders its bytes before this warp's reads
        if (!warp_ok(full(st), spar(k), kSiteConsumerFull)) break;
        St *tb = tile(st);
        const float *dec = decays(m);
        float h = went[m * DT + lane];
        float xa[W], xb[W];
#pragma unroll
        for (int j = 0; j < W; ++j) {
            float x[1];
            unpack_lanes<St, 1>(tb + j * DT + lane, x);
            xb[j] = x[0];
            xa[j] = dec[j * DT + lane];
        }
        __syncwarp();  // every lane read the slot's decays and entering state
        if (lane == 0) mbar_arrive(slot_free(m));
#pragma unroll
        for (int j = 0; j < W; ++j) {
            if (j < nrows) {
                h = __fmaf_rn(xa[j], h, xb[j]);
                float hv[1] = {h};
                store_lanes<St, 1>(tb + j * DT + lane, hv);
            }
        }
        if (last != nullptr && lane_ok && rbase + nrows == T) last[static_cast<size_t>(brow) * D + d] = h;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&tm_out, smem_addr(tb), d0, rbase, brow);
            bulk_commit();
        }
        prev_st = st;
    }
    if (lane == 0) bulk_wait<0>();  // every out store landed before the CTA's shared memory goes away
}

}  // namespace lrscan
