// Single-pass scan over (lane tile, time window) CTAs with decoupled
// look-back.  For long sequences with few lanes, one CTA per lane tile
// walking all of T leaves most SMs idle, and the three-phase chunked path
// moves 5 / 7 elements per (t, d) instead of 3 / 5.  Here every CTA owns one
// window of W = S*L rows of DT = 32 lanes:
//
//   1. it takes a ticket (global atomic counter); tickets are time-major
//      (window k of every lane tile before window k+1), so a CTA only ever
//      waits on CTAs that took their ticket earlier and are already running;
//   2. it loads its window with one bulk tensor copy, summarizes its S
//      sub-chunks (as the windowed kernel does) and composes them into the
//      window's map h -> P*h + Q per lane, which it publishes (status A);
//   3. its lane threads (warp 0) look back over the earlier windows of the
//      same lane tile: a window with an inclusive state (status P) ends the
//      walk, a window with only its map is composed in and the walk goes on
//      (triton_training_scan.py's chunk prefix, with the decoupled look-back
//      of single-pass GPU scans instead of a separate pass);
//   4. it publishes its inclusive state (status P), walks its sub-chunk maps
//      from the entry state and replays.
//
// Every wait is bounded: a flag that does not appear in time records
// LRSCAN_ETIMEOUT and the CTA finishes without waiting further.  Each
// window's data is read from HBM once: 3 elements per (t, d) forward.
//
// Workspace: flags [nwin][nlt] u32 (zeroed before every launch together with
// the ticket), maps [nwin][D] float2, inclusive states [nwin][D] float.
#pragma once

#include "window_kernels.cuh"

namespace lrscan {

struct LookbackArgs {
    unsigned int *ticket;    // one counter per launch (zeroed before it)
    unsigned int *flags;     // [nwin][nlt]: 0 none, 1 map published, 2 inclusive published
    float2 *maps;            // [nwin][B*D] window maps (P, Q)
    float *incl;             // [nwin][B*D] state after the window
    int nlt;                 // lane tiles per batch row times batch rows (tiles per window index)
};

constexpr unsigned kLbMap = 1, kLbIncl = 2;

// Flag accesses: release store after the window's data, acquire load before
// reading them (GPU scope).
__device__ __forceinline__ unsigned ld_flag_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_flag_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Warp 0 publishes its lanes' data: every lane's stores, a fence, the warp
// barrier, then lane 0 fences again (cumulative) and releases the flag.
__device__ __forceinline__ void publish(unsigned *flag, unsigned value) {
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        __threadfence();
        st_flag_release(flag, value);
    }
}

// Forward.  Shape: windowed lane-scan tile with DT = 32 lanes (warp 0 are
// the lane threads), NIN = 2 (a, b).
template <class C>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
lb_fwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              typename C::St *__restrict__ out, float *__restrict__ last, const __grid_constant__ WinGeom geom,
              const __grid_constant__ LookbackArgs lb, int lanes_per_row, DevStatus *status, uint64_t timeout_ns) {
    static_assert(!C::SEQ && !C::PT && C::NIN == 2 && C::DT == 32, "look-back forward: lane-scan tile of 32 lanes");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ unsigned s_ticket;
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    win_init<C>(sm, NT / 32, S);
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) s_ticket = atomicAdd(lb.ticket, 1u);
    __syncthreads();
    const unsigned id = s_ticket;
    const int tile = static_cast<int>(id % static_cast<unsigned>(lb.nlt));  // (batch row, lane tile)
    const int k = static_cast<int>(id / static_cast<unsigned>(lb.nlt));      // time window
    const int brow = tile / lanes_per_row;
    const int d0 = (tile - brow * lanes_per_row) * DT;
    const int T = geom.T, D = geom.D;
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const tms[2] = {&tm_a, &tm_b};
            for (int i = 0; i < 2; ++i) prefetch_tensormap(tms[i]);
            const uint32_t fb = sm.full_bar(0);
            mbar_arrive_expect_tx(fb, sm.stage_bytes);
            for (int i = 0; i < 2; ++i)
                tma_load_3d(smem_addr(sm.tile<C>(0, i)), tms[i], d0, k * sm.W, brow, fb);
            // the copy always lands before the CTA may exit (bounded wait)
            const uint64_t start = global_timer_ns();
            while (!mbar_try_wait(fb, 0)) {
                if (global_timer_ns() - start > timeout_ns) {
                    record_error(wc, kErrTimeout, kSiteDrain);
                    break;
                }
            }
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int lane = threadIdx.x & 31;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const int rbase = k * sm.W + s * L;
    const int n = min(max(T - rbase, 0), L);
    const bool ok = mbar_wait(sm.full_bar(0), 0, wc, kSiteConsumerFull);
    float xa[L][V], xb[L][V];
    {
        const St *ta = sm.tile<C>(0, 0) + (s * L) * DT + lg * V;
        const St *tb = sm.tile<C>(0, 1) + (s * L) * DT + lg * V;
        if (ok) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
                unpack_lanes<St, V>(ta + j * DT, xa[j]);
                unpack_lanes<St, V>(tb + j * DT, xb[j]);
            }
        }
    }
    float P[V], Q[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
    if (n < L) {
#pragma unroll
        for (int j = 0; j < L; ++j) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                xa[j][v] = j < n ? xa[j][v] : 1.0f;
                xb[j][v] = j < n ? xb[j][v] : 0.0f;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < L; ++j) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            P[v] = __fmul_rn(xa[j][v], P[v]);
            Q[v] = __fmaf_rn(xa[j][v], Q[v], xb[j][v]);
        }
    }
    float2 *pq = sm.sPQ<C>(0);
#pragma unroll
    for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
    bool failed = bar_sync_or(1, NT, !ok);

    // warp 0: window map, publish, look back, publish the inclusive state,
    // then the sub-chunk entry states
    float *entry = sm.sEntry<C>();
    if (threadIdx.x < DT && !failed) {
        const int i_lane = threadIdx.x;  // lane index v*G + g of the scan arrays
        const int ch = lane_channel<C>(d0, i_lane);
        const size_t gl = static_cast<size_t>(brow) * D + ch;  // global lane
        const size_t nl = static_cast<size_t>(lb.nlt / lanes_per_row) * D;  // B*D lanes
        // window map: composition of the S sub-chunk maps in order (identity
        // maps leave it unchanged)
        float wp = 1.0f, wq = 0.0f;
        for (int i = 0; i < S; ++i) {
            const float2 m = pq[i * DT + i_lane];
            wq = __fmaf_rn(m.x, wq, m.y);
            wp = __fmul_rn(m.x, wp);
        }
        float c = 0.0f;  // state entering this window
        unsigned *myflag = lb.flags + static_cast<size_t>(k) * lb.nlt + tile;
        if (k == 0) {
            // the first window's entry is h_{-1} = 0: publish the inclusive state at once
            if (ch < D) lb.incl[gl] = wq;
            publish(myflag, kLbIncl);
        } else {
            if (ch < D) lb.maps[static_cast<size_t>(k) * nl + gl] = make_float2(wp, wq);
            publish(myflag, kLbMap);
            // look back: acc = (maps of windows j+1 .. k-1 composed)
            float ap = 1.0f, aq = 0.0f;
            bool timed_out = false;
            for (int j = k - 1; j >= 0; --j) {
                const unsigned *fp = lb.flags + static_cast<size_t>(j) * lb.nlt + tile;
                unsigned f = 0;
                if (lane == 0) {
                    const uint64_t start = global_timer_ns();
                    while ((f = ld_flag_acquire(fp)) == 0u) {
                        if (global_timer_ns() - start > timeout_ns) {
                            record_error(wc, kErrTimeout, kSiteConsumerFull);
                            break;
                        }
                    }
                }
                f = __shfl_sync(0xffffffffu, f, 0);
                if (f == 0u) { timed_out = true; break; }
                __threadfence();  // lane 0 acquired the flag; its data are visible to the warp
                if (f == kLbIncl) {
                    const float h = ch < D ? __ldcg(lb.incl + static_cast<size_t>(j) * nl + gl) : 0.0f;
                    c = __fmaf_rn(ap, h, aq);
                    break;
                }
                const float2 m = ch < D ? __ldcg(lb.maps + static_cast<size_t>(j) * nl + gl) : make_float2(1.0f, 0.0f);
                // acc <- acc o m_j  (m_j applies first)
                aq = __fmaf_rn(ap, m.y, aq);
                ap = __fmul_rn(ap, m.x);
            }
            if (!timed_out) {
                if (ch < D) lb.incl[static_cast<size_t>(k) * nl + gl] = __fmaf_rn(wp, c, wq);
                publish(myflag, kLbIncl);
            } else {
                *sm.abort_flag() = 1;
            }
        }
        // sub-chunk entry states from the window's entry state
        for (int i = 0; i < S; ++i) {
            const float2 m = pq[i * DT + i_lane];
            entry[i * DT + i_lane] = c;
            c = __fmaf_rn(m.x, c, m.y);
        }
    }
    failed = bar_sync_or(1, NT, failed || *sm.abort_flag() != 0);
    if (failed) return;
    float h[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h[v] = entry[s * DT + v * G + lg];
    St *op = out + (row0 + rbase) * D + d;
#pragma unroll
    for (int j = 0; j < L; ++j) {
#pragma unroll
        for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
        if (lane_ok && (n == L || j < n)) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
    }
    if (last != nullptr && lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
        for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
    }
}

}  // namespace lrscan
