// Persistent single-pass scan over time chunks, for few lanes and long
// sequences (the chunked decomposition of triton_training_scan.py,
// _real_chunk_summary / _real_chunk_prefix / _real_chunk_replay, with the
// prefix taken by look-back inside the one kernel instead of a phase of its
// own).
//
// Every lane group (batch row x lane tile of DT lanes) is cut in time into
// chunks of NWC windows of W = S * L rows.  A fixed grid of CTAs takes chunks
// from a ticket counter, chunk-major over the groups (forward: earliest chunk
// first; backward: latest first), and passes over each chunk twice:
//   summary  the window tiles stream in through the bulk-copy ring (from HBM);
//            the sub-chunk maps of each window are composed by the lane
//            threads into the chunk's map h -> P h + Q, which is published;
//   prefix   the lane threads look back over the chunks before it: the
//            nearest one whose leaving state is published, composed with the
//            maps of the chunks in between, gives the entering state; the
//            chunk's own leaving state P h_in + Q is published in turn;
//   replay   the same tiles stream in again, now from L2 (the chunks in
//            flight on the whole GPU take a few tens of MB), and the windowed
//            kernel's maps, lane walk and replay write the outputs through
//            the staged bulk tensor stores.
// So HBM carries the scan's own traffic (forward a, b in and out; backward
// a, out, grad_out in and grad_a, grad_b out), one pass.
//
// Publication: one flag word per chunk (0 before the call, kChunkAgg once the
// map is out, kChunkIncl once the leaving state is out), stored with release
// semantics after a fence by every writer; readers acquire.  The look-back
// waits only on chunks with earlier tickets, which CTAs that are running hold,
// so it always ends; still every wait is bounded (timeout: LRSCAN_ETIMEOUT in
// the status word, and the kernel returns).
#pragma once

#include "window_kernels.cuh"

namespace lrscan {

constexpr uint32_t kChunkAgg = 1, kChunkIncl = 2;

enum StreamSite : int { kSiteLookback = 8 };


__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Entering state of chunk `cc` (ticket order within group row `g0` of the
// workspace) for lane thread i; one warp of lane threads calls it together.
// Lane l of the warp inspects chunk base - l: the nearest chunk with a
// published leaving state bounds the walk, and every chunk before it (in
// ticket order) must have its map out.  Maps are composed outermost first:
// h_in = M_base o M_base-1 o ... (h_incl).  Chunk -1 leaves the zero state.
// Returns false when the wait expired or the CTA is aborting.
template <int DT>
__device__ bool stream_lookback(const StreamArgs &sa, size_t g0, int cc, int i, float &h_in, const WaitCtx &wc) {
    const int lane = threadIdx.x & 31;
    float aP = 1.0f, aQ = 0.0f;
    int base = cc - 1;
    uint64_t start = 0;
    bool timed = false;
    for (;;) {
        if (base < 0) {
            h_in = aQ;  // aP * 0 + aQ
            return true;
        }
        const int ci = base - lane;
        int tstar = 32;
        for (uint32_t spin = 0;; ++spin) {
            const uint32_t f = ci >= 0 ? ld_acquire_gpu(sa.flag + g0 + ci) : kChunkIncl;
            const uint32_t ready = __ballot_sync(0xffffffffu, f != 0u);
            const uint32_t inclm = __ballot_sync(0xffffffffu, f == kChunkIncl);
            tstar = inclm ? __ffs(inclm) - 1 : 32;
            const uint32_t need = tstar >= 31 ? 0xffffffffu : ((2u << tstar) - 1u);
            if ((ready & need) == need) break;
            if ((spin & 31u) == 31u) {
                bool stop = *wc.abort_flag != 0;
                if (!timed) {
                    start = global_timer_ns();
                    timed = true;
                } else if (global_timer_ns() - start > wc.timeout_ns) {
                    stop = true;
                    if (lane == 0) record_error(wc, kErrTimeout, kSiteLookback);
                }
                if (__any_sync(0xffffffffu, stop)) return false;
            }
        }
        // the maps and states read below were published before flags that
        // other lanes of this warp acquired
        __threadfence();
        const int nagg = tstar < 32 ? tstar : 32;
#pragma unroll 4
        for (int t = 0; t < nagg; ++t) {
            const float2 m = __ldcg(sa.agg + (g0 + base - t) * DT + i);
            aQ = __fmaf_rn(aP, m.y, aQ);
            aP = __fmul_rn(aP, m.x);
        }
        if (tstar < 32) {
            const int cb = base - tstar;
            const float hb = cb >= 0 ? __ldcg(sa.incl + (g0 + cb) * DT + i) : 0.0f;
            h_in = __fmaf_rn(aP, hb, aQ);
            return true;
        }
        base -= 32;
    }
}

// Named barrier over the lane threads (threads 0 .. DT-1, whole warps); the
// second form also ANDs a predicate over them.
template <int DT> __device__ __forceinline__ void lane_bar() {
    asm volatile("bar.sync 2, %0;" ::"n"(DT) : "memory");
}
template <int DT> __device__ __forceinline__ bool lane_bar_and(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 2, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(flag ? 1u : 0u), "n"(DT)
        : "memory");
    return r != 0;
}

// One kernel for both directions.  Forward tiles: a, b (row t); outputs out.
// Backward tiles: a one row late (a_{t+1}), out one row early (h_{t-1}),
// grad_out; outputs grad_a, grad_b.  tm_3 / tm_4: the output maps.
template <class C, bool BWD>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
stream_kernel(const __grid_constant__ CUtensorMap tm_0, const __grid_constant__ CUtensorMap tm_1,
              const __grid_constant__ CUtensorMap tm_2, const __grid_constant__ CUtensorMap tm_3,
              const __grid_constant__ CUtensorMap tm_4, float *__restrict__ last,
              const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns,
              const __grid_constant__ StreamArgs sa) {
    static_assert(!C::SEQ && !C::PT && !C::EX, "stream tile: lane-scan windowed shape");
    static_assert(C::NIN == (BWD ? 3 : 2), "forward tiles a, b; backward a, out, grad_out");
    static_assert(C::DT % 32 == 0, "lane threads in whole warps");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    constexpr int NP = BWD ? 2 : 1;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    const int W = sm.W;
    // chunk ticket of each stage's current fill (-1: no more chunks)
    int *meta = reinterpret_cast<int *>(smem_raw + win_out_smem(geom, NP, 2));
    win_init<C>(sm, NT / 32, S);
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int T = geom.T, D = geom.D;
    const int nwc = sa.nwc;
    const int CH = nwc * W;
    const long long total = static_cast<long long>(sa.ng) * sa.nc;

    if (static_cast<int>(threadIdx.x) >= NT) {  // producer warp
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[3] = {&tm_0, &tm_1, &tm_2};
#pragma unroll
            for (int i = 0; i < C::NIN; ++i) prefetch_tensormap(maps[i]);
            int stage = 0, use = 0;
            long long fills = 0;
            bool stop = false;
            while (!stop) {
                const long long j = static_cast<long long>(atomicAdd(sa.ticket, 1u));
                const bool done = j >= total;
                int c = 0, brow = 0, x0 = 0;
                if (!done) {
                    const int cc = static_cast<int>(j / sa.ng);
                    const int gi = static_cast<int>(j - static_cast<long long>(cc) * sa.ng);
                    c = BWD ? sa.nc - 1 - cc : cc;
                    brow = gi / sa.ndt;
                    x0 = (gi - brow * sa.ndt) * DT;
                }
                const int nfill = done ? 1 : 2 * nwc;
                for (int q = 0; q < nfill; ++q) {
                    if (use > 0 && !mbar_wait(sm.empty_bar(stage), (use - 1) & 1, wc, kSiteProducerEmpty)) {
                        stop = true;
                        break;
                    }
                    meta[stage] = done ? -1 : static_cast<int>(j);
                    const uint32_t fb = sm.full_bar(stage);
                    if (done) {
                        mbar_arrive(fb);
                    } else {
                        const int qw = q % nwc;
                        const int w = BWD ? nwc - 1 - qw : qw;
                        const int y = c * CH + w * W;
                        mbar_arrive_expect_tx(fb, sm.stage_bytes);
#pragma unroll
                        for (int i = 0; i < C::NIN; ++i) {
                            const int dy = BWD ? (i == 0 ? 1 : (i == 1 ? -1 : 0)) : 0;
                            tma_load_3d(smem_addr(sm.tile<C>(stage, i)), maps[i], x0, y + dy, brow, fb);
                        }
                    }
                    ++fills;
                    if (++stage == sm.nstage) { stage = 0; ++use; }
                }
                if (done) stop = true;
            }
            // every copy issued has landed before the CTA can exit
            const long long first = fills > sm.nstage ? fills - sm.nstage : 0;
            for (long long k = first; k < fills; ++k) {
                const uint32_t fb = sm.full_bar(static_cast<int>(k % sm.nstage));
                const uint32_t par = static_cast<uint32_t>((k / sm.nstage) & 1);
                if (mbar_try_wait(fb, par)) continue;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(fb, par)) {
                    if (global_timer_ns() - t0 > wc.timeout_ns) {
                        record_error(wc, kErrTimeout, kSiteDrain);
                        break;
                    }
                }
            }
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const bool lt = static_cast<int>(threadIdx.x) < DT;  // lane thread: owns entry i = threadIdx.x of the maps
    const bool issuer = static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    const OutStage<NP, St> ost = make_out_stage<NP, St>(smem_raw, geom);
    const CUtensorMap *omaps[NP];
    if constexpr (BWD) {
        omaps[0] = &tm_3;
        omaps[1] = &tm_4;
    } else {
        omaps[0] = &tm_3;
    }
    float2 *pq = sm.sPQ<C>(0);
    float *entry = sm.sEntry<C>();
    int stage = 0, use = 0;
    int rw = 0;              // replay windows staged so far (output buffer parity)
    bool pending = false;    // the last staged window's tile still has to be stored
    int px = 0, py = 0, pz = 0, pw = 0;
    bool failed = false;

    for (;;) {
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if (bar_sync_or(1, NT, !ok)) { failed = true; break; }
        const int j = meta[stage];
        if (j < 0) break;  // no more chunks (every consumer thread reads the same word)
        const int cc = j / sa.ng;
        const int gi = j - cc * sa.ng;
        const int c = BWD ? sa.nc - 1 - cc : cc;
        const int brow = gi / sa.ndt;
        const int x0 = (gi - brow * sa.ndt) * DT;
        const size_t g0 = static_cast<size_t>(gi) * sa.nc;
        const int d = x0 + lg * V;
        const bool lane_ok = d < D;

        // ------------------------------------------------------------ summary
        float Pc = 1.0f, Qc = 0.0f;  // lane threads: the chunk's map so far
        for (int q = 0; q < nwc; ++q) {
            if (q > 0) ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
            const int w = BWD ? nwc - 1 - q : q;
            const int rbase = c * CH + w * W + s * L;
            const int n = min(max(T - rbase, 0), L);
            float xa[L][V], xb[L][V];  // forward a_t, b_t; backward a_{t+1}, grad_out_t
            if (ok) {
                const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;
                const St *tb = sm.tile<C>(stage, C::NIN - 1) + (s * L) * DT + lg * V;
#pragma unroll
                for (int r = 0; r < L; ++r) {
                    unpack_lanes<St, V>(ta + r * DT, xa[r]);
                    unpack_lanes<St, V>(tb + r * DT, xb[r]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
            if (++stage == sm.nstage) { stage = 0; ++use; }
            if (n < L) {
                // steps past T are identity steps (a = 1, addend 0)
#pragma unroll
                for (int r = 0; r < L; ++r) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        xa[r][v] = r < n ? xa[r][v] : 1.0f;
                        xb[r][v] = r < n ? xb[r][v] : 0.0f;
                    }
                }
            }
            float P[V], Q[V];
#pragma unroll
            for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
            for (int rr = 0; rr < L; ++rr) {
                const int r = BWD ? L - 1 - rr : rr;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    P[v] = __fmul_rn(xa[r][v], P[v]);
                    Q[v] = __fmaf_rn(xa[r][v], Q[v], xb[r][v]);
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
            if (bar_sync_or(1, NT, !ok)) { failed = true; break; }
            if (issuer && pending) {
                // the previous chunk's last window; once issued, the store
                // before it must have finished reading the other buffer
                ost.store(omaps, pw, px, py, pz);
                bulk_wait_read<1>();
                pending = false;
            }
            if (lt) {
                // compose the window's sub-chunk maps into the chunk's, in
                // chain order (backward: last sub-chunk first)
                for (int i = 0; i < S; ++i) {
                    const int sc = BWD ? S - 1 - i : i;
                    const float2 m = pq[sc * DT + threadIdx.x];
                    Qc = __fmaf_rn(m.x, Qc, m.y);
                    Pc = __fmul_rn(m.x, Pc);
                }
            }
            bar_sync_or(1, NT, false);  // pq is free again
        }
        if (failed) break;

        // ------------------------------------------------------------- prefix
        float carry = 0.0f;
        bool lb_ok = true;
        if (lt) {
            const size_t slot = g0 + cc;
            sa.agg[slot * DT + threadIdx.x] = make_float2(Pc, Qc);
            __threadfence();
            lane_bar<DT>();
            if (threadIdx.x == 0) st_release_gpu(sa.flag + slot, kChunkAgg);
            lb_ok = stream_lookback<DT>(sa, g0, cc, threadIdx.x, carry, wc);
            sa.incl[slot * DT + threadIdx.x] = __fmaf_rn(Pc, carry, Qc);
            __threadfence();
            lb_ok = lane_bar_and<DT>(lb_ok);
            if (threadIdx.x == 0 && lb_ok) st_release_gpu(sa.flag + slot, kChunkIncl);
        }

        // ------------------------------------------------------------- replay
        for (int q = 0; q < nwc; ++q) {
            ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
            const int w = BWD ? nwc - 1 - q : q;
            const int wbase = c * CH + w * W;
            const int rbase = wbase + s * L;
            const int n = min(max(T - rbase, 0), L);
            float xa[L][V], xb[L][V], xh[BWD ? L : 1][V];
            if (ok) {
                const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;
                const St *tb = sm.tile<C>(stage, C::NIN - 1) + (s * L) * DT + lg * V;
#pragma unroll
                for (int r = 0; r < L; ++r) {
                    unpack_lanes<St, V>(ta + r * DT, xa[r]);
                    unpack_lanes<St, V>(tb + r * DT, xb[r]);
                }
                if constexpr (BWD) {
                    const St *th = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;
#pragma unroll
                    for (int r = 0; r < L; ++r) unpack_lanes<St, V>(th + r * DT, xh[r]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
            if (++stage == sm.nstage) { stage = 0; ++use; }
            if (n < L) {
#pragma unroll
                for (int r = 0; r < L; ++r) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        xa[r][v] = r < n ? xa[r][v] : 1.0f;
                        xb[r][v] = r < n ? xb[r][v] : 0.0f;
                    }
                }
            }
            float P[V], Q[V];
#pragma unroll
            for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
            for (int rr = 0; rr < L; ++rr) {
                const int r = BWD ? L - 1 - rr : rr;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    P[v] = __fmul_rn(xa[r][v], P[v]);
                    Q[v] = __fmaf_rn(xa[r][v], Q[v], xb[r][v]);
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
            if (bar_sync_or(1, NT, !ok || !lb_ok)) { failed = true; break; }
            if (issuer && pending) {
                ost.store(omaps, pw, px, py, pz);
                bulk_wait_read<1>();
                pending = false;
            }
            // lane threads push the chunk's entering state through the
            // window's sub-chunk maps (backward: last sub-chunk first)
            if (lt) carry = lane_walk<BWD, DT>(pq, entry, S, threadIdx.x, carry);
            bar_sync_or(1, NT, false);
            float h[V];
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = entry[s * DT + v * G + lg];
            if constexpr (BWD) {
                St *sga = ost.plane(rw, 0) + (s * L) * DT + lg * V;
                St *sgb = ost.plane(rw, 1) + (s * L) * DT + lg * V;
                bwd_rows<C, false, true>(xa, xh, xb, h, n, lane_ok, sgb, sga, D, 0u);
            } else {
                St *op = ost.plane(rw, 0) + (s * L) * DT + lg * V;
#pragma unroll
                for (int r = 0; r < L; ++r) {
#pragma unroll
                    for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[r][v], h[v], xb[r][v]);
                    store_lanes<St, V>(op + r * DT, h);
                }
                // the thread whose sub-chunk holds step T-1 owns the final state
                if (last != nullptr && lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
                    for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
                }
            }
            fence_proxy_async_smem();
            // windows wholly past T have nothing to store
            pending = wbase < T;
            pw = rw;
            px = x0;
            py = wbase;
            pz = brow;
            ++rw;
        }
        if (failed) break;
    }
    // the last staged tile (not after an abort), then every store complete
    // before the CTA's shared memory goes away
    const bool aborted = bar_sync_or(1, NT, failed);
    if (issuer) {
        if (!aborted && pending) ost.store(omaps, pw, px, py, pz);
        bulk_wait<0>();
    }
}

}  // namespace lrscan
