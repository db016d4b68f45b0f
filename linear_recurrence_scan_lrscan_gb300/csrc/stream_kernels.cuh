// Persistent single-pass scan over time chunks, for few lanes and long
// sequences (the chunked decomposition of triton_training_scan.py,
// _real_chunk_summary / _real_chunk_prefix / _real_chunk_replay, with the
// prefix taken by look-back inside the one kernel instead of a phase of its
// own).
//
// Every lane group (batch row x lane tile of DT lanes) is cut in time into
// chunks of NWC windows of W rows.  A fixed grid of CTAs takes chunks from a
// ticket counter, chunk-major over the groups (forward: earliest chunk first;
// backward: latest first).  A CTA has NWC window warps (warp w owns window w
// of every chunk, all DT lanes, V lanes per thread), two scan warps (chunks
// alternate between them) and a ticket warp, and passes over each chunk
// twice:
//   summary  each window warp copies its window's tiles in (bulk tensor
//            copies, from HBM) and reduces them to the affine map
//            h -> P h + Q of its rows, one lane per thread;
//   prefix   the last window warp to finish composes the window maps into
//            the chunk's map and publishes it; a scan warp looks back over
//            the chunks before it (the nearest one whose leaving state is
//            published, composed with the maps of the chunks in between,
//            gives the entering state), publishes the chunk's leaving state,
//            and hands every window warp the state entering its window;
//   replay   each window warp copies the same tiles in again, now from L2,
//            runs its rows with the sequential step from its entering state
//            and stores every output row straight to global memory (a warp
//            writes whole rows of its DT lanes).
// The replay of chunk k follows the summaries of chunks k+1 and k+2, and two
// scan warps look back for consecutive chunks at once, so the look-back's
// latency (a few L2 round trips) hides behind two chunks of work; the three
// chunks between a summary and its replay are what L2 holds.  Each window
// warp owns two ring stages (summary and replay tiles), so one tile loads
// while it works on the other.
// HBM carries the scan's own traffic: forward a, b in, out out; backward a,
// out, grad_out in, grad_a, grad_b out.  Results agree with the sequential
// definition to rounding; which published states a look-back composes depends
// on timing, so two calls can differ in the last bits.
//
// Publication: one flag word per chunk (0 before the call, kChunkAgg once the
// map is out, kChunkIncl once the leaving state is out): the warp's lanes
// write their lanes' values, a warp barrier, then lane 0 stores the flag with
// release semantics; readers acquire the flags, pass a warp barrier, and read
// the values past L1.  The look-back waits only on chunks with earlier
// tickets, which running CTAs hold, so it always ends; still every wait is
// bounded (timeout: LRSCAN_ETIMEOUT in the status word, and the kernel
// returns).
#pragma once

#include "scan_common.cuh"
#include "stream_args.h"

namespace lrscan {

constexpr uint32_t kChunkAgg = 1, kChunkIncl = 2;

enum StreamSite : int { kSiteLookback = 8, kSiteStreamStep = 9 };

// Chunks a replay trails its summary by, scan warps, and map / entering-state
// buffers (one per chunk between a summary and its replay, plus one).
constexpr int kStreamLag = 2, kStreamScanWarps = 2, kStreamBufs = kStreamLag + 1;

// Compiled shape: storage type, lanes per CTA, lanes per thread, rows per
// window (per window warp), windows per chunk, CTAs per SM the registers must
// allow.  One warp spans the DT lanes of a window row.
template <class St_, int DT_, int V_, int W_, int NWC_, int MINB_>
struct StreamShape {
    using St = St_;
    static constexpr int DT = DT_, V = V_, W = W_, NWC = NWC_, MINB = MINB_;
    static constexpr int THREADS = (NWC + kStreamScanWarps + 1) * 32;
    static_assert(DT == 32 * V, "one warp spans a tile row");
    static_assert(W % 8 == 0, "rows are taken eight at a time");
};

// Steps a CTA keeps tickets for (ring of step slots).
constexpr int kStreamStepSlots = 8;

// Shared-memory layout (bytes from the 1024-aligned base), host and device.
struct StreamGeom {
    int nstage;      // ring stages (window tiles): 2 * NWC, two per window warp
    int tile_bytes;  // one plane of one window: W * DT * elem
    int stage_bytes; // NIN planes
    int bar_off;     // full[nstage], step_free[nstage], step_full[slots], maps_ready[bufs], entries_ready[bufs]
    int ticket_off;  // step tickets [slots]
    int map_off;     // window maps [bufs][NWC][DT] float2
    int entry_off;   // window entering states [bufs][NWC][DT] float
    int cmap_off;    // chunk maps [bufs][DT] float2, composed by the last window warp
    int count_off;   // window warps done with a chunk's summary [bufs]
    int flag_off;    // abort flag
    int smem_bytes;
};

template <class C, int NIN>
__host__ __device__ inline StreamGeom make_stream_geom(int nstage) {
    StreamGeom g{};
    g.nstage = nstage;
    g.tile_bytes = C::W * C::DT * static_cast<int>(sizeof(typename C::St));
    g.stage_bytes = NIN * g.tile_bytes;
    g.bar_off = nstage * g.stage_bytes;
    const int nbar = 2 * nstage + kStreamStepSlots + 2 * kStreamBufs;
    g.ticket_off = g.bar_off + nbar * 8;
    g.map_off = (g.ticket_off + kStreamStepSlots * 4 + 15) / 16 * 16;
    g.entry_off = g.map_off + kStreamBufs * C::NWC * C::DT * 8;
    g.cmap_off = g.entry_off + kStreamBufs * C::NWC * C::DT * 4;
    g.count_off = g.cmap_off + kStreamBufs * C::DT * 8;
    g.flag_off = g.count_off + kStreamBufs * 4;
    g.smem_bytes = g.flag_off + 16;
    return g;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int atom_add_acq_rel_cta(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v)
                 : "memory");
    return old;
}

// Entering state of chunk `cc` (ticket order within group gi) for lanes
// i0 .. i0+V-1, from the chunk maps and leaving states other CTAs published;
// the whole warp calls it.  Lane l of the warp inspects chunk base - l: the
// nearest chunk whose leaving state is out bounds the walk, and every chunk
// between (in ticket order) must have its map out.  Maps are composed
// outermost first: h_in = M_base o M_base-1 o ... (h_state); chunk -1 leaves
// the zero state.  Returns false when the wait expired or the CTA is aborting.
template <int DT, int V, int BATCH>
__device__ bool stream_lookback(const StreamArgs &sa, int gi, int cc, int i0, float (&h_in)[V], const WaitCtx &wc) {
    static_assert(32 % BATCH == 0, "whole batches per round");
    const int lane = threadIdx.x & 31;
    const size_t g0 = static_cast<size_t>(gi) * sa.nc;
    float aP[V], aQ[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { aP[v] = 1.0f; aQ[v] = 0.0f; }
    int base = cc - 1;
    uint64_t start = 0;
    bool timed = false;
    for (;;) {
        if (base < 0) {
#pragma unroll
            for (int v = 0; v < V; ++v) h_in[v] = aQ[v];  // aP * 0 + aQ
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
        // other lanes of this warp acquired: the warp barrier orders those
        // acquires before every lane's reads (loads bypass L1)
        __syncwarp();
        const int nagg = tstar < 32 ? tstar : 32;
        // the maps of up to 32 chunks: every load of a batch issued before
        // any is used (one L2 round trip per batch), then folded in order
#pragma unroll
        for (int t0 = 0; t0 < 32; t0 += BATCH) {
            if (t0 >= nagg) break;
            float2 m[BATCH][V];
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                if (t0 + t < nagg) {
                    const float2 *row = sa.agg + (g0 + base - t0 - t) * DT + i0;
#pragma unroll
                    for (int v = 0; v < V; ++v) m[t][v] = __ldcg(row + v);
                }
            }
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                if (t0 + t < nagg) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        aQ[v] = __fmaf_rn(aP[v], m[t][v].y, aQ[v]);
                        aP[v] = __fmul_rn(aP[v], m[t][v].x);
                    }
                }
            }
        }
        if (tstar < 32) {
            const int cb = base - tstar;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float hb = cb >= 0 ? __ldcg(sa.incl + (g0 + cb) * DT + i0 + v) : 0.0f;
                h_in[v] = __fmaf_rn(aP[v], hb, aQ[v]);
            }
            return true;
        }
        base -= 32;
    }
}

// Bounded wait on an mbarrier by a whole warp, the outcome agreed.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx &wc, int site) {
    const bool ok = mbar_wait(bar, parity, wc, site);
    return __all_sync(0xffffffffu, ok);
}

// Rows r0 .. r0+7 of one window tile to registers: lanes lane*V ...
template <class St, int V, int DT>
__device__ __forceinline__ void load8(const St *tile, int r0, int lane, float (&x)[8][V]) {
#pragma unroll
    for (int r = 0; r < 8; ++r) unpack_lanes<St, V>(tile + (r0 + r) * DT + lane * V, x[r]);
}

// One kernel for both directions.  Forward tiles: a, b (row t); output out.
// Backward tiles: a one row late (a_{t+1}), out one row early (h_{t-1}),
// grad_out; outputs grad_a (out0), grad_b (out1).  Outputs are written
// directly to global memory.
//
// Steps: step k takes ticket k (-1 once the chunks are gone) and runs the
// summary of ticket k, then the replay of ticket k - kStreamLag.  Window warp w
// keeps its summary tiles in stage w and its replay tiles in stage NWC + w and
// issues their bulk copies itself, each as soon as the stage's previous tile
// is done (the next summary's before this step's replay, the next replay's
// after it).  A ticket warp fetches ticket k once the window warps have
// finished step k - 3 and publishes it in a ring of step slots.
template <class C, bool BWD>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
stream_kernel(const __grid_constant__ CUtensorMap tm_0, const __grid_constant__ CUtensorMap tm_1,
              const __grid_constant__ CUtensorMap tm_2, typename C::St *__restrict__ out0,
              typename C::St *__restrict__ out1, float *__restrict__ last, int T, int D, int nstage,
              DevStatus *status, uint64_t timeout_ns, const __grid_constant__ StreamArgs sa) {
    using St = typename C::St;
    constexpr int DT = C::DT, V = C::V, W = C::W, NWC = C::NWC;
    constexpr int NIN = BWD ? 3 : 2;
    constexpr int LAG = kStreamLag, NB = kStreamBufs, SLOTS = kStreamStepSlots;
    constexpr int AHEAD = 3;  // the ticket warp fetches ticket k after the window warps finish step k - AHEAD
    static_assert(SLOTS % kStreamScanWarps == 0, "a scan warp sees every use of its step slots");
    static_assert(SLOTS >= AHEAD + 2 * LAG + 1, "a step slot is rewritten only after every reader is done");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const StreamGeom geo = make_stream_geom<C, NIN>(nstage);
    auto tile = [&](int stage, int plane) {
        return reinterpret_cast<St *>(smem_raw + stage * geo.stage_bytes + plane * geo.tile_bytes);
    };
    auto bar = [&](int i) { return smem_addr(smem_raw + geo.bar_off + 8 * i); };
    auto full_bar = [&](int s) { return bar(s); };
    auto free_bar = [&](int q) { return bar(nstage + q); };  // window warps done with step slot q's step
    auto step_bar = [&](int q) { return bar(2 * nstage + q); };
    auto maps_bar = [&](int b) { return bar(2 * nstage + SLOTS + b); };
    auto entries_bar = [&](int b) { return bar(2 * nstage + SLOTS + NB + b); };
    int *step_ticket = reinterpret_cast<int *>(smem_raw + geo.ticket_off);
    float2 *wmap = reinterpret_cast<float2 *>(smem_raw + geo.map_off);    // [NB][NWC][DT]
    float *wentry = reinterpret_cast<float *>(smem_raw + geo.entry_off);  // [NB][NWC][DT]
    float2 *cmap = reinterpret_cast<float2 *>(smem_raw + geo.cmap_off);   // [NB][DT]
    unsigned int *wcount = reinterpret_cast<unsigned int *>(smem_raw + geo.count_off);  // [NB]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + geo.flag_off);
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstage; ++s) mbar_init(full_bar(s), 1);
        for (int q = 0; q < SLOTS; ++q) {
            mbar_init(free_bar(q), NWC);
            mbar_init(step_bar(q), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(maps_bar(b), 1);  // the last window warp, once the chunk's map is out
            mbar_init(entries_bar(b), 1);
            wcount[b] = 0;
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
    const int CH = NWC * W;
    const long long total = static_cast<long long>(sa.ng) * sa.nc;
    // step tickets of the last LAG + 1 steps, newest at hist[0]
    auto push = [](int (&hist)[LAG + 1], int tk) {
#pragma unroll
        for (int i = LAG; i > 0; --i) hist[i] = hist[i - 1];
        hist[0] = tk;
    };
    auto pending = [](const int (&hist)[LAG + 1]) {  // a replay is still to come
        bool any = false;
#pragma unroll
        for (int i = 0; i < LAG; ++i) any = any || hist[i] >= 0;
        return any;
    };

    if (warp == NWC + kStreamScanWarps) {
        // --------------------------------------------------------- ticket warp
        // publishes tickets until every scan warp has seen an invalid one
        if (lane == 0) {
            int invalid = 0;
            for (int j = 0; invalid < kStreamScanWarps; ++j) {
                if (j >= AHEAD) {
                    const int jf = j - AHEAD;
                    if (!mbar_wait(free_bar(jf % SLOTS), static_cast<uint32_t>((jf / SLOTS) & 1), wc,
                                   kSiteProducerEmpty))
                        return;
                }
                int tk = -1;
                if (invalid == 0) {
                    const long long tj = static_cast<long long>(atomicAdd(sa.ticket, 1u));
                    tk = tj < total ? static_cast<int>(tj) : -1;
                }
                if (tk < 0) ++invalid;
                step_ticket[j % SLOTS] = tk;
                mbar_arrive(step_bar(j % SLOTS));
            }
        }
        return;
    }

    if (warp >= NWC) {
        // ---------------------------------------------------------- scan warps
        // scan warp j handles the chunks of steps j, j + 2, j + 4, ...; once a
        // ticket is invalid every later one is too
        const int i0 = lane * V;  // first of this thread's lanes in the tile
        for (int k = warp - NWC;; k += kStreamScanWarps) {
            const int q = k % SLOTS;
            if (!warp_wait(step_bar(q), static_cast<uint32_t>((k / SLOTS) & 1), wc, kSiteStreamStep)) return;
            const int tk = step_ticket[q];
            if (tk < 0) return;
            const int cc = tk / sa.ng;
            const int gi = tk - cc * sa.ng;
            const size_t g0 = static_cast<size_t>(gi) * sa.nc;
            const int b = k % NB;
            if (!warp_wait(maps_bar(b), static_cast<uint32_t>((k / NB) & 1), wc, kSiteStreamStep)) return;
            const float2 *mp = wmap + b * NWC * DT;
            float Pc[V], Qc[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float2 m = cmap[b * DT + i0 + v];
                Pc[v] = m.x;
                Qc[v] = m.y;
            }
            const size_t slot = g0 + cc;
            float h[V];
            // batches of maps in flight: as many as the registers hold
            constexpr int BATCH = C::MINB > 1 ? 16 / V : 32 / V;
            if (!stream_lookback<DT, V, BATCH>(sa, gi, cc, i0, h, wc)) return;
#pragma unroll
            for (int v = 0; v < V; ++v) sa.incl[slot * DT + i0 + v] = __fmaf_rn(Pc[v], h[v], Qc[v]);
            __syncwarp();  // every lane's state written before lane 0's release
            if (lane == 0) st_release_gpu(sa.flag + slot, kChunkIncl);
            // the state entering every window, in chain order
            float *ep = wentry + b * NWC * DT;
            for (int j = 0; j < NWC; ++j) {
                const int w = BWD ? NWC - 1 - j : j;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    ep[w * DT + i0 + v] = h[v];
                    const float2 m = mp[w * DT + i0 + v];
                    h[v] = __fmaf_rn(m.x, h[v], m.y);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(entries_bar(b));
        }
    }

    // --------------------------------------------------------- window warps
    const int w = warp;  // window of every chunk this warp owns
    const int sA = w, sB = NWC + w;  // summary and replay stages
    const CUtensorMap *const maps[3] = {&tm_0, &tm_1, &tm_2};
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NIN; ++i) prefetch_tensormap(maps[i]);
    }
    // bulk copies of window w of ticket t into stage st (lane 0)
    auto issue = [&](int st, int t, bool replay) {
        const int cc = t / sa.ng;
        const int gi = t - cc * sa.ng;
        const int c = BWD ? sa.nc - 1 - cc : cc;
        const int brow = gi / sa.ndt;
        const int x0 = (gi - brow * sa.ndt) * DT;
        const bool skip_out = BWD && !replay;  // the backward summary needs a and grad_out only
        const uint32_t fb = full_bar(st);
        mbar_arrive_expect_tx(fb, (skip_out ? NIN - 1 : NIN) * geo.tile_bytes);
        const int y = c * CH + w * W;
#pragma unroll
        for (int i = 0; i < NIN; ++i) {
            if (skip_out && i == 1) continue;
            const int dy = BWD ? (i == 0 ? 1 : (i == 1 ? -1 : 0)) : 0;
            tma_load_3d(smem_addr(tile(st, i)), maps[i], x0, y + dy, brow, fb);
        }
    };
    int uA = 0, uB = 0;  // copies waited on per stage (phase parity)
    int iA = 0, iB = 0;  // copies issued per stage
    // before leaving early: every copy this warp issued has landed (bounded,
    // blind to the abort flag: copies in flight always land)
    auto drain = [&]() {
        if (lane != 0) return;
        const int st[2] = {sA, sB};
        const int issued[2] = {iA, iB};
        const int waited[2] = {uA, uB};
        for (int i = 0; i < 2; ++i) {
            if (issued[i] == waited[i]) continue;
            const uint32_t fb = full_bar(st[i]);
            const uint32_t par = static_cast<uint32_t>(waited[i] & 1);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(fb, par)) {
                if (global_timer_ns() - t0 > wc.timeout_ns) {
                    record_error(wc, kErrTimeout, kSiteDrain);
                    break;
                }
            }
        }
    };
    int hist[LAG + 1];
#pragma unroll
    for (int i = 0; i <= LAG; ++i) hist[i] = -1;
    if (!warp_wait(step_bar(0), 0u, wc, kSiteStreamStep)) return;
    int tk = step_ticket[0];
    if (tk >= 0) {
        if (lane == 0) issue(sA, tk, false);
        ++iA;
    }
    for (int k = 0;; ++k) {
        push(hist, tk);
        // ------------------------------------------------ summary of ticket k
        if (tk >= 0) {
            const int t = tk;
            const int cc = t / sa.ng;
            const int gi = t - cc * sa.ng;
            const int c = BWD ? sa.nc - 1 - cc : cc;
            const int wbase = c * CH + w * W;
            const int nrows = min(max(T - wbase, 0), W);
            if (!warp_wait(full_bar(sA), static_cast<uint32_t>(uA & 1), wc, kSiteConsumerFull)) { drain(); return; }
            ++uA;
            const St *ta = tile(sA, 0);
            const St *tb = tile(sA, NIN - 1);
            const int b = k % NB;
            // the window's map (rows past T are identity steps)
            float P[V], Q[V];
#pragma unroll
            for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
            for (int g8 = 0; g8 < nrows; g8 += 8) {
                const int r0 = BWD ? ((nrows - 1 - g8) & ~7) : g8;  // groups of eight, chain order
                float xa[8][V], xb[8][V];
                load8<St, V, DT>(ta, r0, lane, xa);
                load8<St, V, DT>(tb, r0, lane, xb);
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int r = BWD ? 7 - rr : rr;
                    if (r0 + r < nrows) {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            P[v] = __fmul_rn(xa[r][v], P[v]);
                            Q[v] = __fmaf_rn(xa[r][v], Q[v], xb[r][v]);
                        }
                    }
                }
            }
            float2 *mp = wmap + b * NWC * DT + w * DT + lane * V;
#pragma unroll
            for (int v = 0; v < V; ++v) mp[v] = make_float2(P[v], Q[v]);
            __syncwarp();
            unsigned int before = 0;
            if (lane == 0) before = atom_add_acq_rel_cta(wcount + b, 1u);
            before = __shfl_sync(0xffffffffu, before, 0);
            if (before == NWC - 1) {
                // the last window warp of this chunk: compose the window maps
                // in chain order and publish the chunk's map at once, so that
                // look-backs elsewhere find it without waiting for this CTA's
                // scan warps
                __syncwarp();
                const float2 *cm = wmap + b * NWC * DT;
                float Pc[V], Qc[V];
#pragma unroll
                for (int v = 0; v < V; ++v) { Pc[v] = 1.0f; Qc[v] = 0.0f; }
                for (int j = 0; j < NWC; ++j) {
                    const int ww = BWD ? NWC - 1 - j : j;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float2 m = cm[ww * DT + lane * V + v];
                        Qc[v] = __fmaf_rn(m.x, Qc[v], m.y);
                        Pc[v] = __fmul_rn(m.x, Pc[v]);
                    }
                }
                const size_t slot = static_cast<size_t>(gi) * sa.nc + cc;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    cmap[b * DT + lane * V + v] = make_float2(Pc[v], Qc[v]);
                    sa.agg[slot * DT + lane * V + v] = make_float2(Pc[v], Qc[v]);
                }
                __syncwarp();  // every lane's map written before lane 0's release
                if (lane == 0) {
                    st_release_gpu(sa.flag + slot, kChunkAgg);
                    wcount[b] = 0;  // next used NB steps on, after the scan warp has taken this chunk
                    mbar_arrive(maps_bar(b));
                }
            }
        }
        // ------------------- next ticket; its summary tile into the free stage
        int tn = -1;
        if (tk >= 0) {
            const int q = (k + 1) % SLOTS;
            if (!warp_wait(step_bar(q), static_cast<uint32_t>(((k + 1) / SLOTS) & 1), wc, kSiteStreamStep)) {
                drain();
                return;
            }
            tn = step_ticket[q];
            __syncwarp();  // the stage's tile read by every lane before it is overwritten
            if (tn >= 0) {
                if (lane == 0) issue(sA, tn, false);
                ++iA;
            }
        }
        // ------------------------------------------- replay of ticket k - LAG
        if (hist[LAG] >= 0) {
            const int t = hist[LAG];
            const int kc = k - LAG;  // the step whose chunk this is
            const int cc = t / sa.ng;
            const int gi = t - cc * sa.ng;
            const int c = BWD ? sa.nc - 1 - cc : cc;
            const int brow = gi / sa.ndt;
            const int x0 = (gi - brow * sa.ndt) * DT;
            const int d = x0 + lane * V;
            const bool lane_ok = d < D;
            const int wbase = c * CH + w * W;
            const int nrows = min(max(T - wbase, 0), W);
            const int b = kc % NB;
            if (!warp_wait(full_bar(sB), static_cast<uint32_t>(uB & 1), wc, kSiteConsumerFull)) { drain(); return; }
            ++uB;
            if (!warp_wait(entries_bar(b), static_cast<uint32_t>((kc / NB) & 1), wc, kSiteStreamStep)) {
                drain();
                return;
            }
            const St *ta = tile(sB, 0);
            const St *tb = tile(sB, NIN - 1);
            float h[V];
            const float *ep = wentry + b * NWC * DT + w * DT + lane * V;
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = ep[v];
            const size_t rowb = static_cast<size_t>(brow) * T;
            if constexpr (!BWD) {
                St *op = out0 + (rowb + wbase) * D + d;
                for (int g8 = 0; g8 < nrows; g8 += 8) {
                    float xa[8][V], xb[8][V];
                    load8<St, V, DT>(ta, g8, lane, xa);
                    load8<St, V, DT>(tb, g8, lane, xb);
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        if (g8 + r < nrows) {
#pragma unroll
                            for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[r][v], h[v], xb[r][v]);
                            if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(g8 + r) * D, h);
                        }
                    }
                }
                if (last != nullptr && lane_ok && nrows > 0 && wbase + nrows == T) {
#pragma unroll
                    for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
                }
            } else {
                const St *th = tile(sB, 1);
                St *gap = out0 + (rowb + wbase) * D + d;
                St *gbp = out1 + (rowb + wbase) * D + d;
                for (int g8 = 0; g8 < nrows; g8 += 8) {
                    const int r0 = (nrows - 1 - g8) & ~7;
                    float xa[8][V], xh[8][V], xg[8][V];
                    load8<St, V, DT>(ta, r0, lane, xa);
                    load8<St, V, DT>(th, r0, lane, xh);
                    load8<St, V, DT>(tb, r0, lane, xg);
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int r = 7 - rr;
                        if (r0 + r < nrows) {
                            float gav[V];
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                h[v] = __fmaf_rn(xa[r][v], h[v], xg[r][v]);
                                gav[v] = __fmul_rn(h[v], xh[r][v]);
                            }
                            if (lane_ok) {
                                store_lanes<St, V>(gbp + static_cast<size_t>(r0 + r) * D, h);
                                store_lanes<St, V>(gap + static_cast<size_t>(r0 + r) * D, gav);
                            }
                        }
                    }
                }
            }
            __syncwarp();  // the stage's tile read by every lane before it is overwritten
        }
        // ------------------------- the next replay's tile into the free stage
        if (hist[LAG - 1] >= 0) {
            if (lane == 0) issue(sB, hist[LAG - 1], true);
            ++iB;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(free_bar(k % SLOTS));
        if (tk < 0 && !pending(hist)) return;
        tk = tn;
    }
}

}  // namespace lrscan
