// Time-tiled scan kernels: a CTA owns one batch row and DT channel lanes and
// walks the whole sequence in windows of W = S*L time steps.  A producer warp
// streams the windows' input tiles into a ring of shared-memory stages with
// 3-D bulk tensor copies (TMA) completed on mbarriers.  Consumer thread
// (s, g) owns lanes [g*V, g*V+V) of sub-chunk s (rows s*L .. s*L+L-1 of the
// window): it copies its rows into registers, releases the stage at once so
// the producer can refill it, and keeps the recurrence state in fp32.
//
//  S == 1  ("seq"): every thread runs the recurrence straight through all
//          windows (L rows each, streamed from shared memory in a fully
//          unrolled loop), one fused multiply-add per step, bit-identical to
//          the sequential definition.  No barrier between consumer warps.
//  S  > 1  ("window"): thread (s, g) summarizes its sub-chunk as the affine
//          map h -> P*h + Q (triton_training_scan.py, _real_chunk_summary);
//          the sub-chunk entry states follow from the window's carried state
//          through the maps in order (the serial prefix of _real_chunk_prefix,
//          inside one CTA; identity maps leave the state bit-for-bit
//          unchanged), either by DT "lane" threads that walk all S maps of
//          one lane and record every entry (few instructions, one extra
//          barrier) or by every thread folding the maps before its own
//          sub-chunk (short critical path); then every thread replays its
//          sub-chunk (_real_chunk_replay).  One pass over HBM: 3 elements per
//          (t, d) forward, 5 backward.
//
// With G = DT/V = 32 a warp is exactly one sub-chunk row range, so its
// shared-memory reads of one row are 32 consecutive words (conflict-free).
//
// Backward windows run last-to-first.  The decay tile is loaded one row late
// (a_{t+1}) and the out tile one row early (h_{t-1}), so the tensor copy's zero
// fill supplies a_T = 0 and h_{-1} = 0 at the sequence ends; the reverse
// recurrence g_t = fma(a_{t+1}, g_{t+1}, grad_out_t) then has the same shape
// as the forward one.
//
// S and the stage count are launch-time parameters; DT, V and L are compiled.
//
// EXT instantiations add the carried state and segment resets (StateArgs):
// the forward starts from h0 and zeroes a_t where a segment starts; the
// backward starts from grad_last (entering through a'_T = 1), zeroes
// a'_{t+1} where step t+1 starts a segment, writes grad_a = +0 where step t
// starts one, reads h0 as h_{-1} and writes grad_h0 = a'_0 * g_0.  Each warp
// turns the segment positions of its rows into a bit mask with one ballot
// per window (loaded one window ahead).  The plain instantiations are
// unchanged.
#pragma once

#include "scan_common.cuh"
#include "state_args.h"

namespace lrscan {

// Compile-time shape.  MAXT / MINB feed __launch_bounds__.  A shape is either
// sequential (launched with S == 1, rows streamed from shared memory) or
// windowed (S > 1, each thread's L rows held in registers).
template <typename St_, int DT_, int V_, int L_, int NIN_, int MAXT_, int MINB_, bool SEQ_, bool PT_ = false,
          bool EX_ = false>
struct WinShape {
    using St = St_;
    static constexpr bool SEQ = SEQ_;
    // windowed prefix: false = lane threads scan the maps, true = every thread
    // folds the maps before its own sub-chunk
    static constexpr bool PT = PT_;
    // exact windowed tile: the lane threads walk the window's rows one step at
    // a time (no sub-chunk maps), so the entry states and every replayed value
    // are the sequential definition's own
    static constexpr bool EX = EX_;
    static_assert(!EX_ || (!SEQ_ && !PT_), "exact walk: a lane-scan windowed shape");
    static constexpr int DT = DT_;    // lanes per CTA
    static constexpr int V = V_;      // lanes per thread
    static constexpr int L = L_;      // steps per sub-chunk (held in registers)
    static constexpr int NIN = NIN_;  // input tiles per window (2 forward, 3 backward)
    static constexpr int G = DT / V;  // lane groups per row
    static constexpr int MAXT = MAXT_;
    static constexpr int MINB = MINB_;
    static constexpr int ROW_BYTES = DT * static_cast<int>(sizeof(St));
    static constexpr int SMAX = SEQ ? 1 : (MAXT - 32) / G;  // most sub-chunks a launch may use
    static_assert(DT % V == 0, "lane tile must split into lane groups");
    static_assert(ROW_BYTES % 16 == 0, "tensor-copy rows are multiples of 16 bytes");
    static_assert(DT <= 256, "tensor-copy box limit");
    static_assert(L >= 1 && L <= 64, "rows per window (sequential) or per sub-chunk");
    static_assert(SEQ || L <= 16 || (EX_ && L <= 32), "windowed sub-chunks are held in registers");
};

// Launch-time geometry (filled by the host from S and the stage count).
struct WinGeom {
    int S;             // sub-chunks per window
    int nstage;        // pipeline depth
    int W;             // rows per window = S*L
    int tile_bytes;    // W * ROW_BYTES
    int stage_bytes;   // NIN * tile_bytes
    int bar_off;       // byte offsets into dynamic shared memory
    int scan_off;
    int flag_off;
    int smem_bytes;
    int T, D, nwin;
};

template <class C>
__host__ __device__ inline WinGeom make_win_geom(int S, int nstage, int T, int D) {
    WinGeom g{};
    g.S = S;
    g.nstage = nstage;
    g.W = S * C::L;
    g.tile_bytes = g.W * C::ROW_BYTES;
    g.stage_bytes = C::NIN * g.tile_bytes;
    g.bar_off = nstage * g.stage_bytes;
    g.scan_off = g.bar_off + 2 * nstage * 8;
    // lane scan: sub-chunk maps (P,Q) [S][DT] float2 and entry states [S][DT];
    // per-thread prefix: maps [2][S][DT] float2 and carried state [2][DT]
    const int scan_bytes = S <= 1 ? 0 : (C::PT ? 2 * S * C::DT * 8 + 2 * C::DT * 4 : S * C::DT * 12);
    g.flag_off = g.scan_off + scan_bytes;
    g.smem_bytes = g.flag_off + 16;
    g.T = T;
    g.D = D;
    g.nwin = (T + g.W - 1) / g.W;
    return g;
}

// Output staging of kernels that write their result tiles back with bulk
// tensor stores: two buffers of one window (W rows x DT lanes, storage type)
// after the rest of the layout.
__host__ __device__ inline int win_out_off(const WinGeom &g) { return (g.smem_bytes + 127) & ~127; }
__host__ __device__ inline int win_out_smem(const WinGeom &g, int planes = 1, int buffers = 2) {
    return win_out_off(g) + buffers * planes * g.tile_bytes;
}
// Window tiles that stage their outputs this way: the lane-scan tiles (out
// forward; grad_a and grad_b backward).
template <class C> __host__ __device__ constexpr bool win_staged() { return !C::SEQ && !C::PT; }

// NP output planes staged per processed window, double-buffered:
// [2][NP][W][DT] storage elements at win_out_off.  Every consumer thread
// writes its rows into plane(k, p) and fences them for the async proxy; after
// the next window's first barrier one thread stores them (store), so the
// buffers alternate and each store overlaps a window of compute.
// NB = 1 keeps one buffer per plane: the thread that stores a window must
// then wait for its reads (bulk_wait_read<0>) before the next replay writes.
template <int NP, class St, int NB = 2>
struct OutStage {
    St *buf;
    int elems;  // W * DT
    __device__ __forceinline__ St *plane(int kw, int p) const {
        const int b = NB == 1 ? 0 : (NB == 2 ? (kw & 1) : kw % NB);
        return buf + (b * NP + p) * elems;
    }
    // bulk tensor stores of processed window kw's planes at (x, y, z), one group
    __device__ __forceinline__ void store(const CUtensorMap *const (&maps)[NP], int kw, int x, int y, int z) const {
#pragma unroll
        for (int p = 0; p < NP; ++p) tma_store_3d(maps[p], smem_addr(plane(kw, p)), x, y, z);
        bulk_commit();
    }
};
template <int NP, class St, int NB = 2>
__device__ __forceinline__ OutStage<NP, St, NB> make_out_stage(unsigned char *smem, const WinGeom &g) {
    return OutStage<NP, St, NB>{reinterpret_cast<St *>(smem + win_out_off(g)),
                                g.tile_bytes / static_cast<int>(sizeof(St))};
}

// Shared-memory layout of one CTA, with the launch geometry copied into
// registers once (reading it through a pointer to the parameter would turn
// every access into a generic load through L1).
struct WinSmem {
    unsigned char *base;
    int stage_bytes, tile_bytes, bar_off, scan_off, flag_off, nstage, S, W, nwin;

    static __device__ __forceinline__ WinSmem make(unsigned char *b, const WinGeom &g) {
        WinSmem m;
        m.base = b;
        m.stage_bytes = g.stage_bytes;
        m.tile_bytes = g.tile_bytes;
        m.bar_off = g.bar_off;
        m.scan_off = g.scan_off;
        m.flag_off = g.flag_off;
        m.nstage = g.nstage;
        m.S = g.S;
        m.W = g.W;
        m.nwin = g.nwin;
        return m;
    }
    template <class C> __device__ __forceinline__ typename C::St *tile(int stage, int which) const {
        return reinterpret_cast<typename C::St *>(base + stage * stage_bytes + which * tile_bytes);
    }
    __device__ __forceinline__ uint32_t full_bar(int stage) const { return smem_addr(base + bar_off + stage * 8); }
    __device__ __forceinline__ uint32_t empty_bar(int stage) const {
        return smem_addr(base + bar_off + (nstage + stage) * 8);
    }
    // (P, Q) of sub-chunk s for lane v*G + g at [par][s][v*G + g]: consecutive
    // threads touch consecutive words (no bank conflicts); par is 0 for the
    // lane scan
    template <class C> __device__ __forceinline__ float2 *sPQ(int par) const {
        return reinterpret_cast<float2 *>(base + scan_off) + par * S * C::DT;
    }
    // lane scan: entry state of sub-chunk s for lane v*G + g at [s][v*G + g]
    template <class C> __device__ __forceinline__ float *sEntry() const {
        return reinterpret_cast<float *>(base + scan_off + S * C::DT * 8);
    }
    // per-thread prefix: carried state [par][v*G + g]
    template <class C> __device__ __forceinline__ float *sCarry(int par) const {
        return reinterpret_cast<float *>(base + scan_off + 2 * S * C::DT * 8) + par * C::DT;
    }
    __device__ __forceinline__ volatile int *abort_flag() const {
        return reinterpret_cast<volatile int *>(base + flag_off);
    }
};

// Producer: one elected lane streams the windows into the stage ring in
// processing order; row_of(k, i) is the time coordinate of input tile i of
// the k-th processed window.  Before returning (normally or on abort) it
// waits, bounded, for every copy it issued, so none lands after the CTA exits.
template <class C, class RowOf>
__device__ __forceinline__ void win_producer(const WinSmem &sm, const CUtensorMap *const (&maps)[C::NIN], int x0,
                                             int z, RowOf row_of, const WaitCtx &wc) {
    const WinSmem &g = sm;
    for (int i = 0; i < C::NIN; ++i) prefetch_tensormap(maps[i]);
    int issued = 0;
    int stage = 0, use = 0;
    for (int k = 0; k < g.nwin; ++k) {
        if (use > 0 && !mbar_wait(sm.empty_bar(stage), (use - 1) & 1, wc, kSiteProducerEmpty)) break;
        const uint32_t fb = sm.full_bar(stage);
        mbar_arrive_expect_tx(fb, g.stage_bytes);
#pragma unroll
        for (int i = 0; i < C::NIN; ++i)
            tma_load_3d(smem_addr(sm.tile<C>(stage, i)), maps[i], x0, row_of(k, i), z, fb);
        issued = k + 1;
        if (++stage == g.nstage) { stage = 0; ++use; }
    }
    // Drain: the most recent fill of each stage must have landed.
    const int first = issued > g.nstage ? issued - g.nstage : 0;
    for (int k = first; k < issued; ++k) {
        const uint32_t fb = sm.full_bar(k % g.nstage);
        const uint32_t par = (k / g.nstage) & 1;
        if (mbar_try_wait(fb, par)) continue;
        // bounded, and deliberately blind to the abort flag: copies in flight always land
        const uint64_t start = global_timer_ns();
        while (!mbar_try_wait(fb, par)) {
            if (global_timer_ns() - start > wc.timeout_ns) {
                record_error(wc, kErrTimeout, kSiteDrain);
                break;
            }
        }
    }
}

// Segment positions of one batch row: rows outside [0, T), and every row when
// there is no position tensor, read as 1 (no reset).
struct SegRow {
    const int32_t *p;
    int T;
    __device__ __forceinline__ int32_t at(int t) const {
        return (p != nullptr && t >= 0 && t < T) ? __ldg(p + t) : 1;
    }
};

// Lane threads of the in-window prefix own lane index i of the [DT] scan
// arrays, i.e. channel d0 + (i % G) * V + i / G.
template <class C>
__device__ __forceinline__ int lane_channel(int d0, int i) {
    return d0 + (i % C::G) * C::V + i / C::G;
}

// Lane scan of one window: lane thread i carries c through the S sub-chunk
// maps pq[s * DT + i] in order (REVERSE: from S-1 down), recording each
// sub-chunk's entry value first.  Maps are read four at a time ahead of their
// fmas, so the loads do not queue behind the entry stores (same fmas, same
// order as a one-map-at-a-time walk).
template <bool REVERSE, int DT>
__device__ __forceinline__ float lane_walk(const float2 *pq, float *entry, int S, int i, float c) {
    for (int i0 = 0; i0 < S; i0 += 4) {
        float2 m[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int s = REVERSE ? S - 1 - (i0 + j) : i0 + j;
            m[j] = (i0 + j < S) ? pq[s * DT + i] : make_float2(1.0f, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (i0 + j < S) {
                const int s = REVERSE ? S - 1 - (i0 + j) : i0 + j;
                entry[s * DT + i] = c;
                c = __fmaf_rn(m[j].x, c, m[j].y);
            }
        }
    }
    return c;
}

// Exact walk of one window (EX tiles).  Lane thread i carries c through the
// window's rows with the sequential step itself, in order (REVERSE: last row
// first), and records the value entering each sub-chunk at entry[s * DT + i];
// the sub-chunk replays then repeat exactly these steps, so every stored
// value is bit-identical to the sequential scan.  ta / tb are the window's
// decay and addend tiles (backward: a_{t+1} and grad_out_t), row stride DT;
// lane thread i reads column (i % G) * V + i / G, the lane its scan index
// stands for.  Rows from `real` on lie past the sequence end and are identity
// steps (a = 1, addend 0); rmask[s] holds the sub-chunk's reset rows (EXT:
// a = 0 there); with ONE_AT (EXT backward) row real - 1, step T-1, takes
// a = 1 (grad_last enters through a'_T = 1).  Every override is the one the
// replay applies to its register copy of the same row.
template <class C, bool REVERSE, bool EXT, bool ONE_AT>
__device__ __forceinline__ float exact_walk(const typename C::St *ta, const typename C::St *tb, float *entry,
                                           const uint32_t *rmask, int S, int i, int real, float c) {
    constexpr int L = C::L, DT = C::DT, G = C::G, V = C::V;
    const int col = (i % G) * V + i / G;
    for (int ii = 0; ii < S; ++ii) {
        const int s = REVERSE ? S - 1 - ii : ii;
        entry[s * DT + i] = c;
        float x[L], y[L];
#pragma unroll
        for (int j = 0; j < L; ++j) {
            float t1[1], t2[1];
            unpack_lanes<typename C::St, 1>(ta + (s * L + j) * DT + col, t1);
            unpack_lanes<typename C::St, 1>(tb + (s * L + j) * DT + col, t2);
            x[j] = t1[0];
            y[j] = t2[0];
        }
        const uint32_t rb = EXT ? rmask[s] : 0u;
#pragma unroll
        for (int jj = 0; jj < L; ++jj) {
            const int j = REVERSE ? L - 1 - jj : jj;
            const int r = s * L + j;
            float xv = ((rb >> j) & 1u) ? 0.0f : x[j];
            float yv = y[j];
            if (r >= real) { xv = 1.0f; yv = 0.0f; }
            else if (ONE_AT && r == real - 1) xv = 1.0f;
            c = __fmaf_rn(xv, c, yv);
        }
    }
    return c;
}

template <class C>
__device__ __forceinline__ void win_init(const WinSmem &sm, int consumer_warps, int S) {
    constexpr int DT = C::DT;
    const WinSmem &g = sm;
    if (threadIdx.x == 0) {
        for (int s = 0; s < g.nstage; ++s) {
            mbar_init(sm.full_bar(s), 1);
            mbar_init(sm.empty_bar(s), consumer_warps);
        }
        *sm.abort_flag() = 0;
        fence_mbar_init();
    }
    if (C::PT && S > 1) {
        // carried state starts at zero (h_{-1} = 0 forward, g_T = 0 backward)
        float *c = reinterpret_cast<float *>(sm.base + g.scan_off + 2 * g.S * DT * 8);
        for (int i = threadIdx.x; i < 2 * DT; i += blockDim.x) c[i] = 0.0f;
    }
    __syncthreads();
}

// ============================================================================
// Forward
// ============================================================================
template <class C, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
win_fwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_out, typename C::St *__restrict__ out, float *__restrict__ last,
               const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns,
               const __grid_constant__ StateArgs sx) {
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    // lane-scan tiles stage out in shared memory (two window buffers, written
    // back by bulk tensor stores that clip rows past T and lanes past D);
    // sequential and per-thread-prefix tiles store from registers
    constexpr bool TS = win_staged<C>();
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    win_init<C>(sm, NT / 32, S);
    pdl_trigger();
    pdl_wait();  // inputs may come from the previous kernel in the stream
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D;

    if (static_cast<int>(threadIdx.x) >= NT) {  // producer warp
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[2] = {&tm_a, &tm_b};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow, [W](int k, int) { return k * W; }, wc);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    float h[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h[v] = 0.0f;
    float carry = 0.0f;  // window-to-window state of lane threadIdx.x (lane scan, threads < DT)
    bool failed = false;
    int stage = 0, use = 0;
    const OutStage<1, St> ost = make_out_stage<1, St>(smem_raw, geom);
    const CUtensorMap *const omaps[1] = {&tm_out};
    // one thread outside the lane scan issues each window's store one window late
    const bool issuer = TS && static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    int replayed = 0;
    // EXT: this warp's rows start at window row wrow; bit j of rbits is a
    // reset at row s*L + j of the current window.  Positions are loaded two
    // windows ahead (pos_next: window k+1, pos_next2: window k+2).
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    const int wrow = ((threadIdx.x & ~31u) / G) * L;
    int32_t pos_next = 1, pos_next2 = 1;
    if constexpr (EXT) {
        static_assert((G >= 32 ? 1 : 32 / G) * L <= 32, "one ballot covers a warp's rows");
        if (sx.h0 != nullptr) {
            const float *h0 = sx.h0 + static_cast<size_t>(brow) * D;
            if (lane_ok) {
#pragma unroll
                for (int v = 0; v < V; ++v) h[v] = h0[d + v];
            }
            if (!C::SEQ && static_cast<int>(threadIdx.x) < DT) {
                const int ch = lane_channel<C>(d0, threadIdx.x);
                const float c0 = ch < D ? h0[ch] : 0.0f;
                if constexpr (C::PT) sm.sCarry<C>(0)[threadIdx.x] = c0;  // read after the first barrier
                else carry = c0;
            }
        }
        pos_next = seg.at(wrow + lane);
        pos_next2 = seg.at(sm.W + wrow + lane);
    }

    for (int k = 0; k < sm.nwin; ++k) {
        uint32_t rbits = 0;
        if constexpr (EXT) {
            rbits = __ballot_sync(0xffffffffu, pos_next == 0) >> (s * L - wrow);
            pos_next = pos_next2;
            pos_next2 = seg.at((k + 2) * sm.W + wrow + lane);
        }
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if constexpr (EXT && C::SEQ) ok = __all_sync(0xffffffffu, ok);  // keep the warp's ballots converged
        const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;
        const St *tb = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;
        if constexpr (C::SEQ) {
            if (!ok) { failed = true; break; }
            // straight through the window's L rows, one fma per step
            const int rbase = k * sm.W;
            const int n = min(T - rbase, L);
            St *op = out + (row0 + rbase) * D + d;
            if (n == L) {
                // full window: rows to registers as packed words first (all the
                // shared-memory loads issue before the dependent chain starts)
                using Raw = typename RawOf<St, V>::T;
                Raw ra[L], rb[L];
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    ra[j] = load_raw<St, V>(ta + j * DT);
                    rb[j] = load_raw<St, V>(tb + j * DT);
                }
                auto rows = [&](auto masked) {
#pragma unroll
                    for (int j = 0; j < L; ++j) {
                        float x[V], y[V];
                        widen_raw(ra[j], x);
                        widen_raw(rb[j], y);
                        if constexpr (decltype(masked)::value) {
#pragma unroll
                            for (int v = 0; v < V; ++v) x[v] = ((rbits >> j) & 1u) ? 0.0f : x[v];
                        }
#pragma unroll
                        for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(x[v], h[v], y[v]);
                        if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
                    }
                };
                // a window without a segment start runs the plain loop (warp-uniform)
                if (EXT && rbits != 0) rows(std::true_type{});
                else rows(std::false_type{});
            } else {
                for (int j = 0; j < n; ++j) {
                    float x[V], y[V];
                    unpack_lanes<St, V>(ta + j * DT, x);
                    unpack_lanes<St, V>(tb + j * DT, y);
                    if constexpr (EXT) {
#pragma unroll
                        for (int v = 0; v < V; ++v) x[v] = ((rbits >> j) & 1u) ? 0.0f : x[v];
                    }
#pragma unroll
                    for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(x[v], h[v], y[v]);
                    if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty_bar(stage));
            if (++stage == sm.nstage) { stage = 0; ++use; }
        } else {
        const int rbase = k * sm.W + s * L;
        const int n = min(max(T - rbase, 0), L);
        float xa[L][V], xb[L][V];
        if (ok) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
                unpack_lanes<St, V>(ta + j * DT, xa[j]);
                unpack_lanes<St, V>(tb + j * DT, xb[j]);
            }
        }
        // exact tiles release the stage only after the walk has read it
        const int cur = stage;
        if constexpr (!C::EX) {
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
        }
        if (++stage == sm.nstage) { stage = 0; ++use; }
        if constexpr (C::EX && EXT) {
            // the walk takes the reset rows of every sub-chunk from here
            if (lg == 0) reinterpret_cast<uint32_t *>(sm.sPQ<C>(0))[s] = rbits & ((1u << L) - 1u);
        }
        // sub-chunk summary h -> P*h + Q (an empty tail sub-chunk is the identity)
        float P[V], Q[V];
#pragma unroll
        for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
        if constexpr (EXT) {
            if (rbits != 0) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
#pragma unroll
                    for (int v = 0; v < V; ++v) xa[j][v] = ((rbits >> j) & 1u) ? 0.0f : xa[j][v];
                }
            }
        }
        if (n < L) {
            // tail sub-chunk: steps past T become exact identity steps (a=1, b=0)
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    xa[j][v] = j < n ? xa[j][v] : 1.0f;
                    xb[j][v] = j < n ? xb[j][v] : 0.0f;
                }
            }
        }
        const int par = C::PT ? (k & 1) : 0;
        float2 *pq = sm.sPQ<C>(par);
        if constexpr (!C::EX) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    P[v] = __fmul_rn(xa[j][v], P[v]);
                    Q[v] = __fmaf_rn(xa[j][v], Q[v], xb[j][v]);
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
        }
        if (bar_sync_or(1, NT, !ok)) { failed = true; break; }
        if (issuer && k > 0) {
            // every thread's rows of window k-1 are staged (fenced before the
            // barrier above); once this store has been issued, the one before
            // it must have finished reading the buffer window k is about to fill
            ost.store(omaps, k - 1, d0, (k - 1) * sm.W, brow);
            bulk_wait_read<1>();
        }
        if constexpr (C::EX) {
            // lane threads walk the window's rows exactly (sequential steps),
            // recording every sub-chunk's entry state; then the stage is free
            float *entry = sm.sEntry<C>();
            if (static_cast<int>(threadIdx.x) < DT)
                carry = exact_walk<C, false, EXT, false>(sm.tile<C>(cur, 0), sm.tile<C>(cur, 1), entry,
                                                         reinterpret_cast<const uint32_t *>(pq), S, threadIdx.x,
                                                         T - k * sm.W, carry);
            bar_sync_or(1, NT, false);
            if (lane == 0) mbar_arrive(sm.empty_bar(cur));
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = entry[s * DT + v * G + lg];
        } else if constexpr (!C::PT) {
            // Threads 0..DT-1 each own one lane: push the carried state through
            // the sub-chunk maps in order, recording every sub-chunk's entry
            // state (_real_chunk_prefix within the window; identity maps exact).
            float *entry = sm.sEntry<C>();
            if (static_cast<int>(threadIdx.x) < DT) carry = lane_walk<false, DT>(pq, entry, S, threadIdx.x, carry);
            bar_sync_or(1, NT, false);
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = entry[s * DT + v * G + lg];
        } else {
            // every thread folds the maps of sub-chunks 0..s-1 into the carried
            // state itself (shorter critical path, more instructions)
            const float *cs = sm.sCarry<C>(par);
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = cs[v * G + lg];
#pragma unroll
            for (int i = 0; i < C::SMAX - 1; ++i) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float2 m = (i < s) ? pq[i * DT + v * G + lg] : make_float2(1.0f, 0.0f);
                    if (i < s) h[v] = __fmaf_rn(m.x, h[v], m.y);
                }
            }
        }
        if constexpr (TS) {
            St *op = ost.plane(k, 0) + (s * L) * DT + lg * V;
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
                store_lanes<St, V>(op + j * DT, h);
            }
            fence_proxy_async_smem();
            replayed = k + 1;
        } else if (n == L) {
            St *op = out + (row0 + rbase) * D + d;
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
                if (lane_ok) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
            }
        } else {
            St *op = out + (row0 + rbase) * D + d;
            // identity steps past T leave h unchanged; their rows are not stored
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(xa[j][v], h[v], xb[j][v]);
                if (lane_ok && j < n) store_lanes<St, V>(op + static_cast<size_t>(j) * D, h);
            }
        }
        if (C::PT && s == S - 1) {
            float *nc = sm.sCarry<C>((k & 1) ^ 1);
#pragma unroll
            for (int v = 0; v < V; ++v) nc[v * G + lg] = h[v];
        }
        // the thread whose sub-chunk holds step T-1 owns the final state
        if (last != nullptr && lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
            for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
        }
        }
    }
    if (C::SEQ && !failed && last != nullptr && lane_ok) {
#pragma unroll
        for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
    }
    if constexpr (TS) {
        // the last window's tile (not after an abort), then every store
        // complete before the CTA's shared memory goes away
        const bool aborted = bar_sync_or(1, NT, replayed != sm.nwin);
        if (issuer) {
            if (!aborted && replayed > 0) ost.store(omaps, replayed - 1, d0, (replayed - 1) * sm.W, brow);
            bulk_wait<0>();
        }
    }
}

// ============================================================================
// Backward
// ============================================================================
// STAGED: gb and ga point into the shared-memory staging tiles (row stride
// DT, every row written; the bulk store clips rows past T and lanes past D).
template <class C, bool MASK, bool STAGED>
__device__ __forceinline__ void bwd_rows(const float (&xa)[C::L][C::V], const float (&xh)[C::L][C::V],
                                         const float (&xg)[C::L][C::V], float (&g)[C::V], int n, bool lane_ok,
                                         typename C::St *gb, typename C::St *ga, int D, uint32_t rbits) {
    using St = typename C::St;
    constexpr int V = C::V, L = C::L;
    // rows past T hold identity steps (a=1, grad_out=0), set by the caller: g
    // passes through them unchanged and they are not stored
#pragma unroll
    for (int j = L - 1; j >= 0; --j) {
        float gav[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            g[v] = __fmaf_rn(xa[j][v], g[v], xg[j][v]);
            gav[v] = __fmul_rn(g[v], xh[j][v]);
            if constexpr (MASK) gav[v] = ((rbits >> j) & 1u) ? 0.0f : gav[v];  // a_t unused at a reset
        }
        if constexpr (STAGED) {
            store_lanes<St, V>(gb + j * C::DT, g);
            store_lanes<St, V>(ga + j * C::DT, gav);
        } else if (lane_ok && (n == L || j < n)) {
            store_lanes<St, V>(gb + static_cast<size_t>(j) * D, g);
            store_lanes<St, V>(ga + static_cast<size_t>(j) * D, gav);
        }
    }
}

// grad_h0 = a'_0 * g_0 for the V lanes of the thread that finished step 0.
template <class C>
__device__ __forceinline__ void store_grad_h0(const StateArgs &sx, const SegRow &seg, size_t row0, int brow, int d,
                                              int D, const float (&g)[C::V]) {
    using St = typename C::St;
    float a0[C::V];
    load_lanes_global<St, C::V>(static_cast<const St *>(sx.a) + row0 * D + d, a0);
    const bool r0 = seg.at(0) == 0;
#pragma unroll
    for (int v = 0; v < C::V; ++v)
        sx.grad_h0[static_cast<size_t>(brow) * D + d + v] = r0 ? 0.0f : __fmul_rn(a0[v], g[v]);
}

template <class C, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
win_bwd_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_out,
               const __grid_constant__ CUtensorMap tm_go, const __grid_constant__ CUtensorMap tm_ga,
               const __grid_constant__ CUtensorMap tm_gb, typename C::St *__restrict__ grad_a,
               typename C::St *__restrict__ grad_b, const __grid_constant__ WinGeom geom, DevStatus *status,
               uint64_t timeout_ns, const __grid_constant__ StateArgs sx) {
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    // lane-scan tiles stage grad_a and grad_b in shared memory (two window
    // buffers of both planes) and write them back with bulk tensor stores
    constexpr bool TS = win_staged<C>();
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    win_init<C>(sm, NT / 32, S);
    pdl_trigger();
    pdl_wait();  // inputs may come from the previous kernel in the stream
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D;
    const int nwin = sm.nwin;

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[3] = {&tm_a, &tm_out, &tm_go};
            const int W = sm.W;
            // tile 0: a one step later; tile 1: out one step earlier; tile 2: grad_out
            win_producer<C>(sm, maps, d0, brow,
                            [W, nwin](int k, int i) { return (nwin - 1 - k) * W + (i == 0 ? 1 : (i == 1 ? -1 : 0)); },
                            wc);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    float g[V];
#pragma unroll
    for (int v = 0; v < V; ++v) g[v] = 0.0f;
    float carry = 0.0f;  // window-to-window adjoint of lane threadIdx.x (lane scan, threads < DT)
    int stage = 0, use = 0;
    bool failed = false;
    const OutStage<2, St> ost = make_out_stage<2, St>(smem_raw, geom);  // planes grad_a, grad_b
    const CUtensorMap *const omaps[2] = {&tm_ga, &tm_gb};
    // one thread outside the lane scan stores processed window kw (time rows
    // from (nwin - 1 - kw) * W) one window late
    const bool issuer = TS && static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    int replayed = 0;
    // EXT: bit j of r0bits / r1bits is a reset at row s*L + j / s*L + j + 1
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    const int wrow = ((threadIdx.x & ~31u) / G) * L;
    int32_t pos0_next = 1, pos1_next = 1, pos0_next2 = 1, pos1_next2 = 1;  // windows k+1, k+2
    float h0v[V];  // h_{-1}
#pragma unroll
    for (int v = 0; v < V; ++v) h0v[v] = 0.0f;
    if constexpr (EXT) {
        static_assert((G >= 32 ? 1 : 32 / G) * L <= 32, "one ballot covers a warp's rows");
        if (sx.h0 != nullptr && lane_ok) {
#pragma unroll
            for (int v = 0; v < V; ++v) h0v[v] = sx.h0[static_cast<size_t>(brow) * D + d + v];
        }
        if (sx.grad_last != nullptr) {
            const float *gl = sx.grad_last + static_cast<size_t>(brow) * D;
            if (lane_ok) {
#pragma unroll
                for (int v = 0; v < V; ++v) g[v] = gl[d + v];
            }
            if (!C::SEQ && static_cast<int>(threadIdx.x) < DT) {
                const int ch = lane_channel<C>(d0, threadIdx.x);
                const float c0 = ch < D ? gl[ch] : 0.0f;
                if constexpr (C::PT) sm.sCarry<C>(0)[threadIdx.x] = c0;  // read after the first barrier
                else carry = c0;
            }
        }
        const int wb0 = (nwin - 1) * sm.W + wrow + lane;
        pos0_next = seg.at(wb0);
        pos1_next = seg.at(wb0 + 1);
        pos0_next2 = seg.at(wb0 - sm.W);
        pos1_next2 = seg.at(wb0 - sm.W + 1);
    }

    for (int k = 0; k < nwin; ++k) {
        uint32_t r0bits = 0, r1bits = 0;
        if constexpr (EXT) {
            r0bits = __ballot_sync(0xffffffffu, pos0_next == 0) >> (s * L - wrow);
            r1bits = __ballot_sync(0xffffffffu, pos1_next == 0) >> (s * L - wrow);
            pos0_next = pos0_next2;
            pos1_next = pos1_next2;
            const int wb = (nwin - 3 - k) * sm.W + wrow + lane;
            pos0_next2 = seg.at(wb);
            pos1_next2 = seg.at(wb + 1);
        }
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if constexpr (EXT && C::SEQ) ok = __all_sync(0xffffffffu, ok);  // keep the warp's ballots converged
        const St *ta = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;  // a_{t+1}
        const St *th = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;  // h_{t-1}
        const St *tg = sm.tile<C>(stage, 2) + (s * L) * DT + lg * V;  // grad_out_t
        const int wbase = (nwin - 1 - k) * sm.W;
        if constexpr (C::SEQ) {
            if (!ok) { failed = true; break; }
            const int n = min(T - wbase, L);
            const size_t gofs = (row0 + wbase) * D + d;
            if (n == L) {
                auto rows = [&](auto special) {
#pragma unroll
                    for (int j = L - 1; j >= 0; --j) {
                        float x[V], hp[V], go[V], gav[V];
                        unpack_lanes<St, V>(ta + j * DT, x);
                        unpack_lanes<St, V>(th + j * DT, hp);
                        unpack_lanes<St, V>(tg + j * DT, go);
                        if constexpr (decltype(special)::value) {
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                // row T-1 takes grad_last through a'_T = 1; a'_{t+1} = 0 at a reset
                                if (j == L - 1) x[v] = k == 0 ? 1.0f : x[v];
                                x[v] = ((r1bits >> j) & 1u) ? 0.0f : x[v];
                                if (j == 0) hp[v] = wbase == 0 ? h0v[v] : hp[v];
                            }
                        }
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            g[v] = __fmaf_rn(x[v], g[v], go[v]);
                            gav[v] = __fmul_rn(g[v], hp[v]);
                            if constexpr (decltype(special)::value) gav[v] = ((r0bits >> j) & 1u) ? 0.0f : gav[v];
                        }
                        if (lane_ok) {
                            store_lanes<St, V>(grad_b + gofs + static_cast<size_t>(j) * D, g);
                            store_lanes<St, V>(grad_a + gofs + static_cast<size_t>(j) * D, gav);
                        }
                    }
                };
                // only the sequence's two end windows and windows with a segment
                // start need the state-carrying steps (warp-uniform)
                if (EXT && ((r0bits | r1bits) != 0 || k == 0 || wbase == 0)) rows(std::true_type{});
                else rows(std::false_type{});
            } else {
                for (int j = n - 1; j >= 0; --j) {
                    float x[V], hp[V], go[V], gav[V];
                    unpack_lanes<St, V>(ta + j * DT, x);
                    unpack_lanes<St, V>(th + j * DT, hp);
                    unpack_lanes<St, V>(tg + j * DT, go);
                    if constexpr (EXT) {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            if (j == n - 1) x[v] = 1.0f;  // row T-1 (this is the last window)
                            x[v] = ((r1bits >> j) & 1u) ? 0.0f : x[v];
                            if (j == 0 && wbase == 0) hp[v] = h0v[v];
                        }
                    }
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        g[v] = __fmaf_rn(x[v], g[v], go[v]);
                        gav[v] = __fmul_rn(g[v], hp[v]);
                        if constexpr (EXT) gav[v] = ((r0bits >> j) & 1u) ? 0.0f : gav[v];
                    }
                    if (lane_ok) {
                        store_lanes<St, V>(grad_b + gofs + static_cast<size_t>(j) * D, g);
                        store_lanes<St, V>(grad_a + gofs + static_cast<size_t>(j) * D, gav);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty_bar(stage));
            if (++stage == sm.nstage) { stage = 0; ++use; }
        } else {
        const int rbase = wbase + s * L;
        const int n = min(max(T - rbase, 0), L);
        float xa[L][V], xh[L][V], xg[L][V];
        if (ok) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
                unpack_lanes<St, V>(ta + j * DT, xa[j]);
                unpack_lanes<St, V>(th + j * DT, xh[j]);
                unpack_lanes<St, V>(tg + j * DT, xg[j]);
            }
        }
        // exact tiles release the stage only after the walk has read it
        const int cur = stage;
        if constexpr (!C::EX) {
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
        }
        if (++stage == sm.nstage) { stage = 0; ++use; }
        if constexpr (C::EX && EXT) {
            // the walk takes the rows whose next step starts a segment from here
            if (lg == 0) reinterpret_cast<uint32_t *>(sm.sPQ<C>(0))[s] = r1bits & ((1u << L) - 1u);
        }
        // reverse sub-chunk summary: g at the sub-chunk's first step as
        // P * (g just after the sub-chunk) + Q
        float P[V], Q[V];
#pragma unroll
        for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
        // rows from na on take a' = 1: steps past T (identity steps) and, with
        // the carried state, step T-1 (grad_last enters through a'_T = 1)
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
            // tail sub-chunk: steps past T become exact identity steps (a=1, grad_out=0)
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    xa[j][v] = j < na ? xa[j][v] : 1.0f;
                    xg[j][v] = j < n ? xg[j][v] : 0.0f;
                }
            }
        }
        const int par = C::PT ? (k & 1) : 0;
        float2 *pq = sm.sPQ<C>(par);
        if constexpr (!C::EX) {
#pragma unroll
            for (int j = L - 1; j >= 0; --j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    P[v] = __fmul_rn(xa[j][v], P[v]);
                    Q[v] = __fmaf_rn(xa[j][v], Q[v], xg[j][v]);
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
        }
        if (bar_sync_or(1, NT, !ok)) { failed = true; break; }
        if (issuer && k > 0) {
            // rows of window k-1 are staged and fenced; after issuing its
            // stores, the ones before must have finished reading the buffer
            // window k is about to fill
            ost.store(omaps, k - 1, d0, wbase + sm.W, brow);
            bulk_wait_read<1>();
        }
        if constexpr (C::EX) {
            // lane threads walk the window's rows exactly, last row first,
            // recording the adjoint entering every sub-chunk from above; then
            // the stage is free
            float *entry = sm.sEntry<C>();
            if (static_cast<int>(threadIdx.x) < DT)
                carry = exact_walk<C, true, EXT, EXT>(sm.tile<C>(cur, 0), sm.tile<C>(cur, 2), entry,
                                                      reinterpret_cast<const uint32_t *>(pq), S, threadIdx.x,
                                                      T - wbase, carry);
            bar_sync_or(1, NT, false);
            if (lane == 0) mbar_arrive(sm.empty_bar(cur));
#pragma unroll
            for (int v = 0; v < V; ++v) g[v] = entry[s * DT + v * G + lg];
        } else if constexpr (!C::PT) {
            // lane threads push the carried adjoint through sub-chunks S-1 .. 0
            float *entry = sm.sEntry<C>();
            if (static_cast<int>(threadIdx.x) < DT) carry = lane_walk<true, DT>(pq, entry, S, threadIdx.x, carry);
            bar_sync_or(1, NT, false);
#pragma unroll
            for (int v = 0; v < V; ++v) g[v] = entry[s * DT + v * G + lg];
        } else {
            const float *cs = sm.sCarry<C>(par);
#pragma unroll
            for (int v = 0; v < V; ++v) g[v] = cs[v * G + lg];
#pragma unroll
            for (int ii = 0; ii < C::SMAX - 1; ++ii) {
                const int i = S - 1 - ii;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float2 m = (i > s) ? pq[i * DT + v * G + lg] : make_float2(1.0f, 0.0f);
                    if (i > s) g[v] = __fmaf_rn(m.x, g[v], m.y);
                }
            }
        }
        if constexpr (TS) {
            St *sga = ost.plane(k, 0) + (s * L) * DT + lg * V;
            St *sgb = ost.plane(k, 1) + (s * L) * DT + lg * V;
            if (EXT && r0bits != 0) bwd_rows<C, true, true>(xa, xh, xg, g, n, lane_ok, sgb, sga, D, r0bits);
            else bwd_rows<C, false, true>(xa, xh, xg, g, n, lane_ok, sgb, sga, D, 0u);
            fence_proxy_async_smem();
            replayed = k + 1;
        } else {
            const size_t gofs = (row0 + rbase) * D + d;
            if (EXT && r0bits != 0)
                bwd_rows<C, true, false>(xa, xh, xg, g, n, lane_ok, grad_b + gofs, grad_a + gofs, D, r0bits);
            else bwd_rows<C, false, false>(xa, xh, xg, g, n, lane_ok, grad_b + gofs, grad_a + gofs, D, 0u);
        }
        if (C::PT && s == 0) {
            float *nc = sm.sCarry<C>((k & 1) ^ 1);
#pragma unroll
            for (int v = 0; v < V; ++v) nc[v * G + lg] = g[v];
        }
        if constexpr (EXT) {
            if (rbase == 0 && sx.grad_h0 != nullptr && lane_ok) store_grad_h0<C>(sx, seg, row0, brow, d, D, g);
        }
        }
    }
    if constexpr (EXT && C::SEQ) {
        if (!failed && sx.grad_h0 != nullptr && lane_ok) store_grad_h0<C>(sx, seg, row0, brow, d, D, g);
    }
    if constexpr (TS) {
        // the last window's tiles (not after an abort), then every store
        // complete before the CTA's shared memory goes away
        const bool aborted = bar_sync_or(1, NT, replayed != nwin);
        if (issuer) {
            if (!aborted && replayed > 0) ost.store(omaps, replayed - 1, d0, (nwin - replayed) * sm.W, brow);
            bulk_wait<0>();
        }
    }
    (void)failed;
}

}  // namespace lrscan
