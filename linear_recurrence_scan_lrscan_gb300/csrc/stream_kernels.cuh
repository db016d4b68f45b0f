// Persistent single-pass scan over time chunks, for few lanes and long
// sequences (the chunked decomposition of triton_training_scan.py,
// _real_chunk_summary / _real_chunk_prefix / _real_chunk_replay, with the
// prefix taken by look-back inside the one kernel instead of a phase of its
// own).
//
// Every lane group (batch row x lane tile of DT lanes) is cut in time into
// chunks of NWIN windows of W rows.  A fixed grid of CTAs (one per SM) takes
// chunks from a ticket counter, chunk-major over the groups (forward: earliest
// chunk first; backward: latest first), and passes over each chunk twice:
// once to reduce it to its affine map h -> P h + Q (tiles from HBM), once to
// replay it from its entering state (the same tiles again, from L2).  A CTA's
// warps have one role each:
//   ticket warp     fetches chunk tickets one chunk ahead of the summaries;
//   NW summary      warp w reduces windows w, w + NW, ... of every chunk,
//   warps           streaming its tiles through S stages of its own (S - 1
//                   copies in flight ahead of the tile it reduces); the last
//                   to finish a chunk composes the window maps and publishes
//                   the chunk's map;
//   NSCAN scan      chunk k goes to scan warp k mod NSCAN: it looks back over
//   warps           the chunks before it for the entering state, publishes
//                   the leaving state and hands out each window's entering
//                   state;
//   NW replay       warp w replays the windows its summary twin reduced,
//   warps           through SR stages of its own: each row's result
//                   overwrites the input it consumed in shared memory, and
//                   the window leaves by bulk tensor stores.
// Summaries run ahead of replays by up to NB - 1 chunks (the map and
// entering-state buffers are the only link), so a chunk's map is out as soon
// as its tiles have landed, whatever the replays wait for; NB is kept small
// so that a chunk's tiles are still in L2 when its replay reads them (loads
// for the replay carry an evict-first hint, the summaries' an evict-last one).
//
// HBM carries the scan's own traffic: forward a, b in, out out; backward a,
// out, grad_out in, grad_a, grad_b out.  Results agree with the sequential
// definition to rounding; which published states a look-back composes depends
// on timing, so two calls can differ in the last bits.  The look-back waits
// only on chunks with earlier tickets, which running CTAs hold, so it always
// ends; still every wait is bounded (timeout: LRSCAN_ETIMEOUT in the status
// word, and the kernel returns).
#pragma once

#include "packed_f32x2.cuh"
#include "scan_common.cuh"
#include "state_args.h"
#include "stream_args.h"

namespace lrscan {

enum StreamSite : int { kSiteLookback = 8, kSiteStreamStep = 9 };

__device__ __forceinline__ unsigned int atom_add_acq_rel_cta(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v)
                 : "memory");
    return old;
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


// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// L2 eviction priorities: a summary's tiles are read again by the replay
// (evict last), a replay's tiles and the outputs are not (evict first).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_load_3d with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *m, int x, int y, int z, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// tma_store_3d with an L2 cache policy.
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap *m, uint32_t src, int x, int y, int z,
                                                  uint64_t policy) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::
                     "l"(reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y), "r"(z), "l"(policy)
                 : "memory");
}

// Publication without flags or fences.  The workspace's chunk maps and
// leaving states start filled with kUnset words; a lane publishes its map as
// one 64-bit word (P low, Q high) and its leaving state as one 32-bit word,
// each a single-copy-atomic relaxed store at GPU scope, so a reader that sees
// a word other than kUnset sees the whole value.  A value whose bits are
// kUnset (a NaN) is published as another NaN.
constexpr uint32_t kUnset = 0xffffffffu;

__device__ __forceinline__ uint32_t unset_safe_bits(float x) {
    const uint32_t u = __float_as_uint(x);
    return u == kUnset ? 0x7fffffffu : u;
}
__device__ __forceinline__ void publish_map(float2 *p, float P, float Q) {
    const uint64_t word = (static_cast<uint64_t>(unset_safe_bits(Q)) << 32) | unset_safe_bits(P);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(word) : "memory");
}
__device__ __forceinline__ void publish_state(float *p, float h) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(unset_safe_bits(h)) : "memory");
}
__device__ __forceinline__ uint64_t peek_map(const float2 *p) {
    uint64_t word;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(word) : "l"(p) : "memory");
    return word;
}
__device__ __forceinline__ uint32_t peek_state(const float *p) {
    uint32_t word;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(word) : "l"(p) : "memory");
    return word;
}

// Entering state of chunk `cc` (ticket order within group gi) for lanes
// i0 .. i0+V-1; the whole warp calls it.  Each lane walks back on its own:
// per round it reads the leaving states and maps of its next BATCH chunks (one
// L2 round trip), folds maps in until it meets a published leaving state
// (done) or a chunk with nothing out yet (read again next round).  Maps are
// composed outermost first: h_in = M_cc-1 o M_cc-2 o ... (h_state); chunk -1
// leaves the zero state, or with START the state at h_start[0 .. V-1]
// (carried state: h0 forward, grad_last backward; null: zeros), read only by a
// walk that gets there.  Returns false when the wait expired or the CTA is
// aborting.
template <int DT, int V, int BATCH, bool START = false>
__device__ bool stream_lookback(const StreamArgs &sa, int gi, int cc, int i0, float (&h_in)[V], const WaitCtx &wc,
                                const float *h_start = nullptr) {
    const int lane = threadIdx.x & 31;
    const size_t g0 = static_cast<size_t>(gi) * sa.nc;
    float aP[V], aQ[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { aP[v] = 1.0f; aQ[v] = 0.0f; }
    int j = cc - 1;  // the next chunk this lane folds
    bool done = false;
    uint64_t start = 0;
    bool timed = false;
    for (uint32_t spin = 0;; ++spin) {
        if (!done) {
            uint32_t st[BATCH][V];
            uint64_t mw[BATCH][V];
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                if (j - t >= 0) {
                    const size_t row = (g0 + j - t) * DT + i0;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        st[t][v] = peek_state(sa.incl + row + v);
                        mw[t][v] = peek_map(sa.agg + row + v);
                    }
                }
            }
            bool go = true;
            int folded = 0;
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                if (go) {
                    if (j - t < 0) {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            if constexpr (START)
                                h_in[v] = h_start != nullptr ? __fmaf_rn(aP[v], h_start[v], aQ[v]) : aQ[v];
                            else
                                h_in[v] = aQ[v];  // aP * 0 + aQ
                        }
                        done = true;
                        go = false;
                    } else {
                        bool has_state = true, has_map = true;
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            has_state = has_state && st[t][v] != kUnset;
                            has_map = has_map && static_cast<uint32_t>(mw[t][v]) != kUnset;
                        }
                        if (has_state) {
#pragma unroll
                            for (int v = 0; v < V; ++v) h_in[v] = __fmaf_rn(aP[v], __uint_as_float(st[t][v]), aQ[v]);
                            done = true;
                            go = false;
                        } else if (has_map) {
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                const float P = __uint_as_float(static_cast<uint32_t>(mw[t][v]));
                                const float Q = __uint_as_float(static_cast<uint32_t>(mw[t][v] >> 32));
                                aQ[v] = __fmaf_rn(aP[v], Q, aQ[v]);
                                aP[v] = __fmul_rn(aP[v], P);
                            }
                            ++folded;
                        } else {
                            go = false;  // not out yet: read it again next round
                        }
                    }
                }
            }
            j -= folded;
        }
        if (__all_sync(0xffffffffu, done)) return true;
        if ((spin & 7u) == 7u) {
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
}

// Complex steps in the nested fused multiply-add order of the sequential
// complex scan: x * h + b, and conj(x) * h + b.
__device__ __forceinline__ void cx_step(float xr, float xi, float hr, float hi, float br, float bi, float &nr,
                                        float &ni) {
    nr = __fmaf_rn(xr, hr, __fmaf_rn(-xi, hi, br));
    ni = __fmaf_rn(xi, hr, __fmaf_rn(xr, hi, bi));
}
__device__ __forceinline__ void cxc_step(float xr, float xi, float hr, float hi, float br, float bi, float &nr,
                                         float &ni) {
    nr = __fmaf_rn(xr, hr, __fmaf_rn(xi, hi, br));
    ni = __fmaf_rn(xr, hi, __fmaf_rn(-xi, hr, bi));
}

// Complex look-back: as stream_lookback, for complex maps (two words per lane
// and chunk: P = (re, im), Q = (re, im)) and leaving states (one word).
template <int DT, int V, int BATCH, bool START = false>
__device__ bool stream_lookback_cx(const StreamArgs &sa, int gi, int cc, int i0, float (&hr_in)[V],
                                   float (&hi_in)[V], const WaitCtx &wc, const float *sr = nullptr,
                                   const float *si = nullptr) {
    const int lane = threadIdx.x & 31;
    const size_t g0 = static_cast<size_t>(gi) * sa.nc;
    const float2 *states = reinterpret_cast<const float2 *>(sa.incl);
    float aPr[V], aPi[V], aQr[V], aQi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { aPr[v] = 1.0f; aPi[v] = 0.0f; aQr[v] = 0.0f; aQi[v] = 0.0f; }
    int j = cc - 1;
    bool done = false;
    uint64_t start = 0;
    bool timed = false;
    for (uint32_t spin = 0;; ++spin) {
        if (!done) {
            uint64_t sw[BATCH][V], pw[BATCH][V], qw[BATCH][V];
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                if (j - t >= 0) {
                    const size_t row = (g0 + j - t) * DT + i0;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        sw[t][v] = peek_map(states + row + v);
                        pw[t][v] = peek_map(sa.agg + 2 * (row + v));
                        qw[t][v] = peek_map(sa.agg + 2 * (row + v) + 1);
                    }
                }
            }
            bool go = true;
            int folded = 0;
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                if (go) {
                    if (j - t < 0) {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            if (START && (sr != nullptr || si != nullptr)) {
                                // the chain's start (h0 forward, grad_last backward)
                                cx_step(aPr[v], aPi[v], sr != nullptr ? sr[v] : 0.0f, si != nullptr ? si[v] : 0.0f,
                                        aQr[v], aQi[v], hr_in[v], hi_in[v]);
                            } else {
                                hr_in[v] = aQr[v];
                                hi_in[v] = aQi[v];
                            }
                        }
                        done = true;
                        go = false;
                    } else {
                        bool has_state = true, has_map = true;
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            has_state = has_state && static_cast<uint32_t>(sw[t][v]) != kUnset;
                            has_map = has_map && static_cast<uint32_t>(pw[t][v]) != kUnset &&
                                      static_cast<uint32_t>(qw[t][v]) != kUnset;
                        }
                        if (has_state) {
#pragma unroll
                            for (int v = 0; v < V; ++v)
                                cx_step(aPr[v], aPi[v], __uint_as_float(static_cast<uint32_t>(sw[t][v])),
                                        __uint_as_float(static_cast<uint32_t>(sw[t][v] >> 32)), aQr[v], aQi[v],
                                        hr_in[v], hi_in[v]);
                            done = true;
                            go = false;
                        } else if (has_map) {
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                const float Pr = __uint_as_float(static_cast<uint32_t>(pw[t][v]));
                                const float Pi = __uint_as_float(static_cast<uint32_t>(pw[t][v] >> 32));
                                const float Qr = __uint_as_float(static_cast<uint32_t>(qw[t][v]));
                                const float Qi = __uint_as_float(static_cast<uint32_t>(qw[t][v] >> 32));
                                float nQr, nQi, nPr, nPi;
                                cx_step(aPr[v], aPi[v], Qr, Qi, aQr[v], aQi[v], nQr, nQi);
                                cx_step(aPr[v], aPi[v], Pr, Pi, 0.0f, 0.0f, nPr, nPi);
                                aQr[v] = nQr; aQi[v] = nQi; aPr[v] = nPr; aPi[v] = nPi;
                            }
                            ++folded;
                        } else {
                            go = false;
                        }
                    }
                }
            }
            j -= folded;
        }
        if (__all_sync(0xffffffffu, done)) return true;
        if ((spin & 7u) == 7u) {
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
}

// Compiled shape: storage type, lanes per CTA, lanes per thread, rows per
// window, summary (= replay) warps, windows per warp and chunk, summary and
// replay stages per warp, scan warps, chunk buffers, complex scan (re / im
// planes).
template <class St_, int DT_, int V_, int W_, int NW_, int R_, int S_, int SR_, int NSCAN_, int NB_,
          bool CPLX_ = false>
struct StreamShape {
    using St = St_;
    static constexpr int DT = DT_, V = V_, W = W_, NW = NW_, R = R_, S = S_, SR = SR_, NSCAN = NSCAN_, NB = NB_;
    static constexpr bool CPLX = CPLX_;
    static constexpr int K = CPLX ? 2 : 1;  // floats per value (re, im)
    static constexpr int NWIN = NW * R;     // windows per chunk
    static constexpr int THREADS = (2 * NW + NSCAN + 1) * 32;
    static constexpr int MINB = 1;
    static_assert(DT == 32 * V, "one warp spans a tile row");
    static_assert(W % 8 == 0, "rows are taken eight at a time");
    static_assert(NB % NSCAN == 0, "a scan warp sees every use of its buffers");
    static_assert(S >= 2 && S - 1 <= R, "tiles in flight stay within the next chunk");
    static_assert(SR == 2 || SR == 3, "a replay tile is prefetched one window ahead");
};

constexpr int kStreamSlots = 8;  // ticket ring of the ticket warp

// Tensor maps of one call: inputs in kernel order (real forward a, b;
// backward a, out, grad_out; complex forward ar, ai, br, bi; backward ar, ai,
// out_r, out_i, grad_out_r, grad_out_i), outputs (real forward out; backward
// grad_a, grad_b; complex forward out_r, out_i; backward grad_ar, grad_ai,
// grad_br, grad_bi).
struct StreamMaps {
    CUtensorMap in[6];
    CUtensorMap out[4];
};

// Planes of a direction.  Summary planes: the decay's K parts (backward: one
// row late), then the drive's K parts (forward b, backward grad_out).  Replay
// planes: every input, the decay one row late and out one row early in the
// backward.  Output o is staged over replay plane K + o (forward: over b;
// backward: grad_a over out, grad_b over grad_out).
template <class C, bool BWD>
struct StreamPlanes {
    static constexpr int K = C::K;
    static constexpr int NS = 2 * K;
    static constexpr int NIN = K * (BWD ? 3 : 2);
    static constexpr int NOUT = BWD ? 2 * K : K;
    __device__ static int sum_map(int p) { return p < K ? p : (BWD ? 2 * K + (p - K) : p); }
    __device__ static int sum_dy(int p) { return p < K && BWD ? 1 : 0; }
    __device__ static int rep_dy(int p) { return BWD ? (p < K ? 1 : (p < 2 * K ? -1 : 0)) : 0; }
};

// Shared-memory layout, host and device.  Summary warp w owns stages
// w*S .. w*S+S-1 of the summary ring (NS planes each), replay warp w owns
// stages w*SR .. w*SR+SR-1 of the replay ring (NIN planes each; the outputs
// overwrite their inputs there and leave by bulk tensor stores).
struct StreamGeom {
    int tile_bytes;    // one plane of one window: W * DT * elem
    int sstage_bytes;  // summary stage
    int rstage_bytes;  // replay stage
    int rring_off;     // replay ring after the summary ring
    int bar_off;       // sfull[NW*S], rfull[NW*SR], step_full[slots], step_req[slots], maps[NB], entries[NB],
                       // buf_free[NB], mask_full[slots]
    int ticket_off;    // step tickets [slots]
    int tick_off;      // chunk tickets per buffer [NB] (-1: end mark)
    int map_off;       // window maps [NB][NWIN][DT][2K] floats (P, Q)
    int cmap_off;      // chunk maps [NB][DT][2K] floats
    int entry_off;     // window entering states [NB][NWIN][DT][K] floats
    int mask_off;      // carried-state calls: window reset masks [NB][NWIN][2] (step t, step t+1)
    int tmask_off;     // carried-state calls: per ticket slot, each window's resets [slots][NWIN]
    int count_off;     // summary warps done per buffer [NB]
    int flag_off;      // abort flag
    int smem_bytes;
};

template <class C, bool BWD>
__host__ __device__ inline StreamGeom make_stream_geom() {
    constexpr int K = C::K;
    StreamGeom g{};
    g.tile_bytes = C::W * C::DT * static_cast<int>(sizeof(typename C::St));
    g.sstage_bytes = 2 * K * g.tile_bytes;
    g.rstage_bytes = K * (BWD ? 3 : 2) * g.tile_bytes;
    g.rring_off = C::NW * C::S * g.sstage_bytes;
    g.bar_off = g.rring_off + C::NW * C::SR * g.rstage_bytes;
    const int nbar = C::NW * C::S + C::NW * C::SR + 3 * kStreamSlots + 3 * C::NB;
    g.ticket_off = g.bar_off + nbar * 8;
    g.tick_off = g.ticket_off + kStreamSlots * 4;
    g.map_off = (g.tick_off + C::NB * 4 + 15) / 16 * 16;
    g.cmap_off = g.map_off + C::NB * C::NWIN * C::DT * 8 * K;
    g.entry_off = g.cmap_off + C::NB * C::DT * 8 * K;
    g.mask_off = g.entry_off + C::NB * C::NWIN * C::DT * 4 * K;
    g.tmask_off = g.mask_off + C::NB * C::NWIN * 16;
    g.count_off = g.tmask_off + kStreamSlots * C::NWIN * 8;
    g.flag_off = g.count_off + C::NB * 4;
    g.smem_bytes = g.flag_off + 16;
    return g;
}

// One kernel for both directions and both element kinds (StreamPlanes lists
// the planes).  Outputs overwrite the replay tile planes they were computed
// from and leave by bulk tensor stores; `last` / `last_i` (forward, may be
// NULL) receive the state after the final step.  EXT (real scan): carried
// state and segment resets as in the tiled kernels -- a_t = 0 where
// segment_pos is 0 (backward: a_{t+1} = 0 where step t+1 resets, 1 past the
// end, where grad_last enters), the chain started from h0 (forward) or
// grad_last (backward), out_{-1} = h0 in grad_a, grad_a = +0 at a reset, and
// grad_h0 = a'_0 * g_0 from the window holding step 0.
template <class C, bool BWD, bool EXT = false>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
stream_kernel(const __grid_constant__ StreamMaps tm, float *__restrict__ last, float *__restrict__ last_i, int T,
              int D, DevStatus *status, uint64_t timeout_ns, const __grid_constant__ StreamArgs sa,
              const __grid_constant__ StateArgs sx, const __grid_constant__ CStateArgs cx) {
    using St = typename C::St;
    using PL = StreamPlanes<C, BWD>;
    constexpr int DT = C::DT, V = C::V, W = C::W, NW = C::NW, R = C::R, S = C::S, SR = C::SR, NSCAN = C::NSCAN;
    constexpr int NB = C::NB, K = C::K;
    constexpr int NWIN = C::NWIN;
    constexpr int NS = PL::NS, NIN = PL::NIN, NOUT = PL::NOUT;
    constexpr int SLOTS = kStreamSlots;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const StreamGeom geo = make_stream_geom<C, BWD>();
    auto stile = [&](int st, int plane) {  // summary ring
        return reinterpret_cast<St *>(smem_raw + st * geo.sstage_bytes + plane * geo.tile_bytes);
    };
    auto rtile = [&](int st, int plane) {  // replay ring: planes in tensor-map order
        return reinterpret_cast<St *>(smem_raw + geo.rring_off + st * geo.rstage_bytes + plane * geo.tile_bytes);
    };
    auto bar = [&](int i) { return smem_addr(smem_raw + geo.bar_off + 8 * i); };
    constexpr int BS = NW * S;  // summary-ring barriers first
    auto sfull = [&](int st) { return bar(st); };
    auto rfull = [&](int st) { return bar(BS + st); };
    constexpr int BR = BS + NW * SR;  // then the replay ring's
    auto step_full = [&](int q) { return bar(BR + q); };
    auto step_req = [&](int q) { return bar(BR + SLOTS + q); };
    auto maps_bar = [&](int b) { return bar(BR + 2 * SLOTS + b); };
    auto entries_bar = [&](int b) { return bar(BR + 2 * SLOTS + NB + b); };
    auto buf_free = [&](int b) { return bar(BR + 2 * SLOTS + 2 * NB + b); };
    auto mask_full = [&](int q) { return bar(BR + 2 * SLOTS + 3 * NB + q); };
    int *step_ticket = reinterpret_cast<int *>(smem_raw + geo.ticket_off);
    volatile int *tick_of = reinterpret_cast<volatile int *>(smem_raw + geo.tick_off);
    float *wmap = reinterpret_cast<float *>(smem_raw + geo.map_off);     // [NB][NWIN][DT][2K]
    float *cmap = reinterpret_cast<float *>(smem_raw + geo.cmap_off);    // [NB][DT][2K]
    float *wentry = reinterpret_cast<float *>(smem_raw + geo.entry_off); // [NB][NWIN][DT][K]
    [[maybe_unused]] uint64_t *wmask = reinterpret_cast<uint64_t *>(smem_raw + geo.mask_off);  // [NB][NWIN][2]
    // [slots][NWIN]: bit r = a reset at step r of the window; backward, bit W
    // = one at the step after it
    [[maybe_unused]] uint64_t *tmask = reinterpret_cast<uint64_t *>(smem_raw + geo.tmask_off);
    unsigned int *wcount = reinterpret_cast<unsigned int *>(smem_raw + geo.count_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + geo.flag_off);
    if (threadIdx.x == 0) {
        for (int st = 0; st < BS; ++st) mbar_init(sfull(st), 1);
        for (int st = 0; st < NW * SR; ++st) mbar_init(rfull(st), 1);
        for (int q = 0; q < SLOTS; ++q) {
            mbar_init(step_full(q), 1);
            mbar_init(step_req(q), NW);
            mbar_init(mask_full(q), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(maps_bar(b), 1);  // the last summary warp (or the end mark)
            mbar_init(entries_bar(b), 1);
            mbar_init(buf_free(b), NW);
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
    const int CH = NWIN * W;
    const long long total = static_cast<long long>(sa.ng) * sa.nc;
    // chunk coordinates of ticket t
    struct Chunk {
        int cc, gi, c, brow, x0;
    };
    auto decode = [&](int t) {
        Chunk ch;
        ch.cc = t / sa.ng;
        ch.gi = t - ch.cc * sa.ng;
        ch.c = BWD ? sa.nc - 1 - ch.cc : ch.cc;
        ch.brow = ch.gi / sa.ndt;
        ch.x0 = (ch.gi - ch.brow * sa.ndt) * DT;
        return ch;
    };
    // bounded wait, blind to the abort flag, for a copy this warp issued
    auto drain_one = [&](uint32_t fb, uint32_t par) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(fb, par)) {
            if (global_timer_ns() - t0 > wc.timeout_ns) {
                record_error(wc, kErrTimeout, kSiteDrain);
                break;
            }
        }
    };

    if (warp == 2 * NW + NSCAN) {
        // ------------------------------------------------------------ tickets
        if constexpr (EXT) {
            if ((C::CPLX ? cx.seg : sx.seg) != nullptr) {
                // carried-state calls with resets: the whole warp also turns
                // each ticket's segment positions into its windows' reset
                // masks, published (mask_full) after the ticket itself, about
                // a chunk ahead of the summary that uses them (no global load
                // on the summary warps' path)
                static_assert(W <= 32 && 32 % W == 0 && (NWIN * W) % 32 == 0 && NWIN <= 32,
                              "whole windows per ballot, one window per lane");
                const int32_t *segp = C::CPLX ? cx.seg : sx.seg;
                for (int j = 0;; ++j) {
                    if (j >= 1) {
                        const int m = j - 1;
                        if (!warp_wait(step_req(m % SLOTS), static_cast<uint32_t>((m / SLOTS) & 1), wc,
                                       kSiteProducerEmpty))
                            return;
                    }
                    long long tj = 0;
                    if (lane == 0) tj = static_cast<long long>(atomicAdd(sa.ticket, 1u));
                    tj = __shfl_sync(0xffffffffu, tj, 0);
                    const int tk = tj < total ? static_cast<int>(tj) : -1;
                    if (lane == 0) {
                        step_ticket[j % SLOTS] = tk;
                        mbar_arrive(step_full(j % SLOTS));
                    }
                    if (tk < 0) return;
                    {
                        const Chunk ch = decode(tk);
                        const int32_t *srow = segp + static_cast<size_t>(ch.brow) * T;
                        const int t0 = ch.c * CH;
                        constexpr int NBAL = NWIN * W / 32;  // ballots of 32 rows
                        constexpr int WPB = 32 / W;          // windows per ballot
                        int pos[NBAL];
#pragma unroll
                        for (int i = 0; i < NBAL; ++i) {
                            const int t = t0 + i * 32 + lane;
                            pos[i] = t < T ? __ldg(srow + t) : 1;
                        }
                        uint64_t mine = 0;
#pragma unroll
                        for (int i = 0; i < NBAL; ++i) {
                            const uint32_t m = __ballot_sync(0xffffffffu, pos[i] == 0);
#pragma unroll
                            for (int q = 0; q < WPB; ++q) {
                                const uint32_t mw = W == 32 ? m : ((m >> (q * W)) & ((1u << (W < 32 ? W : 0)) - 1u));
                                if (lane == i * WPB + q) mine = mw;
                            }
                        }
                        if constexpr (BWD) {
                            // bit W: a reset at the step after the window (the
                            // next window's first; after the chunk's last
                            // window, the next chunk's first step)
                            const int te = t0 + CH;
                            const int pe = (lane == 0 && te < T) ? __ldg(srow + te) : 1;
                            const uint64_t eb = __ballot_sync(0xffffffffu, pe == 0) & 1u;
                            const uint64_t nb = __shfl_down_sync(0xffffffffu, mine, 1) & 1u;
                            mine |= (lane == NWIN - 1 ? eb : nb) << W;
                        }
                        if (lane < NWIN) tmask[(j % SLOTS) * NWIN + lane] = mine;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(mask_full(j % SLOTS));
                }
            }
        }
        if (lane == 0) {
            // ticket 0 at once; ticket j >= 1 once every summary warp has asked
            // for it (at the start of its chunk j - 1, request slot (j-1) mod SLOTS)
            for (int j = 0;; ++j) {
                if (j >= 1) {
                    const int m = j - 1;
                    if (!mbar_wait(step_req(m % SLOTS), static_cast<uint32_t>((m / SLOTS) & 1), wc,
                                   kSiteProducerEmpty))
                        return;
                }
                const long long tj = static_cast<long long>(atomicAdd(sa.ticket, 1u));
                const int tk = tj < total ? static_cast<int>(tj) : -1;
                step_ticket[j % SLOTS] = tk;
                mbar_arrive(step_full(j % SLOTS));
                if (tk < 0) return;
            }
        }
        return;
    }

    if (warp < NW) {
        // ------------------------------------------------------ summary warps
        const int w = warp;
        int u_iss = 0, u_done = 0;  // tiles issued / reduced, counted over this warp's chunks (R per chunk)
        auto sissue = [&](int u, int t) {  // lane 0: tile u (window (u % R) * NW + w of ticket t)
            const Chunk ch = decode(t);
            const int st = w * S + u % S;
            const uint32_t fb = sfull(st);
            mbar_arrive_expect_tx(fb, NS * geo.tile_bytes);
            const int y = ch.c * CH + ((u % R) * NW + w) * W;
            const uint64_t keep = l2_evict_last_policy();
#pragma unroll
            for (int p = 0; p < NS; ++p)
                tma_load_3d_hint(smem_addr(stile(st, p)), &tm.in[PL::sum_map(p)], ch.x0, y + PL::sum_dy(p), ch.brow,
                                 fb, keep);
        };
        auto drain = [&]() {
            if (lane != 0) return;
            for (int u = u_done; u < u_iss; ++u) drain_one(sfull(w * S + u % S), static_cast<uint32_t>((u / S) & 1));
        };
        if (!warp_wait(step_full(0), 0u, wc, kSiteStreamStep)) return;
        int tk = step_ticket[0];
        for (int k = 0;; ++k) {
            const int b = k % NB;
            if (tk < 0) {
                // no more chunks: summary warp 0 marks the end in the next NSCAN
                // buffers (each once the replays of its previous chunk are done),
                // so that every scan warp and the replay warps see it
                if (w == 0) {
                    for (int i = 0; i < NSCAN; ++i) {
                        const int ke = k + i, be = ke % NB;
                        if (ke >= NB && !warp_wait(buf_free(be), static_cast<uint32_t>(((ke / NB) - 1) & 1), wc,
                                                   kSiteStreamStep)) {
                            drain();
                            return;
                        }
                        if (lane == 0) {
                            tick_of[be] = -1;
                            mbar_arrive(maps_bar(be));
                        }
                        __syncwarp();
                    }
                }
                drain();
                return;
            }
            // ask for the next ticket now and read it when its first tile is due
            // (a ticket is taken about one chunk before its summary starts, so
            // look-backs rarely wait on a chunk whose CTA has not begun it)
            if (lane == 0) mbar_arrive(step_req(k % SLOTS));
            const int q1 = (k + 1) % SLOTS;
            int tn = -2;  // not read yet
            const Chunk ch = decode(tk);
            // window maps h -> P h + Q: P[r][v][0..K-1], Q[r][v][0..K-1]
            float P[R][V][K], Q[R][V][K];
            // carried-state calls: each window's resets at step t and at step t+1
            [[maybe_unused]] uint64_t mcur[R], mnext[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int u = k * R + r;
                // keep S - 1 tiles in flight ahead of this one (chunks k and k + 1)
                while (u_iss <= u + S - 1) {
                    if (u_iss / R != k && tn == -2) {
                        if (!warp_wait(step_full(q1), static_cast<uint32_t>(((k + 1) / SLOTS) & 1), wc,
                                       kSiteStreamStep)) {
                            drain();
                            return;
                        }
                        tn = step_ticket[q1];
                    }
                    const int t = u_iss / R == k ? tk : tn;
                    if (t < 0) break;
                    if (lane == 0) sissue(u_iss, t);
                    ++u_iss;
                }
                const int wbase = ch.c * CH + (r * NW + w) * W;
                const int nrows = min(max(T - wbase, 0), W);
                const int st = w * S + u % S;
                if (!warp_wait(sfull(st), static_cast<uint32_t>((u / S) & 1), wc, kSiteConsumerFull)) {
                    drain();
                    return;
                }
                // the window's map (rows past T are identity steps)
#pragma unroll
                for (int v = 0; v < V; ++v) {
#pragma unroll
                    for (int q = 0; q < K; ++q) { P[r][v][q] = q == 0 ? 1.0f : 0.0f; Q[r][v][q] = 0.0f; }
                }
                // resets of the decays this window uses (backward: a_{t+1})
                [[maybe_unused]] uint64_t rbits = 0;
                if constexpr (EXT) {
                    uint64_t rc = 0, rn = 0;
                    if ((C::CPLX ? cx.seg : sx.seg) != nullptr) {
                        // the ticket warp's masks for this chunk (its ticket
                        // slot k % SLOTS)
                        if (r == 0 && !warp_wait(mask_full(k % SLOTS), static_cast<uint32_t>((k / SLOTS) & 1), wc,
                                                 kSiteStreamStep)) {
                            drain();
                            return;
                        }
                        const uint64_t full = tmask[(k % SLOTS) * NWIN + r * NW + w];
                        if constexpr (BWD) {
                            rc = full & ((1ull << W) - 1);
                            rn = full >> 1;
                        } else {
                            rc = full;
                        }
                    }
                    mcur[r] = rc;
                    mnext[r] = rn;
                    rbits = BWD ? rn : rc;
                }
                if constexpr (!C::CPLX) {
                    const St *ta = stile(st, 0);
                    const St *tb = stile(st, 1);
                    for (int g8 = 0; g8 < nrows; g8 += 8) {
                        const int r0 = BWD ? ((nrows - 1 - g8) & ~7) : g8;  // groups of eight, chain order
                        float xa[8][V], xb[8][V];
                        load8<St, V, DT>(ta, r0, lane, xa);
                        load8<St, V, DT>(tb, r0, lane, xb);
                        if constexpr (EXT) {
                            // the group's resets (0) and, backward, its row past
                            // the end (a'_T = 1), as selects ahead of the chain
                            const uint32_t m8 = static_cast<uint32_t>(rbits >> r0) & 0xffu;
                            const int pe = BWD ? T - 1 - (wbase + r0) : -1;
                            // warp-uniform: most groups have neither
                            if (m8 != 0u || static_cast<unsigned>(pe) < 8u) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
#pragma unroll
                                    for (int v = 0; v < V; ++v)
                                        xa[q][v] = q == pe ? 1.0f : (((m8 >> q) & 1u) ? 0.0f : xa[q][v]);
                                }
                            }
                        }
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr) {
                            const int row = BWD ? 7 - rr : rr;
                            if (r0 + row < nrows) {
                                if constexpr (V == 2) {
                                    // both lanes in one packed instruction (the
                                    // scalar roundings)
                                    mul_x2(P[r][0][0], P[r][1][0], xa[row][0], xa[row][1], P[r][0][0], P[r][1][0]);
                                    fma_x2(Q[r][0][0], Q[r][1][0], xa[row][0], xa[row][1], Q[r][0][0], Q[r][1][0],
                                           xb[row][0], xb[row][1]);
                                } else {
#pragma unroll
                                    for (int v = 0; v < V; ++v) {
                                        P[r][v][0] = __fmul_rn(xa[row][v], P[r][v][0]);
                                        Q[r][v][0] = __fmaf_rn(xa[row][v], Q[r][v][0], xb[row][v]);
                                    }
                                }
                            }
                        }
                    }
                } else {
                    // complex: planes a_r, a_i, b_r, b_i (backward: conj of a_{t+1}, grad_out)
                    for (int g8 = 0; g8 < nrows; g8 += 8) {
                        const int r0 = BWD ? ((nrows - 1 - g8) & ~7) : g8;
                        float xr[8][V], xi[8][V], br[8][V], bi[8][V];
                        load8<St, V, DT>(stile(st, 0), r0, lane, xr);
                        load8<St, V, DT>(stile(st, 1), r0, lane, xi);
                        load8<St, V, DT>(stile(st, 2), r0, lane, br);
                        load8<St, V, DT>(stile(st, 3), r0, lane, bi);
                        if constexpr (EXT) {
                            // resets (a = 0) and, backward, the row past the end
                            // (a'_T = 1), as selects ahead of the chain
                            const uint32_t m8 = static_cast<uint32_t>(rbits >> r0) & 0xffu;
                            const int pe = BWD ? T - 1 - (wbase + r0) : -1;
                            if (m8 != 0u || static_cast<unsigned>(pe) < 8u) {  // warp-uniform
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const bool z = (m8 >> q) & 1u;
#pragma unroll
                                    for (int v = 0; v < V; ++v) {
                                        xr[q][v] = q == pe ? 1.0f : (z ? 0.0f : xr[q][v]);
                                        xi[q][v] = q == pe ? 0.0f : (z ? 0.0f : xi[q][v]);
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr) {
                            const int row = BWD ? 7 - rr : rr;
                            if (r0 + row < nrows) {
#pragma unroll
                                for (int v = 0; v < V; ++v) {
                                    float nPr, nPi, nQr, nQi;
                                    if constexpr (BWD) {
                                        cxc_step(xr[row][v], xi[row][v], P[r][v][0], P[r][v][1], 0.0f, 0.0f, nPr, nPi);
                                        cxc_step(xr[row][v], xi[row][v], Q[r][v][0], Q[r][v][1], br[row][v],
                                                 bi[row][v], nQr, nQi);
                                    } else {
                                        cx_step(xr[row][v], xi[row][v], P[r][v][0], P[r][v][1], 0.0f, 0.0f, nPr, nPi);
                                        cx_step(xr[row][v], xi[row][v], Q[r][v][0], Q[r][v][1], br[row][v],
                                                bi[row][v], nQr, nQi);
                                    }
                                    P[r][v][0] = nPr; P[r][v][1] = nPi; Q[r][v][0] = nQr; Q[r][v][1] = nQi;
                                }
                            }
                        }
                    }
                }
                __syncwarp();  // every lane done with the stage before it is refilled
                ++u_done;
            }
            // buffer b is free once the replays of chunk k - NB are done
            if (k >= NB && !warp_wait(buf_free(b), static_cast<uint32_t>(((k / NB) - 1) & 1), wc, kSiteStreamStep)) {
                drain();
                return;
            }
            if constexpr (EXT) {
                if (lane == 0) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        wmask[(b * NWIN + r * NW + w) * 2] = mcur[r];
                        wmask[(b * NWIN + r * NW + w) * 2 + 1] = mnext[r];
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float *mp = wmap + ((b * NWIN + r * NW + w) * DT + lane * V) * 2 * K;
#pragma unroll
                for (int v = 0; v < V; ++v) {
#pragma unroll
                    for (int q = 0; q < K; ++q) {
                        mp[v * 2 * K + q] = P[r][v][q];
                        mp[v * 2 * K + K + q] = Q[r][v][q];
                    }
                }
            }
            __syncwarp();
            unsigned int before = 0;
            if (lane == 0) before = atom_add_acq_rel_cta(wcount + b, 1u);
            before = __shfl_sync(0xffffffffu, before, 0);
            if (before == NW - 1) {
                // the last summary warp of this chunk: compose the window maps in
                // chain order and publish the chunk's map at once
                __syncwarp();
                const float *cm = wmap + b * NWIN * DT * 2 * K;
                float Pc[V][K], Qc[V][K];
#pragma unroll
                for (int v = 0; v < V; ++v) {
#pragma unroll
                    for (int q = 0; q < K; ++q) { Pc[v][q] = q == 0 ? 1.0f : 0.0f; Qc[v][q] = 0.0f; }
                }
                for (int jw = 0; jw < NWIN; ++jw) {
                    const int ww = BWD ? NWIN - 1 - jw : jw;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float *m = cm + (ww * DT + lane * V + v) * 2 * K;
                        if constexpr (!C::CPLX) {
                            Qc[v][0] = __fmaf_rn(m[0], Qc[v][0], m[1]);
                            Pc[v][0] = __fmul_rn(m[0], Pc[v][0]);
                        } else {
                            float nQr, nQi, nPr, nPi;
                            cx_step(m[0], m[1], Qc[v][0], Qc[v][1], m[2], m[3], nQr, nQi);
                            cx_step(m[0], m[1], Pc[v][0], Pc[v][1], 0.0f, 0.0f, nPr, nPi);
                            Qc[v][0] = nQr; Qc[v][1] = nQi; Pc[v][0] = nPr; Pc[v][1] = nPi;
                        }
                    }
                }
                const size_t slot_g = static_cast<size_t>(ch.gi) * sa.nc + ch.cc;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    float *cp = cmap + (b * DT + lane * V + v) * 2 * K;
#pragma unroll
                    for (int q = 0; q < K; ++q) { cp[q] = Pc[v][q]; cp[K + q] = Qc[v][q]; }
                    const size_t gidx = slot_g * DT + lane * V + v;
                    if constexpr (!C::CPLX) {
                        publish_map(sa.agg + gidx, Pc[v][0], Qc[v][0]);
                    } else {
                        publish_map(sa.agg + 2 * gidx, Pc[v][0], Pc[v][1]);
                        publish_map(sa.agg + 2 * gidx + 1, Qc[v][0], Qc[v][1]);
                    }
                }
                __syncwarp();  // every lane's cmap entries written before the maps_ready arrive
                if (lane == 0) {
                    tick_of[b] = tk;
                    wcount[b] = 0;  // next used NB chunks on, after this buffer's replays
                    mbar_arrive(maps_bar(b));
                }
            }
            if (tn == -2) {
                if (!warp_wait(step_full(q1), static_cast<uint32_t>(((k + 1) / SLOTS) & 1), wc, kSiteStreamStep)) {
                    drain();
                    return;
                }
                tn = step_ticket[q1];
            }
            tk = tn;
        }
    }

    if (warp >= 2 * NW) {
        // --------------------------------------------------------- scan warps
        // scan warp j takes chunks j, j + NSCAN, ... until an end mark
        const int i0 = lane * V;
        for (int k = warp - 2 * NW;; k += NSCAN) {
            const int b = k % NB;
            if (!warp_wait(maps_bar(b), static_cast<uint32_t>((k / NB) & 1), wc, kSiteStreamStep)) return;
            const int t = tick_of[b];
            if (t < 0) return;
            const Chunk ch = decode(t);
            float h[V][K];
            const size_t slot_g = static_cast<size_t>(ch.gi) * sa.nc + ch.cc;
            if constexpr (!C::CPLX) {
                float hin[V];
                // the chain's start: h0 forward, grad_last backward (lanes past D
                // read none: their results are clipped)
                const float *st0 = nullptr;
                if constexpr (EXT) {
                    const float *s0 = BWD ? sx.grad_last : sx.h0;
                    if (s0 != nullptr && ch.x0 + i0 < D) st0 = s0 + static_cast<size_t>(ch.brow) * D + ch.x0 + i0;
                }
                if (!stream_lookback<DT, V, 16 / V, EXT>(sa, ch.gi, ch.cc, i0, hin, wc, st0)) return;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float *cp = cmap + (b * DT + i0 + v) * 2;
                    h[v][0] = hin[v];
                    publish_state(sa.incl + slot_g * DT + i0 + v, __fmaf_rn(cp[0], hin[v], cp[1]));
                }
            } else {
                float hr[V], hi[V];
                // the chain's start: complex h0 forward, grad_last backward
                const float *sr0 = nullptr, *si0 = nullptr;
                if constexpr (EXT) {
                    if (ch.x0 + i0 < D) {
                        const size_t o0 = static_cast<size_t>(ch.brow) * D + ch.x0 + i0;
                        const float *r0p = BWD ? cx.gl_r : cx.h0_r;
                        const float *i0p = BWD ? cx.gl_i : cx.h0_i;
                        sr0 = r0p != nullptr ? r0p + o0 : nullptr;
                        si0 = i0p != nullptr ? i0p + o0 : nullptr;
                    }
                }
                if (!stream_lookback_cx<DT, V, 8 / V, EXT>(sa, ch.gi, ch.cc, i0, hr, hi, wc, sr0, si0)) return;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float *cp = cmap + (b * DT + i0 + v) * 4;
                    float lr, li;
                    cx_step(cp[0], cp[1], hr[v], hi[v], cp[2], cp[3], lr, li);
                    publish_map(reinterpret_cast<float2 *>(sa.incl) + slot_g * DT + i0 + v, lr, li);
                    h[v][0] = hr[v];
                    h[v][1] = hi[v];
                }
            }
            // the state entering every window, in chain order
            const float *mp = wmap + b * NWIN * DT * 2 * K;
            float *ep = wentry + b * NWIN * DT * K;
            for (int jw = 0; jw < NWIN; ++jw) {
                const int ww = BWD ? NWIN - 1 - jw : jw;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float *m = mp + (ww * DT + i0 + v) * 2 * K;
                    float *e = ep + (ww * DT + i0 + v) * K;
#pragma unroll
                    for (int q = 0; q < K; ++q) e[q] = h[v][q];
                    if constexpr (!C::CPLX) {
                        h[v][0] = __fmaf_rn(m[0], h[v][0], m[1]);
                    } else {
                        float nr, ni;
                        cx_step(m[0], m[1], h[v][0], h[v][1], m[2], m[3], nr, ni);
                        h[v][0] = nr;
                        h[v][1] = ni;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(entries_bar(b));
        }
    }

    // ------------------------------------------------------------ replay warps
    const int w = warp - NW;
    const uint64_t drop = l2_evict_first_policy();  // replay tiles and outputs: not read again here
    int u_iss = 0, u_done = 0;  // tiles issued / replayed, counted over this warp's chunks (R per chunk)
    auto rissue = [&](int u, int t) {  // lane 0: tile u (window (u % R) * NW + w of ticket t)
        // the stage last held tile u - SR, whose outputs were committed SR - 2
        // bulk groups before the newest: wait until they have left it
        bulk_wait_read<SR - 2>();
        const Chunk ch = decode(t);
        const int st = w * SR + u % SR;
        const uint32_t fb = rfull(st);
        mbar_arrive_expect_tx(fb, NIN * geo.tile_bytes);
        const int y = ch.c * CH + ((u % R) * NW + w) * W;
#pragma unroll
        for (int p = 0; p < NIN; ++p)
            tma_load_3d_hint(smem_addr(rtile(st, p)), &tm.in[p], ch.x0, y + PL::rep_dy(p), ch.brow, fb, drop);
    };
    auto drain = [&]() {
        if (lane != 0) return;
        for (int u = u_done; u < u_iss; ++u) drain_one(rfull(w * SR + u % SR), static_cast<uint32_t>((u / SR) & 1));
        bulk_wait<0>();  // the outputs in flight have left shared memory and landed
    };
    for (int k = 0;; ++k) {
        const int b = k % NB;
        if (!warp_wait(maps_bar(b), static_cast<uint32_t>((k / NB) & 1), wc, kSiteStreamStep)) {
            drain();
            return;
        }
        const int t = tick_of[b];
        if (t < 0) {
            drain();
            return;
        }
        const Chunk ch = decode(t);
        const int d = ch.x0 + lane * V;
        for (int r = 0; r < R; ++r) {
            const int u = k * R + r;
            if (u_iss == u) {  // not prefetched
                if (lane == 0) rissue(u, t);
                ++u_iss;
            }
            // the next tile into the next stage; past this chunk only if the
            // next chunk's map is already out
            if (u_iss == u + 1) {
                if (r + 1 < R) {
                    if (lane == 0) rissue(u + 1, t);
                    ++u_iss;
                } else {
                    int did = 0;
                    if (lane == 0) {
                        const int b1 = (k + 1) % NB;
                        if (mbar_test_wait(maps_bar(b1), static_cast<uint32_t>(((k + 1) / NB) & 1))) {
                            const int t1 = tick_of[b1];
                            if (t1 >= 0) {
                                rissue(u + 1, t1);
                                did = 1;
                            }
                        }
                    }
                    u_iss += __shfl_sync(0xffffffffu, did, 0);
                }
            }
            if (r == 0 && !warp_wait(entries_bar(b), static_cast<uint32_t>((k / NB) & 1), wc, kSiteStreamStep)) {
                drain();
                return;
            }
            const int st = w * SR + u % SR;
            if (!warp_wait(rfull(st), static_cast<uint32_t>((u / SR) & 1), wc, kSiteConsumerFull)) {
                drain();
                return;
            }
            const int wi = r * NW + w;
            const int wbase = ch.c * CH + wi * W;
            const int nrows = min(max(T - wbase, 0), W);
            float h[V][K];
            const float *ep = wentry + ((b * NWIN + wi) * DT + lane * V) * K;
#pragma unroll
            for (int v = 0; v < V; ++v) {
#pragma unroll
                for (int q = 0; q < K; ++q) h[v][q] = ep[v * K + q];
            }
            if constexpr (!C::CPLX && !BWD) {
                // out_t over b_t in the tile (each lane rewrites what it read)
                St *ta = rtile(st, 0);
                St *tb = rtile(st, 1);
                [[maybe_unused]] uint64_t rbits = 0;
                if constexpr (EXT) rbits = wmask[(b * NWIN + wi) * 2];
                for (int g8 = 0; g8 < nrows; g8 += 8) {
                    float xa[8][V], xb[8][V];
                    load8<St, V, DT>(ta, g8, lane, xa);
                    load8<St, V, DT>(tb, g8, lane, xb);
                    if constexpr (EXT) {
                        const uint32_t m8 = static_cast<uint32_t>(rbits >> g8) & 0xffu;
                        if (m8 != 0u) {  // warp-uniform
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
#pragma unroll
                                for (int v = 0; v < V; ++v) xa[q][v] = ((m8 >> q) & 1u) ? 0.0f : xa[q][v];
                            }
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        if (g8 + rr < nrows) {
                            float hv[V];
                            if constexpr (V == 2) {
                                fma_x2(h[0][0], h[1][0], xa[rr][0], xa[rr][1], h[0][0], h[1][0], xb[rr][0], xb[rr][1]);
                                hv[0] = h[0][0];
                                hv[1] = h[1][0];
                            } else {
#pragma unroll
                                for (int v = 0; v < V; ++v) hv[v] = h[v][0] = __fmaf_rn(xa[rr][v], h[v][0], xb[rr][v]);
                            }
                            store_lanes<St, V>(tb + (g8 + rr) * DT + lane * V, hv);
                        }
                    }
                }
            } else if constexpr (!C::CPLX) {
                // grad_b_t over grad_out_t, grad_a_t over h_{t-1}
                St *ta = rtile(st, 0);
                St *th = rtile(st, 1);
                St *tb = rtile(st, 2);
                // EXT: resets of a_{t+1} (rnext) and of step t itself (rcur), and
                // out_{-1} = h0
                [[maybe_unused]] uint64_t rnext = 0, rcur = 0;
                [[maybe_unused]] float h0v[V];
                if constexpr (EXT) {
                    rcur = wmask[(b * NWIN + wi) * 2];
                    rnext = wmask[(b * NWIN + wi) * 2 + 1];
#pragma unroll
                    for (int v = 0; v < V; ++v)  // out_{-1} = h0: read by the window holding step 0 only
                        h0v[v] = (wbase == 0 && sx.h0 != nullptr && d + v < D)
                                     ? sx.h0[static_cast<size_t>(ch.brow) * D + d + v]
                                     : 0.0f;
                }
                for (int g8 = 0; g8 < nrows; g8 += 8) {
                    const int r0 = (nrows - 1 - g8) & ~7;
                    float xa[8][V], xh[8][V], xg[8][V];
                    load8<St, V, DT>(ta, r0, lane, xa);
                    load8<St, V, DT>(th, r0, lane, xh);
                    load8<St, V, DT>(tb, r0, lane, xg);
                    [[maybe_unused]] uint32_t zmask = 0;  // rows whose grad_a is +0 (resets)
                    if constexpr (EXT) {
                        // the group's resets of a_{t+1} (0), the row past the end
                        // (a'_T = 1: grad_last enters there), out_{-1} = h0, as
                        // selects ahead of the chain
                        const uint32_t mn = static_cast<uint32_t>(rnext >> r0) & 0xffu;
                        zmask = static_cast<uint32_t>(rcur >> r0) & 0xffu;
                        const int pe = T - 1 - (wbase + r0);
                        if (mn != 0u || static_cast<unsigned>(pe) < 8u) {  // warp-uniform
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
#pragma unroll
                                for (int v = 0; v < V; ++v)
                                    xa[q][v] = q == pe ? 1.0f : (((mn >> q) & 1u) ? 0.0f : xa[q][v]);
                            }
                        }
                        if (wbase + r0 == 0) {
#pragma unroll
                            for (int v = 0; v < V; ++v) xh[0][v] = h0v[v];
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int row = 7 - rr;
                        if (r0 + row < nrows) {
                            float gv[V], gav[V];
                            if constexpr (V == 2) {
                                fma_x2(h[0][0], h[1][0], xa[row][0], xa[row][1], h[0][0], h[1][0], xg[row][0],
                                       xg[row][1]);
                                mul_x2(gav[0], gav[1], h[0][0], h[1][0], xh[row][0], xh[row][1]);
                                gv[0] = h[0][0];
                                gv[1] = h[1][0];
                            } else {
#pragma unroll
                                for (int v = 0; v < V; ++v) {
                                    gv[v] = h[v][0] = __fmaf_rn(xa[row][v], h[v][0], xg[row][v]);
                                    gav[v] = __fmul_rn(h[v][0], xh[row][v]);
                                }
                            }
                            if constexpr (EXT) {
#pragma unroll
                                for (int v = 0; v < V; ++v) gav[v] = ((zmask >> row) & 1u) ? 0.0f : gav[v];
                            }
                            store_lanes<St, V>(tb + (r0 + row) * DT + lane * V, gv);
                            store_lanes<St, V>(th + (r0 + row) * DT + lane * V, gav);
                        }
                    }
                }
                if constexpr (EXT) {
                    // grad_h0 = a'_0 * g_0 from the window holding step 0 (h holds g_0)
                    if (sx.grad_h0 != nullptr && wbase == 0 && d < D) {
                        float a0[V];
                        unpack_lanes<St, V>(static_cast<const St *>(sx.a) + static_cast<size_t>(ch.brow) * T * D + d,
                                            a0);
#pragma unroll
                        for (int v = 0; v < V; ++v)
                            sx.grad_h0[static_cast<size_t>(ch.brow) * D + d + v] =
                                (rcur & 1) ? 0.0f : __fmul_rn(a0[v], h[v][0]);
                    }
                }
            } else if constexpr (!BWD) {
                // complex: out_t over b_t (planes 2, 3)
                [[maybe_unused]] uint64_t rbits = 0;
                if constexpr (EXT) rbits = wmask[(b * NWIN + wi) * 2];
                for (int g8 = 0; g8 < nrows; g8 += 8) {
                    float xr[8][V], xi[8][V], br[8][V], bi[8][V];
                    load8<St, V, DT>(rtile(st, 0), g8, lane, xr);
                    load8<St, V, DT>(rtile(st, 1), g8, lane, xi);
                    load8<St, V, DT>(rtile(st, 2), g8, lane, br);
                    load8<St, V, DT>(rtile(st, 3), g8, lane, bi);
                    if constexpr (EXT) {
                        const uint32_t m8 = static_cast<uint32_t>(rbits >> g8) & 0xffu;
                        if (m8 != 0u) {  // warp-uniform
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const bool z = (m8 >> q) & 1u;
#pragma unroll
                                for (int v = 0; v < V; ++v) {
                                    xr[q][v] = z ? 0.0f : xr[q][v];
                                    xi[q][v] = z ? 0.0f : xi[q][v];
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        if (g8 + rr < nrows) {
                            float or_[V], oi[V];
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                cx_step(xr[rr][v], xi[rr][v], h[v][0], h[v][1], br[rr][v], bi[rr][v], or_[v], oi[v]);
                                h[v][0] = or_[v];
                                h[v][1] = oi[v];
                            }
                            store_lanes<St, V>(rtile(st, 2) + (g8 + rr) * DT + lane * V, or_);
                            store_lanes<St, V>(rtile(st, 3) + (g8 + rr) * DT + lane * V, oi);
                        }
                    }
                }
            } else {
                // complex backward: g = conj(a_{t+1}) g + grad_out; grad_b = g over
                // grad_out (planes 4, 5), grad_a = g conj(h_{t-1}) over out (2, 3)
                // EXT: resets of a_{t+1} (rnext) and of step t itself (rcur), and
                // out_{-1} = h0
                [[maybe_unused]] uint64_t rnext = 0, rcur = 0;
                [[maybe_unused]] float h0r[V], h0i[V];
                if constexpr (EXT) {
                    rcur = wmask[(b * NWIN + wi) * 2];
                    rnext = wmask[(b * NWIN + wi) * 2 + 1];
                    const size_t hs = static_cast<size_t>(ch.brow) * D + d;
#pragma unroll
                    for (int v = 0; v < V; ++v) {  // read by the window holding step 0 only
                        const bool in0 = wbase == 0 && d + v < D;
                        h0r[v] = (in0 && cx.h0_r != nullptr) ? cx.h0_r[hs + v] : 0.0f;
                        h0i[v] = (in0 && cx.h0_i != nullptr) ? cx.h0_i[hs + v] : 0.0f;
                    }
                }
                for (int g8 = 0; g8 < nrows; g8 += 8) {
                    const int r0 = (nrows - 1 - g8) & ~7;
                    float xr[8][V], xi[8][V], hr[8][V], hi[8][V], gr[8][V], gi[8][V];
                    load8<St, V, DT>(rtile(st, 0), r0, lane, xr);
                    load8<St, V, DT>(rtile(st, 1), r0, lane, xi);
                    load8<St, V, DT>(rtile(st, 2), r0, lane, hr);
                    load8<St, V, DT>(rtile(st, 3), r0, lane, hi);
                    load8<St, V, DT>(rtile(st, 4), r0, lane, gr);
                    load8<St, V, DT>(rtile(st, 5), r0, lane, gi);
                    [[maybe_unused]] uint32_t zmask = 0;  // rows whose grad_a is +0 (resets)
                    if constexpr (EXT) {
                        // conj(a'_{t+1}): 0 where step t+1 starts a segment, 1 at
                        // the row past the end (grad_last enters there);
                        // out_{-1} = h0
                        const uint32_t mn = static_cast<uint32_t>(rnext >> r0) & 0xffu;
                        zmask = static_cast<uint32_t>(rcur >> r0) & 0xffu;
                        const int pe = T - 1 - (wbase + r0);
                        if (mn != 0u || static_cast<unsigned>(pe) < 8u) {  // warp-uniform
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const bool z = (mn >> q) & 1u;
#pragma unroll
                                for (int v = 0; v < V; ++v) {
                                    xr[q][v] = q == pe ? 1.0f : (z ? 0.0f : xr[q][v]);
                                    xi[q][v] = q == pe ? 0.0f : (z ? 0.0f : xi[q][v]);
                                }
                            }
                        }
                        if (wbase + r0 == 0) {
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                hr[0][v] = h0r[v];
                                hi[0][v] = h0i[v];
                            }
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int row = 7 - rr;
                        if (r0 + row < nrows) {
                            float ngr[V], ngi[V], gar[V], gai[V];
#pragma unroll
                            for (int v = 0; v < V; ++v) {
                                cxc_step(xr[row][v], xi[row][v], h[v][0], h[v][1], gr[row][v], gi[row][v], ngr[v],
                                         ngi[v]);
                                h[v][0] = ngr[v];
                                h[v][1] = ngi[v];
                                // g * conj(h_{t-1}); +0 where step t starts a segment
                                gar[v] = __fmaf_rn(ngr[v], hr[row][v], __fmul_rn(ngi[v], hi[row][v]));
                                gai[v] = __fmaf_rn(ngi[v], hr[row][v], -__fmul_rn(ngr[v], hi[row][v]));
                                if constexpr (EXT) {
                                    const bool z = (zmask >> row) & 1u;
                                    gar[v] = z ? 0.0f : gar[v];
                                    gai[v] = z ? 0.0f : gai[v];
                                }
                            }
                            const int o = (r0 + row) * DT + lane * V;
                            store_lanes<St, V>(rtile(st, 4) + o, ngr);
                            store_lanes<St, V>(rtile(st, 5) + o, ngi);
                            store_lanes<St, V>(rtile(st, 2) + o, gar);
                            store_lanes<St, V>(rtile(st, 3) + o, gai);
                        }
                    }
                }
                if constexpr (EXT) {
                    // grad_h0 = conj(a'_0) * g_0 from the window holding step 0
                    // (h holds g_0), +0 where step 0 starts a segment
                    if ((cx.gh0_r != nullptr || cx.gh0_i != nullptr) && wbase == 0 && d < D) {
                        const size_t ao = static_cast<size_t>(ch.brow) * T * D + d;
                        float ar0[V], ai0[V];
                        unpack_lanes<St, V>(static_cast<const St *>(cx.ar) + ao, ar0);
                        unpack_lanes<St, V>(static_cast<const St *>(cx.ai) + ao, ai0);
                        const size_t hs = static_cast<size_t>(ch.brow) * D + d;
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const bool z = rcur & 1;
                            const float gr0 = z ? 0.0f : __fmaf_rn(ar0[v], h[v][0], __fmul_rn(ai0[v], h[v][1]));
                            const float gi0 = z ? 0.0f : __fmaf_rn(ar0[v], h[v][1], -__fmul_rn(ai0[v], h[v][0]));
                            if (cx.gh0_r != nullptr) cx.gh0_r[hs + v] = gr0;
                            if (cx.gh0_i != nullptr) cx.gh0_i[hs + v] = gi0;
                        }
                    }
                }
            }
            if constexpr (!BWD) {
                if (last != nullptr && d < D && nrows > 0 && wbase + nrows == T) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        last[static_cast<size_t>(ch.brow) * D + d + v] = h[v][0];
                        if constexpr (C::CPLX) last_i[static_cast<size_t>(ch.brow) * D + d + v] = h[v][1];
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int o = 0; o < NOUT; ++o)
                    tma_store_3d_hint(&tm.out[o], smem_addr(rtile(st, K + o)), ch.x0, wbase, ch.brow, drop);
                bulk_commit();
            }
            __syncwarp();  // every lane done with the stage before it is refilled
            ++u_done;
        }
        if (lane == 0) mbar_arrive(buf_free(b));  // the buffer's entering states are read
    }
}

}  // namespace lrscan
