// Complex diagonal scan on separate real / imaginary planes
// (triton_training_scan.py, _complex_forward / _complex_backward):
//
//   forward   h_t = a_t * h_{t-1} + b_t               (complex, h_{-1} = 0)
//   backward  g_t = go_t + conj(a_{t+1}) * g_{t+1},  grad_b = g,
//             grad_a = g * conj(h_{t-1})
//
// with each component two nested fused multiply-adds (the oracle's order):
//   h_r = fma(ar, h_r, fma(-ai, h_i, br)),   h_i = fma(ai, h_r, fma(ar, h_i, bi))
//   g_r = fma(ar', g_r, fma(ai', g_i, go_r)), g_i = fma(ar', g_i, fma(-ai', g_r, go_i))
//   grad_ar = fma(g_r, p_r, g_i*p_i),        grad_ai = fma(g_i, p_r, -(g_r*p_i))
//
// The tiled kernels are the sequential (S = 1) form of the time-tiled scan:
// a producer warp streams NIN planes per window into the shared-memory stage
// ring with bulk tensor copies (4 forward: ar, ai, br, bi; 6 backward: ar and
// ai one row late, out_r and out_i one row early, go_r, go_i, so that the
// copies' zero fill gives a_T = 0 and h_{-1} = 0), and every consumer thread
// walks its V lanes through all windows in registers.  Full windows are
// taken CH rows at a time: the CH rows of every plane are copied from shared
// memory into registers first, so all those loads issue before the dependent
// chain (and before the chunk's global stores, which the compiler cannot
// reorder them across).
//
// EXT instantiations add the carried state and segment resets (CStateArgs,
// triton_training_scan.py, _samu_tiled_serial_forward / _backward): the
// forward starts from h0 and zeroes a_t where a segment starts; the backward
// starts from grad_last (entering step T-1 through a'_T = 1), zeroes
// conj(a'_{t+1}) where step t+1 starts a segment, writes grad_a = +0 where
// step t starts one, reads h0 as h_{-1} and writes grad_h0 = conj(a'_0) g_0.
// Each warp turns the segment positions of its rows into bit masks with one
// ballot per window (loaded one window ahead).  EXT = false compiles all of
// it out.
#pragma once

#include "window_kernels.cuh"

namespace lrscan {

template <class C, int CH, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
cwin_fwd_kernel(const __grid_constant__ CUtensorMap tm_ar, const __grid_constant__ CUtensorMap tm_ai,
                const __grid_constant__ CUtensorMap tm_br, const __grid_constant__ CUtensorMap tm_bi,
                typename C::St *__restrict__ out_r, typename C::St *__restrict__ out_i,
                float *__restrict__ last_r, float *__restrict__ last_i, const __grid_constant__ WinGeom geom,
                DevStatus *status, uint64_t timeout_ns, const __grid_constant__ CStateArgs sx) {
    static_assert(C::SEQ && C::NIN == 4, "complex forward: sequential shape, four input planes");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int NT = G;
    win_init<C>(sm, NT / 32, 1);
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D;

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[4] = {&tm_ar, &tm_ai, &tm_br, &tm_bi};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow, [W](int k, int) { return k * W; }, wc);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int d = d0 + threadIdx.x * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    float hr[V], hi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) hr[v] = hi[v] = 0.0f;
    bool failed = false;
    int stage = 0, use = 0;
    const int off = threadIdx.x * V;
    // EXT: bit j of rbits is a reset at row j of the current window (lane l
    // holds the position of row l, one window ahead)
    static_assert(!EXT || L <= 32, "one ballot covers a window's rows");
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    int32_t pos_next = 1;
    if constexpr (EXT) {
        if (lane_ok) {
            const size_t hs = static_cast<size_t>(brow) * D + d;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                hr[v] = sx.h0_r != nullptr ? sx.h0_r[hs + v] : 0.0f;
                hi[v] = sx.h0_i != nullptr ? sx.h0_i[hs + v] : 0.0f;
            }
        }
        pos_next = seg.at(lane < L ? lane : -1);
    }
    for (int k = 0; k < sm.nwin; ++k) {
        uint32_t rbits = 0;
        if constexpr (EXT) {
            rbits = __ballot_sync(0xffffffffu, pos_next == 0);
            pos_next = seg.at(lane < L ? (k + 1) * sm.W + lane : -1);
        }
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if constexpr (EXT) ok = __all_sync(0xffffffffu, ok);  // keep the warp's ballots converged
        if (!ok) { failed = true; break; }
        const St *tar = sm.tile<C>(stage, 0) + off;
        const St *tai = sm.tile<C>(stage, 1) + off;
        const St *tbr = sm.tile<C>(stage, 2) + off;
        const St *tbi = sm.tile<C>(stage, 3) + off;
        const int rbase = k * sm.W;
        const int n = min(T - rbase, L);
        const size_t o = (row0 + rbase) * D + d;
        // MASK: a'_t = 0 on the window's reset rows (warp-uniform choice)
        auto compute = [&](int j, float (&xr)[V], float (&xi)[V], const float (&yr)[V], const float (&yi)[V],
                           bool masked) {
            if (EXT && masked) {
                if ((rbits >> j) & 1u) {
#pragma unroll
                    for (int v = 0; v < V; ++v) xr[v] = xi[v] = 0.0f;
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float nr = __fmaf_rn(xr[v], hr[v], __fmaf_rn(-xi[v], hi[v], yr[v]));
                const float ni = __fmaf_rn(xi[v], hr[v], __fmaf_rn(xr[v], hi[v], yi[v]));
                hr[v] = nr;
                hi[v] = ni;
            }
            if (lane_ok) {
                store_lanes<St, V>(out_r + o + static_cast<size_t>(j) * D, hr);
                store_lanes<St, V>(out_i + o + static_cast<size_t>(j) * D, hi);
            }
        };
        auto rows = [&](bool masked) {
            if (n == L) {
                using Raw = typename RawOf<St, V>::T;
#pragma unroll
                for (int j0 = 0; j0 < L; j0 += CH) {
                    Raw r0[CH], r1[CH], r2[CH], r3[CH];
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        r0[j] = load_raw<St, V>(tar + (j0 + j) * DT);
                        r1[j] = load_raw<St, V>(tai + (j0 + j) * DT);
                        r2[j] = load_raw<St, V>(tbr + (j0 + j) * DT);
                        r3[j] = load_raw<St, V>(tbi + (j0 + j) * DT);
                    }
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        float xr[V], xi[V], yr[V], yi[V];
                        widen_raw(r0[j], xr);
                        widen_raw(r1[j], xi);
                        widen_raw(r2[j], yr);
                        widen_raw(r3[j], yi);
                        compute(j0 + j, xr, xi, yr, yi, masked);
                    }
                }
            } else {
                for (int j = 0; j < n; ++j) {
                    float xr[V], xi[V], yr[V], yi[V];
                    unpack_lanes<St, V>(tar + j * DT, xr);
                    unpack_lanes<St, V>(tai + j * DT, xi);
                    unpack_lanes<St, V>(tbr + j * DT, yr);
                    unpack_lanes<St, V>(tbi + j * DT, yi);
                    compute(j, xr, xi, yr, yi, masked);
                }
            }
        };
        if (EXT && rbits != 0) rows(true);
        else rows(false);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
    }
    if (!failed && lane_ok) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            if (last_r) last_r[static_cast<size_t>(brow) * D + d + v] = hr[v];
            if (last_i) last_i[static_cast<size_t>(brow) * D + d + v] = hi[v];
        }
    }
}

// grad_h0 = conj(a'_0) * g_0 for V lanes (+0 where step 0 starts a segment),
// in the oracle's order: (fma(ar, gr, ai*gi), fma(ar, gi, -(ai*gr))).
template <typename St, int V>
__device__ __forceinline__ void store_cgrad_h0(const CStateArgs &sx, bool reset0, size_t a_off, size_t hs,
                                               const float (&gr)[V], const float (&gi)[V]) {
    float ar[V], ai[V];
    load_lanes_global<St, V>(static_cast<const St *>(sx.ar) + a_off, ar);
    load_lanes_global<St, V>(static_cast<const St *>(sx.ai) + a_off, ai);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const float hr = reset0 ? 0.0f : __fmaf_rn(ar[v], gr[v], __fmul_rn(ai[v], gi[v]));
        const float hi = reset0 ? 0.0f : __fmaf_rn(ar[v], gi[v], -__fmul_rn(ai[v], gr[v]));
        if (sx.gh0_r != nullptr) sx.gh0_r[hs + v] = hr;
        if (sx.gh0_i != nullptr) sx.gh0_i[hs + v] = hi;
    }
}

template <class C, int CH, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
cwin_bwd_kernel(const __grid_constant__ CUtensorMap tm_ar, const __grid_constant__ CUtensorMap tm_ai,
                const __grid_constant__ CUtensorMap tm_or, const __grid_constant__ CUtensorMap tm_oi,
                const __grid_constant__ CUtensorMap tm_gr, const __grid_constant__ CUtensorMap tm_gi,
                typename C::St *__restrict__ grad_ar, typename C::St *__restrict__ grad_ai,
                typename C::St *__restrict__ grad_br, typename C::St *__restrict__ grad_bi,
                const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns,
                const __grid_constant__ CStateArgs sx) {
    static_assert(C::SEQ && C::NIN == 6, "complex backward: sequential shape, six input planes");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int NT = G;
    win_init<C>(sm, NT / 32, 1);
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D;
    const int nwin = sm.nwin;

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[6] = {&tm_ar, &tm_ai, &tm_or, &tm_oi, &tm_gr, &tm_gi};
            const int W = sm.W;
            // planes 0, 1: a one step later; 2, 3: out one step earlier; 4, 5: grad_out
            win_producer<C>(sm, maps, d0, brow,
                            [W, nwin](int k, int i) { return (nwin - 1 - k) * W + (i < 2 ? 1 : (i < 4 ? -1 : 0)); },
                            wc);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int d = d0 + threadIdx.x * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    float gr[V], gi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) gr[v] = gi[v] = 0.0f;
    int stage = 0, use = 0;
    const int off = threadIdx.x * V;
    // EXT: bit j of r0bits / r1bits is a reset at row j / j + 1 of the current
    // window (positions loaded one window ahead); h_{-1} = h0
    static_assert(!EXT || L <= 32, "one ballot covers a window's rows");
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    const size_t hs = static_cast<size_t>(brow) * D + d;
    int32_t pos0_next = 1, pos1_next = 1;
    float h0r[V], h0i[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h0r[v] = h0i[v] = 0.0f;
    bool failed = false;
    if constexpr (EXT) {
        if (lane_ok) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                gr[v] = sx.gl_r != nullptr ? sx.gl_r[hs + v] : 0.0f;
                gi[v] = sx.gl_i != nullptr ? sx.gl_i[hs + v] : 0.0f;
                h0r[v] = sx.h0_r != nullptr ? sx.h0_r[hs + v] : 0.0f;
                h0i[v] = sx.h0_i != nullptr ? sx.h0_i[hs + v] : 0.0f;
            }
        }
        const int wb0 = (nwin - 1) * sm.W + lane;
        pos0_next = seg.at(lane < L ? wb0 : -1);
        pos1_next = seg.at(lane < L ? wb0 + 1 : -1);
    }
    for (int k = 0; k < nwin; ++k) {
        uint32_t r0bits = 0, r1bits = 0;
        if constexpr (EXT) {
            r0bits = __ballot_sync(0xffffffffu, pos0_next == 0);
            r1bits = __ballot_sync(0xffffffffu, pos1_next == 0);
            const int wb = (nwin - 2 - k) * sm.W + lane;
            pos0_next = seg.at(lane < L ? wb : -1);
            pos1_next = seg.at(lane < L ? wb + 1 : -1);
        }
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if constexpr (EXT) ok = __all_sync(0xffffffffu, ok);  // keep the warp's ballots converged
        if (!ok) { failed = true; break; }
        const St *tar = sm.tile<C>(stage, 0) + off;  // a_{t+1}
        const St *tai = sm.tile<C>(stage, 1) + off;
        const St *tpr = sm.tile<C>(stage, 2) + off;  // h_{t-1}
        const St *tpi = sm.tile<C>(stage, 3) + off;
        const St *tgr = sm.tile<C>(stage, 4) + off;  // grad_out_t
        const St *tgi = sm.tile<C>(stage, 5) + off;
        const int wbase = (nwin - 1 - k) * sm.W;
        const int n = min(T - wbase, L);
        const size_t o = (row0 + wbase) * D + d;
        // SPECIAL (EXT, warp-uniform): this window holds a reset, step T-1 or step 0
        auto compute = [&](int j, float (&xr)[V], float (&xi)[V], float (&pr)[V], float (&pi)[V],
                           const float (&yr)[V], const float (&yi)[V], bool special) {
            if (EXT && special) {
                // conj(a'_{t+1}): 1 at step T-1 (grad_last enters), 0 where step t+1 starts a segment
                const bool one = k == 0 && j == n - 1;
                const bool zero = (r1bits >> j) & 1u;
                const bool first = wbase + j == 0;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    xr[v] = one ? 1.0f : (zero ? 0.0f : xr[v]);
                    xi[v] = one ? 0.0f : (zero ? 0.0f : xi[v]);
                    pr[v] = first ? h0r[v] : pr[v];
                    pi[v] = first ? h0i[v] : pi[v];
                }
            }
            float far_[V], fai[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float nr = __fmaf_rn(xr[v], gr[v], __fmaf_rn(xi[v], gi[v], yr[v]));
                const float ni = __fmaf_rn(xr[v], gi[v], __fmaf_rn(-xi[v], gr[v], yi[v]));
                gr[v] = nr;
                gi[v] = ni;
                far_[v] = __fmaf_rn(gr[v], pr[v], __fmul_rn(gi[v], pi[v]));
                fai[v] = __fmaf_rn(gi[v], pr[v], -__fmul_rn(gr[v], pi[v]));
            }
            if (EXT && special) {
                if ((r0bits >> j) & 1u) {  // a_t unused at a segment start
#pragma unroll
                    for (int v = 0; v < V; ++v) far_[v] = fai[v] = 0.0f;
                }
            }
            if (lane_ok) {
                const size_t oj = o + static_cast<size_t>(j) * D;
                store_lanes<St, V>(grad_br + oj, gr);
                store_lanes<St, V>(grad_bi + oj, gi);
                store_lanes<St, V>(grad_ar + oj, far_);
                store_lanes<St, V>(grad_ai + oj, fai);
            }
        };
        auto rows = [&](bool special) {
            if (n == L) {
                using Raw = typename RawOf<St, V>::T;
#pragma unroll
                for (int j1 = L; j1 > 0; j1 -= CH) {  // rows j1-CH .. j1-1, last first
                    Raw r[6][CH];
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const int row = (j1 - CH + j) * DT;
                        r[0][j] = load_raw<St, V>(tar + row);
                        r[1][j] = load_raw<St, V>(tai + row);
                        r[2][j] = load_raw<St, V>(tpr + row);
                        r[3][j] = load_raw<St, V>(tpi + row);
                        r[4][j] = load_raw<St, V>(tgr + row);
                        r[5][j] = load_raw<St, V>(tgi + row);
                    }
#pragma unroll
                    for (int j = CH - 1; j >= 0; --j) {
                        float xr[V], xi[V], pr[V], pi[V], yr[V], yi[V];
                        widen_raw(r[0][j], xr);
                        widen_raw(r[1][j], xi);
                        widen_raw(r[2][j], pr);
                        widen_raw(r[3][j], pi);
                        widen_raw(r[4][j], yr);
                        widen_raw(r[5][j], yi);
                        compute(j1 - CH + j, xr, xi, pr, pi, yr, yi, special);
                    }
                }
            } else {
                for (int j = n - 1; j >= 0; --j) {
                    float xr[V], xi[V], pr[V], pi[V], yr[V], yi[V];
                    unpack_lanes<St, V>(tar + j * DT, xr);
                    unpack_lanes<St, V>(tai + j * DT, xi);
                    unpack_lanes<St, V>(tpr + j * DT, pr);
                    unpack_lanes<St, V>(tpi + j * DT, pi);
                    unpack_lanes<St, V>(tgr + j * DT, yr);
                    unpack_lanes<St, V>(tgi + j * DT, yi);
                    compute(j, xr, xi, pr, pi, yr, yi, special);
                }
            }
        };
        if (EXT && ((r0bits | r1bits) != 0 || k == 0 || wbase == 0)) rows(true);
        else rows(false);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
    }
    if constexpr (EXT) {
        if (!failed && lane_ok && (sx.gh0_r != nullptr || sx.gh0_i != nullptr))
            store_cgrad_h0<St, V>(sx, seg.at(0) == 0, row0 * D + d, hs, gr, gi);
    }
    (void)failed;
}

// ---------------------------------------------------------------------------
// Windowed complex forward (S > 1 sub-chunks of L rows per window, lane-scan
// prefix): the window kernel's structure with complex maps.  Thread (s, g)
// holds L rows of its lanes' four planes, summarizes its sub-chunk as the
// complex affine map h -> P*h + Q (P = product of the decays, Q = the
// sub-chunk's scan from zero, both with the recurrence's nested fmas), the
// lane threads walk the S maps in order from the window's carried state, and
// every thread replays its rows from its entry state.  Shared-memory scan
// area per sub-chunk and lane: the map (Pr, Pi, Qr, Qi) and the entry state.
template <class C>
__host__ __device__ inline WinGeom make_cwin_geom(int S, int nstage, int T, int D) {
    WinGeom g = make_win_geom<C>(S, nstage, T, D);
    g.flag_off = g.scan_off + S * C::DT * 24;
    g.smem_bytes = g.flag_off + 16;
    return g;
}

__device__ __forceinline__ void cmul_add(float xr, float xi, float hr, float hi, float br, float bi, float &nr,
                                         float &ni) {
    // (xr + i xi) (hr + i hi) + (br + i bi), in the oracle's nested-fma order
    nr = __fmaf_rn(xr, hr, __fmaf_rn(-xi, hi, br));
    ni = __fmaf_rn(xi, hr, __fmaf_rn(xr, hi, bi));
}

template <class C, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
cwinw_fwd_kernel(const __grid_constant__ CUtensorMap tm_ar, const __grid_constant__ CUtensorMap tm_ai,
                 const __grid_constant__ CUtensorMap tm_br, const __grid_constant__ CUtensorMap tm_bi,
                 const __grid_constant__ CUtensorMap tm_or, const __grid_constant__ CUtensorMap tm_oi,
                 float *__restrict__ last_r, float *__restrict__ last_i, const __grid_constant__ WinGeom geom,
                 DevStatus *status, uint64_t timeout_ns, const __grid_constant__ CStateArgs sx) {
    static_assert(!C::SEQ && !C::PT && C::NIN == 4, "windowed complex forward: lane-scan shape, four planes");
    using St = typename C::St;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    win_init<C>(sm, NT / 32, S);
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T, D = geom.D;

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[4] = {&tm_ar, &tm_ai, &tm_br, &tm_bi};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow, [W](int k, int) { return k * W; }, wc);
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int lane = threadIdx.x & 31;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    float4 *pq = reinterpret_cast<float4 *>(smem_raw + geom.scan_off);                          // [S][DT]
    float2 *entry = reinterpret_cast<float2 *>(smem_raw + geom.scan_off + S * DT * 16);         // [S][DT]
    float cr = 0.0f, ci = 0.0f;  // window-to-window state of lane threadIdx.x (threads < DT)
    int stage = 0, use = 0;
    // out_r / out_i tiles staged in shared memory, stored by one thread
    // outside the lane scan a window late (rows past T, lanes past D clipped)
    const OutStage<2, St> ost = make_out_stage<2, St>(smem_raw, geom);
    const CUtensorMap *const omaps[2] = {&tm_or, &tm_oi};
    const bool issuer = static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    int replayed = 0;
    // EXT: this warp's rows start at window row wrow; bit j of rbits is a
    // reset at row s*L + j of the current window (positions loaded two
    // windows ahead)
    static_assert(!EXT || (G >= 32 ? 1 : 32 / G) * L <= 32, "one ballot covers a warp's rows");
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + static_cast<size_t>(brow) * T : nullptr) : nullptr, T};
    const int wrow = ((threadIdx.x & ~31u) / G) * L;
    int32_t pos_next = 1, pos_next2 = 1;
    if constexpr (EXT) {
        if (static_cast<int>(threadIdx.x) < DT) {
            const int ch = lane_channel<C>(d0, threadIdx.x);
            const size_t hs = static_cast<size_t>(brow) * D + ch;
            cr = (ch < D && sx.h0_r != nullptr) ? sx.h0_r[hs] : 0.0f;
            ci = (ch < D && sx.h0_i != nullptr) ? sx.h0_i[hs] : 0.0f;
        }
        pos_next = seg.at(wrow + lane);
        pos_next2 = seg.at(sm.W + wrow + lane);
    }
    for (int k = 0; k < sm.nwin; ++k) {
        const int rbase = k * sm.W + s * L;
        const int n = min(max(T - rbase, 0), L);
        uint32_t rbits = 0;
        if constexpr (EXT) {
            rbits = __ballot_sync(0xffffffffu, pos_next == 0) >> (s * L - wrow);
            pos_next = pos_next2;
            pos_next2 = seg.at((k + 2) * sm.W + wrow + lane);
        }
        float xr[L][V], xi[L][V], yr[L][V], yi[L][V];
        const bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if (ok) {
            const int off = (s * L) * DT + lg * V;
#pragma unroll
            for (int j = 0; j < L; ++j) {
                unpack_lanes<St, V>(sm.tile<C>(stage, 0) + off + j * DT, xr[j]);
                unpack_lanes<St, V>(sm.tile<C>(stage, 1) + off + j * DT, xi[j]);
                unpack_lanes<St, V>(sm.tile<C>(stage, 2) + off + j * DT, yr[j]);
                unpack_lanes<St, V>(sm.tile<C>(stage, 3) + off + j * DT, yi[j]);
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
        if constexpr (EXT) {
            if (rbits != 0) {
                // a'_t = 0 where step t starts a segment
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    const bool z = (rbits >> j) & 1u;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        xr[j][v] = z ? 0.0f : xr[j][v];
                        xi[j][v] = z ? 0.0f : xi[j][v];
                    }
                }
            }
        }
        if (n < L) {
            // tail sub-chunk: steps past T become exact identity steps (a = 1, b = 0)
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    xr[j][v] = j < n ? xr[j][v] : 1.0f;
                    xi[j][v] = j < n ? xi[j][v] : 0.0f;
                    yr[j][v] = j < n ? yr[j][v] : 0.0f;
                    yi[j][v] = j < n ? yi[j][v] : 0.0f;
                }
            }
        }
        // sub-chunk map: P = product of the decays, Q = the scan from zero
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float pr = 1.0f, pi = 0.0f, qr = 0.0f, qi = 0.0f;
#pragma unroll
            for (int j = 0; j < L; ++j) {
                float npr, npi, nqr, nqi;
                cmul_add(xr[j][v], xi[j][v], pr, pi, 0.0f, 0.0f, npr, npi);
                cmul_add(xr[j][v], xi[j][v], qr, qi, yr[j][v], yi[j][v], nqr, nqi);
                pr = npr; pi = npi; qr = nqr; qi = nqi;
            }
            pq[s * DT + v * G + lg] = make_float4(pr, pi, qr, qi);
        }
        if (bar_sync_or(1, NT, !ok)) break;
        if (issuer && k > 0) {
            // window k-1's rows are staged and fenced; once its stores are
            // issued, the ones before must have finished reading the buffers
            // window k is about to fill
            ost.store(omaps, k - 1, d0, (k - 1) * sm.W, brow);
            bulk_wait_read<1>();
        }
        if (static_cast<int>(threadIdx.x) < DT) {
            // maps read four at a time ahead of their complex fmas (the loads
            // do not queue behind the entry stores)
            float hr = cr, hi = ci;
            for (int i0 = 0; i0 < S; i0 += 4) {
                float4 m[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    m[j] = (i0 + j < S) ? pq[(i0 + j) * DT + threadIdx.x] : make_float4(1.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (i0 + j < S) {
                        entry[(i0 + j) * DT + threadIdx.x] = make_float2(hr, hi);
                        float nr, ni;
                        cmul_add(m[j].x, m[j].y, hr, hi, m[j].z, m[j].w, nr, ni);
                        hr = nr; hi = ni;
                    }
                }
            }
            cr = hr; ci = hi;
        }
        bar_sync_or(1, NT, false);
        float hr[V], hi[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float2 e = entry[s * DT + v * G + lg];
            hr[v] = e.x;
            hi[v] = e.y;
        }
        St *const sor = ost.plane(k, 0) + (s * L) * DT + lg * V;
        St *const soi = ost.plane(k, 1) + (s * L) * DT + lg * V;
#pragma unroll
        for (int j = 0; j < L; ++j) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                float nr, ni;
                cmul_add(xr[j][v], xi[j][v], hr[v], hi[v], yr[j][v], yi[j][v], nr, ni);
                hr[v] = nr; hi[v] = ni;
            }
            store_lanes<St, V>(sor + j * DT, hr);
            store_lanes<St, V>(soi + j * DT, hi);
        }
        fence_proxy_async_smem();
        replayed = k + 1;
        if (lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (last_r) last_r[static_cast<size_t>(brow) * D + d + v] = hr[v];
                if (last_i) last_i[static_cast<size_t>(brow) * D + d + v] = hi[v];
            }
        }
    }
    // the last window's tiles (not after an abort), then every store
    // complete before the CTA's shared memory goes away
    const bool aborted = bar_sync_or(1, NT, replayed != sm.nwin);
    if (issuer) {
        if (!aborted && replayed > 0) ost.store(omaps, replayed - 1, d0, (replayed - 1) * sm.W, brow);
        bulk_wait<0>();
    }
}

// conj(x) * h + b in the sequential backward's nested-fma order.
__device__ __forceinline__ void cmulc_add(float xr, float xi, float hr, float hi, float br, float bi, float &nr,
                                          float &ni) {
    nr = __fmaf_rn(xr, hr, __fmaf_rn(xi, hi, br));
    ni = __fmaf_rn(xr, hi, __fmaf_rn(-xi, hr, bi));
}

// ---------------------------------------------------------------------------
// Windowed complex backward (S sub-chunks of L rows per window, processed in
// reverse, lane-scan prefix): thread (s, g) reads its rows of a_{t+1},
// out_{t-1} and grad_out, summarises its sub-chunk as the complex reverse map
// g -> P g + Q (P the product of conj(a_{t+1}) over its rows), takes the
// adjoint entering its last row from the lane threads' reverse walk over the
// S maps, and replays g_t = conj(a_{t+1}) g_{t+1} + grad_out_t with
// grad_a_t = g_t conj(out_{t-1}), grad_b_t = g_t.  out_{t-1} stays packed
// until the replay.  The four gradient planes are staged in shared memory
// (one buffer per plane) and written by bulk tensor stores, which clip rows
// past T and lanes past D.  Rows past T are identity steps (a = 1,
// grad_out = 0); a_T is the zero fill past the end.
template <class C, bool EXT>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
cwinw_bwd_kernel(const __grid_constant__ CUtensorMap tm_ar, const __grid_constant__ CUtensorMap tm_ai,
                 const __grid_constant__ CUtensorMap tm_or, const __grid_constant__ CUtensorMap tm_oi,
                 const __grid_constant__ CUtensorMap tm_gr, const __grid_constant__ CUtensorMap tm_gi,
                 const __grid_constant__ CUtensorMap tm_gar, const __grid_constant__ CUtensorMap tm_gai,
                 const __grid_constant__ CUtensorMap tm_gbr, const __grid_constant__ CUtensorMap tm_gbi,
                 const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns,
                 const __grid_constant__ CStateArgs sx) {
    static_assert(!C::SEQ && !C::PT && C::NIN == 6, "windowed complex backward: lane-scan shape, six planes");
    using St = typename C::St;
    using Raw = typename RawOf<St, C::V>::T;
    constexpr int V = C::V, L = C::L, DT = C::DT, G = C::G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const WinSmem sm = WinSmem::make(smem_raw, geom);
    const int S = geom.S;
    const int NT = S * G;
    win_init<C>(sm, NT / 32, S);
    pdl_trigger();
    pdl_wait();
    const WaitCtx wc{status, sm.abort_flag(), timeout_ns};
    const int d0 = blockIdx.x * DT;
    const int brow = blockIdx.y;
    const int T = geom.T;
    const int nwin = sm.nwin;

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[6] = {&tm_ar, &tm_ai, &tm_or, &tm_oi, &tm_gr, &tm_gi};
            const int W = sm.W;
            // planes 0, 1: a one step later; 2, 3: out one step earlier; 4, 5: grad_out
            win_producer<C>(sm, maps, d0, brow,
                            [W, nwin](int k, int i) { return (nwin - 1 - k) * W + (i < 2 ? 1 : (i < 4 ? -1 : 0)); },
                            wc);
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int lane = threadIdx.x & 31;
    float4 *pq = reinterpret_cast<float4 *>(smem_raw + geom.scan_off);                   // [S][DT]
    float2 *entry = reinterpret_cast<float2 *>(smem_raw + geom.scan_off + S * DT * 16);  // [S][DT]
    const OutStage<4, St, 1> ost = make_out_stage<4, St, 1>(smem_raw, geom);  // grad_ar, grad_ai, grad_br, grad_bi
    const CUtensorMap *const omaps[4] = {&tm_gar, &tm_gai, &tm_gbr, &tm_gbi};
    const bool issuer = static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    int replayed = 0;
    float cr = 0.0f, ci = 0.0f;  // window-to-window adjoint of lane threadIdx.x (threads < DT)
    int stage = 0, use = 0;
    const int off = (s * L) * DT + lg * V;
    // EXT: bit j of r0bits / r1bits is a reset at row s*L + j / s*L + j + 1 of
    // the current window (positions one window ahead); h_{-1} = h0
    static_assert(!EXT || (G >= 32 ? 1 : 32 / G) * L <= 32, "one ballot covers a warp's rows");
    const int D = geom.D;
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const SegRow seg{EXT ? (sx.seg != nullptr ? sx.seg + row0 : nullptr) : nullptr, T};
    const int wrow = ((threadIdx.x & ~31u) / G) * L;
    int32_t pos0_next = 1, pos1_next = 1, pos0_next2 = 1, pos1_next2 = 1;  // windows k+1, k+2
    float h0r[V], h0i[V];
#pragma unroll
    for (int v = 0; v < V; ++v) h0r[v] = h0i[v] = 0.0f;
    if constexpr (EXT) {
        if (lane_ok) {
            const size_t hs = static_cast<size_t>(brow) * D + d;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                h0r[v] = sx.h0_r != nullptr ? sx.h0_r[hs + v] : 0.0f;
                h0i[v] = sx.h0_i != nullptr ? sx.h0_i[hs + v] : 0.0f;
            }
        }
        if (static_cast<int>(threadIdx.x) < DT) {
            const int ch = lane_channel<C>(d0, threadIdx.x);
            const size_t hs = static_cast<size_t>(brow) * D + ch;
            cr = (ch < D && sx.gl_r != nullptr) ? sx.gl_r[hs] : 0.0f;
            ci = (ch < D && sx.gl_i != nullptr) ? sx.gl_i[hs] : 0.0f;
        }
        const int wb0 = (nwin - 1) * sm.W + wrow + lane;
        pos0_next = seg.at(wb0);
        pos1_next = seg.at(wb0 + 1);
        pos0_next2 = seg.at(wb0 - sm.W);
        pos1_next2 = seg.at(wb0 - sm.W + 1);
    }
    for (int k = 0; k < nwin; ++k) {
        const int wbase = (nwin - 1 - k) * sm.W;
        const int rbase = wbase + s * L;
        const int n = min(max(T - rbase, 0), L);
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
        float xr[L][V], xi[L][V], yr[L][V], yi[L][V];
        Raw pr[L], pi[L];
        const bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        if (ok) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
                unpack_lanes<St, V>(sm.tile<C>(stage, 0) + off + j * DT, xr[j]);
                unpack_lanes<St, V>(sm.tile<C>(stage, 1) + off + j * DT, xi[j]);
                pr[j] = load_raw<St, V>(sm.tile<C>(stage, 2) + off + j * DT);
                pi[j] = load_raw<St, V>(sm.tile<C>(stage, 3) + off + j * DT);
                unpack_lanes<St, V>(sm.tile<C>(stage, 4) + off + j * DT, yr[j]);
                unpack_lanes<St, V>(sm.tile<C>(stage, 5) + off + j * DT, yi[j]);
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
        // rows from na on take conj(a') = 1: steps past T (identity steps)
        // and, with the carried state, step T-1 (grad_last enters through a'_T = 1)
        int na = n;
        if constexpr (EXT) {
            if (n > 0 && rbase + n == T) na = n - 1;
            if (r1bits != 0) {
                // conj(a'_{t+1}) = 0 where step t+1 starts a segment
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    const bool z = (r1bits >> j) & 1u;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        xr[j][v] = z ? 0.0f : xr[j][v];
                        xi[j][v] = z ? 0.0f : xi[j][v];
                    }
                }
            }
        }
        if (na < L) {
            // rows past T: identity steps (a = 1, grad_out = 0)
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    xr[j][v] = j < na ? xr[j][v] : 1.0f;
                    xi[j][v] = j < na ? xi[j][v] : 0.0f;
                    yr[j][v] = j < n ? yr[j][v] : 0.0f;
                    yi[j][v] = j < n ? yi[j][v] : 0.0f;
                }
            }
        }
        // reverse sub-chunk map: g at the first row = P g_after + Q
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float Pr = 1.0f, Pi = 0.0f, Qr = 0.0f, Qi = 0.0f;
#pragma unroll
            for (int j = L - 1; j >= 0; --j) {
                float nPr, nPi, nQr, nQi;
                cmulc_add(xr[j][v], xi[j][v], Pr, Pi, 0.0f, 0.0f, nPr, nPi);
                cmulc_add(xr[j][v], xi[j][v], Qr, Qi, yr[j][v], yi[j][v], nQr, nQi);
                Pr = nPr; Pi = nPi; Qr = nQr; Qi = nQi;
            }
            pq[s * DT + v * G + lg] = make_float4(Pr, Pi, Qr, Qi);
        }
        if (bar_sync_or(1, NT, !ok)) break;
        if (issuer && k > 0) {
            // window k-1's rows are staged and fenced: store them, and let the
            // stores finish reading before this window's replay refills the buffers
            ost.store(omaps, k - 1, d0, wbase + sm.W, brow);
            bulk_wait_read<0>();
        }
        if (static_cast<int>(threadIdx.x) < DT) {
            // lane threads walk the carried adjoint through sub-chunks S-1 .. 0,
            // maps read four at a time ahead of their complex fmas
            float hr = cr, hi = ci;
            for (int i0 = 0; i0 < S; i0 += 4) {
                float4 m[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    m[j] = (i0 + j < S) ? pq[(S - 1 - i0 - j) * DT + threadIdx.x] : make_float4(1.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (i0 + j < S) {
                        entry[(S - 1 - i0 - j) * DT + threadIdx.x] = make_float2(hr, hi);
                        float nr, ni;
                        cmul_add(m[j].x, m[j].y, hr, hi, m[j].z, m[j].w, nr, ni);
                        hr = nr; hi = ni;
                    }
                }
            }
            cr = hr; ci = hi;
        }
        bar_sync_or(1, NT, false);
        float gr[V], gi[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float2 e = entry[s * DT + v * G + lg];
            gr[v] = e.x;
            gi[v] = e.y;
        }
        St *const sar = ost.plane(k, 0) + off;
        St *const sai = ost.plane(k, 1) + off;
        St *const sbr = ost.plane(k, 2) + off;
        St *const sbi = ost.plane(k, 3) + off;
#pragma unroll
        for (int j = L - 1; j >= 0; --j) {
            float hr[V], hi[V], far_[V], fai[V];
            widen_raw(pr[j], hr);
            widen_raw(pi[j], hi);
            if constexpr (EXT) {
                if (j == 0 && rbase == 0) {  // h_{-1} = h0 (fp32)
#pragma unroll
                    for (int v = 0; v < V; ++v) { hr[v] = h0r[v]; hi[v] = h0i[v]; }
                }
            }
#pragma unroll
            for (int v = 0; v < V; ++v) {
                float nr, ni;
                cmulc_add(xr[j][v], xi[j][v], gr[v], gi[v], yr[j][v], yi[j][v], nr, ni);
                gr[v] = nr;
                gi[v] = ni;
                far_[v] = __fmaf_rn(gr[v], hr[v], __fmul_rn(gi[v], hi[v]));
                fai[v] = __fmaf_rn(gi[v], hr[v], -__fmul_rn(gr[v], hi[v]));
            }
            if constexpr (EXT) {
                if ((r0bits >> j) & 1u) {  // a_t unused at a segment start
#pragma unroll
                    for (int v = 0; v < V; ++v) far_[v] = fai[v] = 0.0f;
                }
            }
            store_lanes<St, V>(sar + j * DT, far_);
            store_lanes<St, V>(sai + j * DT, fai);
            store_lanes<St, V>(sbr + j * DT, gr);
            store_lanes<St, V>(sbi + j * DT, gi);
        }
        fence_proxy_async_smem();
        replayed = k + 1;
        if constexpr (EXT) {
            if (rbase == 0 && lane_ok && (sx.gh0_r != nullptr || sx.gh0_i != nullptr))
                store_cgrad_h0<St, V>(sx, seg.at(0) == 0, row0 * D + d, static_cast<size_t>(brow) * D + d, gr, gi);
        }
    }
    // the last processed window's tiles (not after an abort), then every store
    // complete before the CTA's shared memory goes away
    const bool aborted = bar_sync_or(1, NT, replayed != nwin);
    if (issuer) {
        if (!aborted && replayed > 0) ost.store(omaps, replayed - 1, d0, (nwin - replayed) * sm.W, brow);
        bulk_wait<0>();
    }
}

// Plain kernels: one lane per thread, plain loads, any alignment (same order
// of operations, bit-identical to the tiled ones).
template <typename St>
__global__ void __launch_bounds__(128)
cplain_fwd(const St *__restrict__ ar, const St *__restrict__ ai, const St *__restrict__ br,
           const St *__restrict__ bi, St *__restrict__ out_r, St *__restrict__ out_i, float *__restrict__ last_r,
           float *__restrict__ last_i, int T, int D, int nlb) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    size_t i = static_cast<size_t>(brow) * T * D + d;
    float hr = 0.0f, hi = 0.0f;
#pragma unroll 4
    for (int t = 0; t < T; ++t) {
        float xr[1], xi[1], yr[1], yi[1];
        load_lanes_global<St, 1>(ar + i, xr);
        load_lanes_global<St, 1>(ai + i, xi);
        load_lanes_global<St, 1>(br + i, yr);
        load_lanes_global<St, 1>(bi + i, yi);
        const float nr = __fmaf_rn(xr[0], hr, __fmaf_rn(-xi[0], hi, yr[0]));
        const float ni = __fmaf_rn(xi[0], hr, __fmaf_rn(xr[0], hi, yi[0]));
        hr = nr;
        hi = ni;
        const float vr[1] = {hr}, vi[1] = {hi};
        store_lanes<St, 1>(out_r + i, vr);
        store_lanes<St, 1>(out_i + i, vi);
        i += D;
    }
    if (last_r) last_r[static_cast<size_t>(brow) * D + d] = hr;
    if (last_i) last_i[static_cast<size_t>(brow) * D + d] = hi;
}

template <typename St>
__global__ void __launch_bounds__(128)
cplain_bwd(const St *__restrict__ ar, const St *__restrict__ ai, const St *__restrict__ out_r,
           const St *__restrict__ out_i, const St *__restrict__ go_r, const St *__restrict__ go_i,
           St *__restrict__ grad_ar, St *__restrict__ grad_ai, St *__restrict__ grad_br, St *__restrict__ grad_bi,
           int T, int D, int nlb) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    const size_t row = static_cast<size_t>(brow) * T * D + d;
    float gr = 0.0f, gi = 0.0f, xr = 0.0f, xi = 0.0f;  // x: a_{t+1} (0 past T)
#pragma unroll 4
    for (int t = T - 1; t >= 0; --t) {
        const size_t i = row + static_cast<size_t>(t) * D;
        float yr[1], yi[1], pr[1] = {0.0f}, pi[1] = {0.0f}, nxr[1], nxi[1];
        load_lanes_global<St, 1>(go_r + i, yr);
        load_lanes_global<St, 1>(go_i + i, yi);
        load_lanes_global<St, 1>(ar + i, nxr);
        load_lanes_global<St, 1>(ai + i, nxi);
        if (t > 0) {
            load_lanes_global<St, 1>(out_r + i - D, pr);
            load_lanes_global<St, 1>(out_i + i - D, pi);
        }
        const float nr = __fmaf_rn(xr, gr, __fmaf_rn(xi, gi, yr[0]));
        const float ni = __fmaf_rn(xr, gi, __fmaf_rn(-xi, gr, yi[0]));
        gr = nr;
        gi = ni;
        const float vbr[1] = {gr}, vbi[1] = {gi};
        const float var[1] = {__fmaf_rn(gr, pr[0], __fmul_rn(gi, pi[0]))};
        const float vai[1] = {__fmaf_rn(gi, pr[0], -__fmul_rn(gr, pi[0]))};
        store_lanes<St, 1>(grad_br + i, vbr);
        store_lanes<St, 1>(grad_bi + i, vbi);
        store_lanes<St, 1>(grad_ar + i, var);
        store_lanes<St, 1>(grad_ai + i, vai);
        xr = nxr[0];
        xi = nxi[0];
    }
}

}  // namespace lrscan
