// Generated-decay forward with one warp per lane slice (triton_training_scan.py,
// _samu_forward with the decay of _samu_precompute_decay rebuilt in the kernel,
// as in gated_kernels.cuh).  The windowed tiles split time inside a CTA and
// meet at two CTA barriers per window around a serial walk of the sub-chunk
// maps; here each warp is on its own:
//   - a warp (a CTA) owns LW lanes (V per thread) of one batch row over all T
//     and streams its b tiles of W rows through a ring of NST stages with bulk
//     tensor copies that it issues itself (lane 0), NST - 1 windows ahead;
//   - its S = 32 / (LW / V) thread groups take consecutive L-row sub-chunks of
//     the window: each builds its rows' decays (a = 2^(-nu2 E_t), E_t =
//     exp(eta_t), one exponential per row, taken by one thread of the group
//     and shared by shuffles), reduces its sub-chunk to the map h -> P h + Q,
//     finds the state entering it by an inclusive shuffle scan of the groups'
//     maps applied to the carried state, replays its rows, and writes out_t
//     over b_t in the stage;
//   - lane 0 sends the window out with a bulk tensor store and refills the
//     stage of the window before (its store has read the stage by then).
// L is odd, so the S groups' rows of one sub-chunk position fall in different
// shared-memory banks (no conflicts on the loads and the in-place stores).
// Rows past T take E = 0 and the copy's zero fill: exact identity steps, so a
// window is one block of code from its loads to its stores.  Every wait is
// bounded (LRSCAN_ETIMEOUT in the status word; the warp returns after its
// copies in flight have landed).  The window maps re-associate the
// recurrence: results agree with the sequential definition to rounding.
#pragma once

#include <cfloat>

#include "gated_kernels.cuh"
#include "packed_f32x2.cuh"

namespace lrscan {

// Compiled shape: storage type, lanes per warp, lanes per thread (2 or 4),
// rows per sub-chunk (odd), ring stages.  One warp per CTA.
template <class St_, int LW_, int V_, int L_, int NST_>
struct GWarpShape {
    using St = St_;
    static constexpr int LW = LW_, V = V_, G = LW_ / V_, S = 32 / G, L = L_, W = S * L_, NST = NST_;
    static constexpr int ROWB = LW * static_cast<int>(sizeof(St));  // bytes of one tile row
    static constexpr int TILE = W * ROWB;
    static_assert((V == 2 || V == 4) && LW % V == 0 && 32 % G == 0 && G < 32, "whole thread groups per warp");
    static_assert(L % 2 == 1, "odd sub-chunk rows: the groups' rows fall in different banks");
    static constexpr int NE = (L + G - 1) / G;  // row exponentials per thread and window
    static_assert(ROWB % 16 == 0, "a bulk tensor copy moves whole 16-byte units per row");
    static_assert(TILE % 128 == 0, "stages stay 128-byte aligned");
    static_assert(NST >= 3, "a stage is refilled one window after its store");
};

// Shared memory: NST tiles, NST full barriers, the abort flag.
template <class C>
__host__ __device__ constexpr int gwarp_smem_bytes() {
    return C::NST * C::TILE + C::NST * 8 + 16;
}

template <class C>
__global__ void __launch_bounds__(32, 8)
gwarp_fwd_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_out,
                 const float *__restrict__ eta, const float *__restrict__ nu_log, float *__restrict__ last, int T,
                 int D, DevStatus *status, uint64_t timeout_ns) {
    using St = typename C::St;
    constexpr int V = C::V, G = C::G, S = C::S, L = C::L, W = C::W, NST = C::NST, LW = C::LW;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    auto tile = [&](int st) { return reinterpret_cast<St *>(smem_raw + st * C::TILE); };
    auto full = [&](int st) { return smem_addr(smem_raw + NST * C::TILE + 8 * st); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + NST * C::TILE + NST * 8);
    const int lane = threadIdx.x;
    if (lane == 0) {
        for (int st = 0; st < NST; ++st) mbar_init(full(st), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    // the next launch's CTAs come in only when this grid's are past their
    // main loop (with early launches, as many idle warps as working ones
    // would sit on every SM)
    pdl_wait();
    const WaitCtx wc{status, abort_flag, timeout_ns};
    const int d0 = blockIdx.x * LW;
    const int brow = blockIdx.y;
    const int nwin = (T + W - 1) / W;
    const int s = lane / G;   // sub-chunk of this thread's group
    const int g = lane % G;   // lanes V*g .. V*g + V - 1 of the slice
    const int d = d0 + V * g;
    // rows are 16-byte multiples here, so D is a multiple of 4: all V lanes or none
    const bool lane_ok = d < D;
    // window k: stage k % NST, phase (k / NST) & 1
    auto issue = [&](int k) {
        const int st = k % NST;
        mbar_arrive_expect_tx(full(st), C::TILE);
        tma_load_3d(smem_addr(tile(st)), &tm_b, d0, k * W, brow, full(st));
    };
    int issued = 0;
    if (lane == 0) {
        for (int k = 0; k < NST && k < nwin; ++k) issue(k);
        issued = NST < nwin ? NST : nwin;
    }
    // -nu2: the decay exponent is (-nu2) * E.  An infinite rate is taken as
    // -FLT_MAX, so that the identity steps past T (E = 0) give 2^(-0) = 1 and
    // not 2^NaN (a NaN rate stays NaN).
    float nnu2[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const float r = lane_ok ? -rate2(nu_log, d + v) : -0.0f;
        nnu2[v] = r < -FLT_MAX ? -FLT_MAX : r;
    }
    const float *eta_row = eta + static_cast<size_t>(brow) * T;
    // thread g of group s takes the E of its group's rows g, g + G, ...: eta
    // of those rows of windows k and k + 1
    constexpr int NE = C::NE;
    auto eta_of = [&](int k, int i) {
        return g + G * i < L ? eta_at(eta_row, k * W + s * L + g + G * i, T) : 0.0f;
    };
    float ev[NE], ev_next[NE];
#pragma unroll
    for (int i = 0; i < NE; ++i) {
        ev[i] = eta_of(0, i);
        ev_next[i] = eta_of(1, i);
    }
    float carry[V];  // state entering the window (identical in every group)
#pragma unroll
    for (int v = 0; v < V; ++v) carry[v] = 0.0f;
    int done = 0;
    for (int k = 0; k < nwin; ++k) {
        const int st = k % NST;
        // the tile first, so that one block of code runs from the loads and
        // exponentials to the stores and the scheduler can overlap them
        if (!__all_sync(0xffffffffu, mbar_wait(full(st), static_cast<uint32_t>((k / NST) & 1), wc,
                                               kSiteConsumerFull)))
            break;
        // E of this group's rows g, g + G, ...; 0 past T, where the bulk copy
        // has filled b with zeros: exact identity steps (a = 2^(-0) = 1, b = 0)
        float e_mine[NE];
#pragma unroll
        for (int i = 0; i < NE; ++i) {
            const int t = k * W + s * L + g + G * i;
            e_mine[i] = t < T ? exp_approx(ev[i]) : 0.0f;
            ev[i] = ev_next[i];
            ev_next[i] = eta_of(k + 2, i);
        }
        St *tb = tile(st) + (s * L) * LW + V * g;
        float xa[L][V], xb[L][V];
#pragma unroll
        for (int j = 0; j < L; ++j) unpack_lanes<St, V>(tb + j * LW, xb[j]);
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const float e = __shfl_sync(0xffffffffu, e_mine[j / G], s * G + j % G);
            float ej[V];
#pragma unroll
            for (int v = 0; v < V; ++v) ej[v] = e;
            vmul(xa[j], nnu2, ej);
#pragma unroll
            for (int v = 0; v < V; ++v) xa[j][v] = ex2_approx(xa[j][v]);
        }
        // the sub-chunk's map, rows in chain order
        float P[V], Q[V];
#pragma unroll
        for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
        for (int j = 0; j < L; ++j) {
            vmul(P, xa[j], P);
            vfma(Q, xa[j], Q, xb[j]);
        }
        // inclusive scan over the groups: (P, Q) <- (P, Q) o (map of the
        // groups before), the later map applied after the earlier one
#pragma unroll
        for (int off = G; off < 32; off *= 2) {
            float pp[V], qq[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                pp[v] = __shfl_up_sync(0xffffffffu, P[v], off);
                qq[v] = __shfl_up_sync(0xffffffffu, Q[v], off);
            }
            if (lane >= off) {
                vfma(Q, P, qq, Q);
                vmul(P, P, pp);
            }
        }
        // state after this group's rows, then the state entering them
        float z[V], h[V];
        vfma(z, P, carry, Q);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float up = __shfl_up_sync(0xffffffffu, z[v], G);
            h[v] = s == 0 ? carry[v] : up;
            carry[v] = __shfl_sync(0xffffffffu, z[v], 32 - G + g);
        }
#pragma unroll
        for (int j = 0; j < L; ++j) {
            vfma(h, xa[j], h, xb[j]);
            store_lanes<St, V>(tb + j * LW, h);
        }
        if (last != nullptr && lane_ok && k == nwin - 1 && s == S - 1) {
            // the last group ends on step T - 1 or on identity steps after it
#pragma unroll
            for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&tm_out, smem_addr(tile(st)), d0, k * W, brow);
            bulk_commit();
            // the store of window k - 1 has read its stage: refill it with
            // window k - 1 + NST
            if (k >= 1 && issued < nwin) {
                bulk_wait_read<1>();
                issue(issued);
                ++issued;
            }
        }
        done = k + 1;
    }
    pdl_trigger();
    if (lane == 0) {
        // after an abort: every copy issued has landed before the CTA's shared
        // memory goes away (bounded, blind to the abort flag)
        if (done < nwin) {
            for (int k = done; k < issued; ++k) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(full(k % NST), static_cast<uint32_t>((k / NST) & 1))) {
                    if (global_timer_ns() - t0 > wc.timeout_ns) {
                        record_error(wc, kErrTimeout, kSiteDrain);
                        break;
                    }
                }
            }
        }
        bulk_wait<0>();  // every out store complete
    }
}

// Backward of the warp-slice forward: the adjoint g_t = grad_out_t + a_{t+1}
// g_{t+1} runs over the windows from the last to the first; grad_b = g,
// and q_t = g_t h_{t-1} a_t ln a_t gives grad_eta[t] (the sum over lanes)
// and grad_nu_log[d] (the sum over time).  A stage holds two tiles: out one
// row early (h_{t-1}; zero fill before t = 0) and grad_out; grad_b is written
// over grad_out and leaves by a bulk tensor store.  A group's L rows need L + 1
// decays (a_{t+1} of its last row is the next group's first).  Per-row sums of
// q / ln 2 over the slice's lanes go to part_eta[blockIdx.x][row] (a column
// per slice), per-lane sums over a group's rows to part_nu[(b * S + s)][d];
// the finishing kernel adds the partials and scales by ln 2.
template <class C>
__host__ __device__ constexpr int gwarp_bwd_smem_bytes() {
    return 2 * C::NST * C::TILE + C::NST * 8 + 16;
}

// Thread g of each group of 8 lanes holds 16 values (rows 0..15); afterwards
// it holds the group's sums of rows 2g and 2g + 1 (three halving exchanges).
__device__ __forceinline__ void group8_transpose_sum(float (&v)[16], float &r0, float &r1) {
    const int g = threadIdx.x & 7;
    float v1[8], v2[4];
    {
        const bool hi = (g & 4) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float keep = hi ? v[i + 8] : v[i];
            const float send = hi ? v[i] : v[i + 8];
            v1[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    }
    {
        const bool hi = (g & 2) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float keep = hi ? v1[i + 4] : v1[i];
            const float send = hi ? v1[i] : v1[i + 4];
            v2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
    }
    const bool hi = (g & 1) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = hi ? v2[i + 2] : v2[i];
        const float send = hi ? v2[i] : v2[i + 2];
        const float t = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        if (i == 0) r0 = t;
        else r1 = t;
    }
}

template <class C>
__global__ void __launch_bounds__(32, 8)
gwarp_bwd_kernel(const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_go,
                 const __grid_constant__ CUtensorMap tm_gb, const float *__restrict__ eta,
                 const float *__restrict__ nu_log, float *__restrict__ part_eta, long long prow,
                 float *__restrict__ part_nu, int T, int D, DevStatus *status, uint64_t timeout_ns) {
    using St = typename C::St;
    constexpr int V = C::V, G = C::G, S = C::S, L = C::L, W = C::W, NST = C::NST, LW = C::LW;
    static_assert(V == 2 && G == 8 && L <= 15, "lane pairs, groups of 8 threads, at most 16 decays per group");
    constexpr int NE = (L + 1 + G - 1) / G;  // row exponentials per thread and window
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    auto tile_h = [&](int st) { return reinterpret_cast<St *>(smem_raw + (2 * st) * C::TILE); };
    auto tile_g = [&](int st) { return reinterpret_cast<St *>(smem_raw + (2 * st + 1) * C::TILE); };
    auto full = [&](int st) { return smem_addr(smem_raw + 2 * NST * C::TILE + 8 * st); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + 2 * NST * C::TILE + NST * 8);
    const int lane = threadIdx.x;
    if (lane == 0) {
        for (int st = 0; st < NST; ++st) mbar_init(full(st), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    pdl_wait();
    const WaitCtx wc{status, abort_flag, timeout_ns};
    const int d0 = blockIdx.x * LW;
    const int brow = blockIdx.y;
    const int nwin = (T + W - 1) / W;
    const int s = lane / G;
    const int g = lane % G;
    const int d = d0 + V * g;
    const bool lane_ok = d < D;  // rows are 16-byte multiples here, so D is even: both lanes or neither
    // processed window i is window k = nwin - 1 - i: stage i % NST, phase (i / NST) & 1
    auto issue = [&](int i) {
        const int st = i % NST;
        const int wbase = (nwin - 1 - i) * W;
        mbar_arrive_expect_tx(full(st), 2 * C::TILE);
        tma_load_3d(smem_addr(tile_h(st)), &tm_out, d0, wbase - 1, brow, full(st));
        tma_load_3d(smem_addr(tile_g(st)), &tm_go, d0, wbase, brow, full(st));
    };
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < NST && i < nwin; ++i) issue(i);
        issued = NST < nwin ? NST : nwin;
    }
    // -nu2, finite (see the forward); the decay exponent l = (-nu2) * E is
    // log2 a, so a ln a = ln 2 * a * l and the sums carry q / ln 2
    float nnu2[V], acc_nu[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const float rt = lane_ok ? -rate2(nu_log, d + v) : -0.0f;
        nnu2[v] = rt < -FLT_MAX ? -FLT_MAX : rt;
        acc_nu[v] = 0.0f;
    }
    const size_t row0 = static_cast<size_t>(brow) * T;
    const float *eta_row = eta + row0;
    // thread g takes the E of its group's rows g, g + G (row L is the next
    // group's first) of processed windows i and i + 1
    auto eta_of = [&](int i, int e) {
        return g + G * e <= L ? eta_at(eta_row, (nwin - 1 - i) * W + s * L + g + G * e, T) : 0.0f;
    };
    float ev[NE], ev_next[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        ev[e] = eta_of(0, e);
        ev_next[e] = eta_of(1, e);
    }
    float carry[V];  // adjoint entering the window from the rows after it
#pragma unroll
    for (int v = 0; v < V; ++v) carry[v] = 0.0f;
    int done = 0;
    for (int i = 0; i < nwin; ++i) {
        const int st = i % NST;
        const int wbase = (nwin - 1 - i) * W;
        const int rbase = wbase + s * L;
        if (!__all_sync(0xffffffffu, mbar_wait(full(st), static_cast<uint32_t>((i / NST) & 1), wc,
                                               kSiteConsumerFull)))
            break;
        // E of rows rbase + g + G e; 0 past T (identity steps: a = 1; the
        // zero fill gives grad_out = 0 and h = 0 there, so q = 0)
        float e_mine[NE];
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int t = rbase + g + G * e;
            e_mine[e] = t < T ? exp_approx(ev[e]) : 0.0f;
            ev[e] = ev_next[e];
            ev_next[e] = eta_of(i + 2, e);
        }
        const St *th = tile_h(st) + (s * L) * LW + V * g;  // h_{t-1}
        St *tg = tile_g(st) + (s * L) * LW + V * g;        // grad_out_t, then grad_b_t
        float a[L + 1][V], w[L][V], xg[L][V];
#pragma unroll
        for (int j = 0; j < L; ++j) {
            unpack_lanes<St, V>(tg + j * LW, xg[j]);
            unpack_lanes<St, V>(th + j * LW, w[j]);
        }
#pragma unroll
        for (int j = 0; j <= L; ++j) {
            const float ee = __shfl_sync(0xffffffffu, e_mine[j / G], s * G + j % G);
            float l[V];
#pragma unroll
            for (int v = 0; v < V; ++v) l[v] = ee;
            vmul(l, nnu2, l);
#pragma unroll
            for (int v = 0; v < V; ++v) a[j][v] = ex2_approx(l[v]);
            if (j < L) {
                // w = h_{t-1} a l, so that q / ln 2 = g w
                float al[V];
                vmul(al, a[j], l);
                vmul(w[j], w[j], al);
            }
        }
        // the group's map g_in -> P g_in + Q, rows last to first
        float P[V], Q[V];
#pragma unroll
        for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
        for (int j = L - 1; j >= 0; --j) {
            vmul(P, a[j + 1], P);
            vfma(Q, a[j + 1], Q, xg[j]);
        }
        // inclusive scan from the last group down: (P, Q) <- (P, Q) o (map of
        // the groups after)
#pragma unroll
        for (int off = G; off < 32; off *= 2) {
            float pp[V], qq[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                pp[v] = __shfl_down_sync(0xffffffffu, P[v], off);
                qq[v] = __shfl_down_sync(0xffffffffu, Q[v], off);
            }
            if (lane + off < 32) {
                vfma(Q, P, qq, Q);
                vmul(P, P, pp);
            }
        }
        // adjoint at this group's first row, then the one entering its last row
        float z[V], gg[V];
        vfma(z, P, carry, Q);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float dn = __shfl_down_sync(0xffffffffu, z[v], G);
            gg[v] = s == S - 1 ? carry[v] : dn;
            carry[v] = __shfl_sync(0xffffffffu, z[v], g);
        }
        float qrow[16];
        qrow[15] = 0.0f;
#pragma unroll
        for (int j = L - 1; j >= 0; --j) {
            vfma(gg, a[j + 1], gg, xg[j]);
            store_lanes<St, V>(tg + j * LW, gg);
            float q[V];
            vmul(q, gg, w[j]);
            vadd(acc_nu, acc_nu, q);
            qrow[j] = q[0] + q[1];
        }
#pragma unroll
        for (int j = L; j < 16; ++j) qrow[j] = 0.0f;
        float r0, r1;
        group8_transpose_sum(qrow, r0, r1);
        float *pe = part_eta + static_cast<size_t>(blockIdx.x) * prow + row0 + rbase;
        if (2 * g < L && rbase + 2 * g < T) pe[2 * g] = r0;
        if (2 * g + 1 < L && rbase + 2 * g + 1 < T) pe[2 * g + 1] = r1;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&tm_gb, smem_addr(tile_g(st)), d0, wbase, brow);
            bulk_commit();
            // the store of processed window i - 1 has read its stage: refill it
            if (i >= 1 && issued < nwin) {
                bulk_wait_read<1>();
                issue(issued);
                ++issued;
            }
        }
        done = i + 1;
    }
    if (done == nwin && lane_ok) {
#pragma unroll
        for (int v = 0; v < V; ++v) part_nu[(static_cast<size_t>(brow) * S + s) * D + d + v] = acc_nu[v];
    }
    pdl_trigger();
    if (lane == 0) {
        // after an abort: every copy issued has landed before the CTA's shared
        // memory goes away (bounded, blind to the abort flag)
        if (done < nwin) {
            for (int i = done; i < issued; ++i) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(full(i % NST), static_cast<uint32_t>((i / NST) & 1))) {
                    if (global_timer_ns() - t0 > wc.timeout_ns) {
                        record_error(wc, kErrTimeout, kSiteDrain);
                        break;
                    }
                }
            }
        }
        bulk_wait<0>();  // every grad_b store complete
    }
}

}  // namespace lrscan
