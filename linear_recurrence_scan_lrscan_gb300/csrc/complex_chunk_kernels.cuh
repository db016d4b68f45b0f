// Three-phase chunked complex scan (triton_training_scan.py, the complex
// affine chunk prefix: _complex_affine_prefix_stage / _extract, and its
// grouped form _complex_affine_group_local / _outer / _correct), for complex
// scans whose B*D lanes are too few to fill the GPU with a lane-tiled walk.
// Time is cut into chunks of C steps; every (row, chunk, lane) is one thread
// in phases 1 and 3 (V lanes per thread, 4 on 16-byte aligned rows, else 1:
// the re and im planes are separate arrays, so a warp reads 32*V consecutive
// lanes of each plane).
//
//   phase 1  summary: chunk c of lane (b,d) as the complex affine map
//            h -> P*h + Q (P = product of the decays, Q = the chunk's scan
//            from zero), each step in the sequential kernels' nested-fma form;
//   phase 2  prefix:  one warp per lane composes 32 maps at a time with
//            shuffles (Kogge-Stone, current∘previous = (Pc*Pp, Pc*Qp + Qc),
//            complex products) and carries the running map across blocks of
//            32; each chunk's entry state is written over Q.  For long chunk
//            sequences the grouped form reduces groups of kGroupChunks maps,
//            scans the group maps and rescans every group from its entry;
//   phase 3  replay:  each chunk reruns the sequential body from its entry
//            state and writes the outputs.
//
// The backward runs the phases on g_t = grad_out_t + conj(a_{t+1}) g_{t+1}
// (chunks last to first); conj(a_{t+1}) at a chunk's last step comes from the
// next chunk (0 past T), h_{t-1} at its first step from the previous chunk
// (0 before 0), and grad_a = g * conj(h_{t-1}).  P and Q are fp32
// [B, Nc, D] per component in a caller- or library-owned workspace.
//
// Carried state and segment resets (CStateArgs, every pointer may be null;
// triton_training_scan.py, _samu_tiled_serial_forward / _backward): the
// forward prefix starts from h0 and a_t is zeroed where segment_pos is 0; the
// backward prefix starts from grad_last, which enters step T-1 through
// a'_T = 1; conj(a'_{t+1}) is zeroed where step t+1 starts a segment, grad_a
// is +0 where step t does, h_{-1} = h0 and chunk 0 writes
// grad_h0 = conj(a'_0) * g_0 (+0 at a reset).
#pragma once

#include "chunk_kernels.cuh"
#include "complex_kernels.cuh"
#include "launch.h"

namespace lrscan {

// Segment start at step t (EXT instantiations only; the plain ones carry no
// state and compile the state handling out).
template <bool EXT>
__device__ __forceinline__ bool cseg_reset(const CStateArgs &sx, int brow, int T, int t) {
    return EXT && sx.seg != nullptr && __ldg(sx.seg + static_cast<size_t>(brow) * T + t) == 0;
}

// a'_t of V lanes (re, im): zero where step t starts a segment.
template <typename St, int V, bool EXT>
__device__ __forceinline__ void load_cdecay(const St *pr, const St *pi, const CStateArgs &sx, int brow, int T, int t,
                                            float (&xr)[V], float (&xi)[V]) {
    load_lanes_global<St, V>(pr, xr);
    load_lanes_global<St, V>(pi, xi);
    if (cseg_reset<EXT>(sx, brow, T, t)) {
#pragma unroll
        for (int v = 0; v < V; ++v) { xr[v] = 0.0f; xi[v] = 0.0f; }
    }
}

// Workspace views: P and Q, re and im, each [B, N, D] fp32.
struct CMaps {
    float *pr, *pi, *qr, *qi;
};

// One complex affine map h -> P*h + Q.  A state h is the map (0, h): a
// composition applied to it keeps P = 0 and carries the state in Q.
struct CMap {
    float pr, pi, qr, qi;
};

// cur ∘ prev = (Pc*Pp, Pc*Qp + Qc), products in the nested-fma form
__device__ __forceinline__ CMap ccompose(const CMap &cur, const CMap &prev) {
    CMap r;
    cmul_add(cur.pr, cur.pi, prev.qr, prev.qi, cur.qr, cur.qi, r.qr, r.qi);
    cmul_add(cur.pr, cur.pi, prev.pr, prev.pi, 0.0f, 0.0f, r.pr, r.pi);
    return r;
}

__device__ __forceinline__ CMap cshfl_up(const CMap &m, int off) {
    return {__shfl_up_sync(0xffffffffu, m.pr, off), __shfl_up_sync(0xffffffffu, m.pi, off),
            __shfl_up_sync(0xffffffffu, m.qr, off), __shfl_up_sync(0xffffffffu, m.qi, off)};
}

__device__ __forceinline__ CMap cshfl(const CMap &m, int src) {
    return {__shfl_sync(0xffffffffu, m.pr, src), __shfl_sync(0xffffffffu, m.pi, src),
            __shfl_sync(0xffffffffu, m.qr, src), __shfl_sync(0xffffffffu, m.qi, src)};
}

// ---------------------------------------------------------------- phase 1 --
template <typename St, int V, bool EXT>
__global__ void __launch_bounds__(128)
cchunk_summary_fwd(const St *__restrict__ ar, const St *__restrict__ ai, const St *__restrict__ br,
                   const St *__restrict__ bi, CMaps m, ChunkGeom g, int C, const CStateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    float pr[V], pi[V], qr[V], qi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { pr[v] = 1.0f; pi[v] = 0.0f; qr[v] = 0.0f; qi[v] = 0.0f; }
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
        const size_t o = base + static_cast<size_t>(j) * g.D;
        float xr[V], xi[V], yr[V], yi[V];
        load_cdecay<St, V, EXT>(ar + o, ai + o, sx, brow, g.T, t0 + j, xr, xi);
        load_lanes_global<St, V>(br + o, yr);
        load_lanes_global<St, V>(bi + o, yi);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float npr, npi, nqr, nqi;
            cmul_add(xr[v], xi[v], pr[v], pi[v], 0.0f, 0.0f, npr, npi);
            cmul_add(xr[v], xi[v], qr[v], qi[v], yr[v], yi[v], nqr, nqi);
            pr[v] = npr; pi[v] = npi; qr[v] = nqr; qi[v] = nqi;
        }
    }
    const size_t so = (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
    store_lanes<float, V>(m.pr + so, pr);
    store_lanes<float, V>(m.pi + so, pi);
    store_lanes<float, V>(m.qr + so, qr);
    store_lanes<float, V>(m.qi + so, qi);
}

// The map from the adjoint entering the chunk's last step (g at the next
// chunk's first step) to g at the chunk's first step.
template <typename St, int V, bool EXT>
__global__ void __launch_bounds__(128)
cchunk_summary_bwd(const St *__restrict__ ar, const St *__restrict__ ai, const St *__restrict__ gor,
                   const St *__restrict__ goi, CMaps m, ChunkGeom g, int C, const CStateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    // a'_{t+1} of the last step: the next chunk's first; past T, 1 when
    // grad_last enters there, else 0
    float xr[V], xi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { xr[v] = EXT && sx.gl_r != nullptr ? 1.0f : 0.0f; xi[v] = 0.0f; }
    if (t0 + n < g.T)
        load_cdecay<St, V, EXT>(ar + base + static_cast<size_t>(n) * g.D, ai + base + static_cast<size_t>(n) * g.D, sx,
                           brow, g.T, t0 + n, xr, xi);
    float pr[V], pi[V], qr[V], qi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { pr[v] = 1.0f; pi[v] = 0.0f; qr[v] = 0.0f; qi[v] = 0.0f; }
#pragma unroll 4
    for (int j = n - 1; j >= 0; --j) {
        const size_t o = base + static_cast<size_t>(j) * g.D;
        float yr[V], yi[V], xnr[V], xni[V];
        load_lanes_global<St, V>(gor + o, yr);
        load_lanes_global<St, V>(goi + o, yi);
        load_cdecay<St, V, EXT>(ar + o, ai + o, sx, brow, g.T, t0 + j, xnr, xni);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float npr, npi, nqr, nqi;
            cmulc_add(xr[v], xi[v], pr[v], pi[v], 0.0f, 0.0f, npr, npi);
            cmulc_add(xr[v], xi[v], qr[v], qi[v], yr[v], yi[v], nqr, nqi);
            pr[v] = npr; pi[v] = npi; qr[v] = nqr; qi[v] = nqi;
            xr[v] = xnr[v];
            xi[v] = xni[v];
        }
    }
    const size_t so = (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
    store_lanes<float, V>(m.pr + so, pr);
    store_lanes<float, V>(m.pi + so, pi);
    store_lanes<float, V>(m.qr + so, qr);
    store_lanes<float, V>(m.qi + so, qi);
}

// ---------------------------------------------------------------- phase 2 --
// Scan of one lane's maps at processing-order indices [lo, hi) (ascending
// chunks forward, descending backward), 32 per step, starting from `acc`
// (a state (0, h), or the identity (1, 0) to compose the range).  WRITE:
// every chunk's entry (its exclusive prefix applied to acc, the Q part) over
// Q.  Returns acc composed with the whole range.  The whole warp calls it.
template <bool REVERSE, bool WRITE>
__device__ __forceinline__ CMap cscan_maps(const CMaps m, size_t base, int D, int N, int lo, int hi, CMap acc) {
    const int lane = threadIdx.x & 31;
    for (int c0 = lo; c0 < hi; c0 += 32) {
        const int idx = c0 + lane;
        const int c = REVERSE ? N - 1 - idx : idx;
        CMap u{1.0f, 0.0f, 0.0f, 0.0f};
        if (idx < hi) {
            const size_t o = base + static_cast<size_t>(c) * D;
            u = {__ldcg(m.pr + o), __ldcg(m.pi + o), __ldcg(m.qr + o), __ldcg(m.qi + o)};
        }
        // inclusive Kogge-Stone: u = u ∘ (maps of the lanes below)
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const CMap p = cshfl_up(u, off);
            if (lane >= off) u = ccompose(u, p);
        }
        if (WRITE) {
            CMap ex = cshfl_up(u, 1);
            if (lane == 0) ex = {1.0f, 0.0f, 0.0f, 0.0f};
            if (idx < hi) {
                const CMap e = ccompose(ex, acc);
                const size_t o = base + static_cast<size_t>(c) * D;
                m.qr[o] = e.qr;
                m.qi[o] = e.qi;
            }
        }
        acc = ccompose(cshfl(u, 31), acc);
    }
    return acc;
}

// Flat prefix: one warp per (row, lane) over all N maps; the state entering
// the first processed chunk is 0.
template <bool REVERSE>
__global__ void __launch_bounds__(256)
cchunk_prefix(CMaps m, int N, int D, long long lanes, const float *__restrict__ init_r,
              const float *__restrict__ init_i) {
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wid >= lanes) return;  // whole warps
    const long long brow = wid / D;
    const int d = static_cast<int>(wid - brow * D);
    const size_t base = static_cast<size_t>(brow) * N * D + d;
    // state entering the first processed chunk: h0 (forward) or grad_last (backward)
    const CMap init{0.0f, 0.0f, init_r != nullptr ? __ldg(init_r + wid) : 0.0f,
                    init_i != nullptr ? __ldg(init_i + wid) : 0.0f};
    cscan_maps<REVERSE, true>(m, base, D, N, 0, N, init);
}

// Grouped prefix (a): one warp per (lane, group) composes the group's maps;
// the result goes to group slot g in chunk order (REVERSE: NG-1-g), so the
// flat prefix over the group maps walks them in processing order.
template <bool REVERSE>
__global__ void __launch_bounds__(256)
cchunk_group_reduce(const CMaps m, CMaps gm, int N, int D, int GC, int NG, long long lanes) {
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wid >= lanes * NG) return;
    const int grp = static_cast<int>(wid % NG);
    const long long ln = wid / NG;
    const long long brow = ln / D;
    const int d = static_cast<int>(ln - brow * D);
    const size_t base = static_cast<size_t>(brow) * N * D + d;
    const int lo = grp * GC, hi = min(N, lo + GC);
    const CMap r = cscan_maps<REVERSE, false>(m, base, D, N, lo, hi, CMap{1.0f, 0.0f, 0.0f, 0.0f});
    if ((threadIdx.x & 31) == 0) {
        const size_t gs = (static_cast<size_t>(brow) * NG + (REVERSE ? NG - 1 - grp : grp)) * D + d;
        gm.pr[gs] = r.pr; gm.pi[gs] = r.pi; gm.qr[gs] = r.qr; gm.qi[gs] = r.qi;
    }
}

// Grouped prefix (c): one warp per (lane, group) rescans the group's maps
// from the group's entry state (written over the group's Q by the prefix).
template <bool REVERSE>
__global__ void __launch_bounds__(256)
cchunk_group_rescan(CMaps m, const CMaps gm, int N, int D, int GC, int NG, long long lanes) {
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wid >= lanes * NG) return;
    const int grp = static_cast<int>(wid % NG);
    const long long ln = wid / NG;
    const long long brow = ln / D;
    const int d = static_cast<int>(ln - brow * D);
    const size_t base = static_cast<size_t>(brow) * N * D + d;
    const int lo = grp * GC, hi = min(N, lo + GC);
    const size_t gs = (static_cast<size_t>(brow) * NG + (REVERSE ? NG - 1 - grp : grp)) * D + d;
    const CMap entry{0.0f, 0.0f, __ldcg(gm.qr + gs), __ldcg(gm.qi + gs)};
    cscan_maps<REVERSE, true>(m, base, D, N, lo, hi, entry);
}

// ---------------------------------------------------------------- phase 3 --
template <typename St, int V, bool EXT>
__global__ void __launch_bounds__(128)
cchunk_replay_fwd(const St *__restrict__ ar, const St *__restrict__ ai, const St *__restrict__ br,
                  const St *__restrict__ bi, const CMaps m, St *__restrict__ out_r, St *__restrict__ out_i,
                  float *__restrict__ last_r, float *__restrict__ last_i, ChunkGeom g, int C,
                  const CStateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    const size_t so = (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
    float hr[V], hi[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { hr[v] = __ldcg(m.qr + so + v); hi[v] = __ldcg(m.qi + so + v); }
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
        const size_t o = base + static_cast<size_t>(j) * g.D;
        float xr[V], xi[V], yr[V], yi[V];
        load_cdecay<St, V, EXT>(ar + o, ai + o, sx, brow, g.T, t0 + j, xr, xi);
        load_lanes_global<St, V>(br + o, yr);
        load_lanes_global<St, V>(bi + o, yi);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float nr, ni;
            cmul_add(xr[v], xi[v], hr[v], hi[v], yr[v], yi[v], nr, ni);
            hr[v] = nr;
            hi[v] = ni;
        }
        store_lanes<St, V>(out_r + o, hr);
        store_lanes<St, V>(out_i + o, hi);
    }
    if (c == g.Nc - 1) {
        const size_t ls = static_cast<size_t>(brow) * g.D + d;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            if (last_r != nullptr) last_r[ls + v] = hr[v];
            if (last_i != nullptr) last_i[ls + v] = hi[v];
        }
    }
}

template <typename St, int V, bool EXT>
__global__ void __launch_bounds__(128)
cchunk_replay_bwd(const St *__restrict__ ar, const St *__restrict__ ai, const St *__restrict__ out_r,
                  const St *__restrict__ out_i, const St *__restrict__ gor, const St *__restrict__ goi,
                  const CMaps m, St *__restrict__ gar, St *__restrict__ gai, St *__restrict__ gbr,
                  St *__restrict__ gbi, ChunkGeom g, int C, const CStateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    const size_t so = (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
    float gr[V], gi[V], xr[V], xi[V];  // adjoint at the next chunk's first step; a'_{t+1}
#pragma unroll
    for (int v = 0; v < V; ++v) {
        gr[v] = __ldcg(m.qr + so + v);
        gi[v] = __ldcg(m.qi + so + v);
        xr[v] = EXT && sx.gl_r != nullptr ? 1.0f : 0.0f;
        xi[v] = 0.0f;
    }
    if (t0 + n < g.T)
        load_cdecay<St, V, EXT>(ar + base + static_cast<size_t>(n) * g.D, ai + base + static_cast<size_t>(n) * g.D, sx,
                           brow, g.T, t0 + n, xr, xi);
#pragma unroll 4
    for (int j = n - 1; j >= 0; --j) {
        const size_t o = base + static_cast<size_t>(j) * g.D;
        float yr[V], yi[V], xnr[V], xni[V], pr[V], pi[V], far[V], fai[V];
        load_lanes_global<St, V>(gor + o, yr);
        load_lanes_global<St, V>(goi + o, yi);
        load_cdecay<St, V, EXT>(ar + o, ai + o, sx, brow, g.T, t0 + j, xnr, xni);
        if (t0 + j > 0) {
            load_lanes_global<St, V>(out_r + o - g.D, pr);
            load_lanes_global<St, V>(out_i + o - g.D, pi);
        } else {
            const size_t hs = static_cast<size_t>(brow) * g.D + d;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                pr[v] = EXT && sx.h0_r != nullptr ? sx.h0_r[hs + v] : 0.0f;
                pi[v] = EXT && sx.h0_i != nullptr ? sx.h0_i[hs + v] : 0.0f;
            }
        }
        const bool rz = cseg_reset<EXT>(sx, brow, g.T, t0 + j);  // a_t unused: grad_a = +0
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float nr, ni;
            cmulc_add(xr[v], xi[v], gr[v], gi[v], yr[v], yi[v], nr, ni);
            gr[v] = nr;
            gi[v] = ni;
            // grad_a = g * conj(h_{t-1})
            far[v] = rz ? 0.0f : __fmaf_rn(gr[v], pr[v], __fmul_rn(gi[v], pi[v]));
            fai[v] = rz ? 0.0f : __fmaf_rn(gi[v], pr[v], -__fmul_rn(gr[v], pi[v]));
            xr[v] = xnr[v];
            xi[v] = xni[v];
        }
        store_lanes<St, V>(gbr + o, gr);
        store_lanes<St, V>(gbi + o, gi);
        store_lanes<St, V>(gar + o, far);
        store_lanes<St, V>(gai + o, fai);
    }
    if (EXT && c == 0 && (sx.gh0_r != nullptr || sx.gh0_i != nullptr)) {
        // x holds a'_0: grad_h0 = conj(a'_0) * g_0, exactly +0 at a reset
        const bool r0 = cseg_reset<EXT>(sx, brow, g.T, 0);
        const size_t hs = static_cast<size_t>(brow) * g.D + d;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float hr = r0 ? 0.0f : __fmaf_rn(xr[v], gr[v], __fmul_rn(xi[v], gi[v]));
            const float hi = r0 ? 0.0f : __fmaf_rn(xr[v], gi[v], -__fmul_rn(xi[v], gr[v]));
            if (sx.gh0_r != nullptr) sx.gh0_r[hs + v] = hr;
            if (sx.gh0_i != nullptr) sx.gh0_i[hs + v] = hi;
        }
    }
}

}  // namespace lrscan
