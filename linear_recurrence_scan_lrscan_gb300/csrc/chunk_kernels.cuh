// Three-phase chunked scan (triton_training_scan.py, _real_chunk_summary /
// _real_chunk_prefix / _real_chunk_replay and the _real_reverse_* mirror),
// for shapes whose B*D lanes are too few to fill the GPU with a sequential
// walk: time is cut into chunks of C steps and every (row, chunk, lane) is
// an independent thread in phases 1 and 3.
//
//   phase 1  summary: chunk c of lane (b,d) as the affine map h -> P*h + Q
//            (P = product of the decays, Q = the chunk's scan from zero);
//   phase 2  prefix:  one warp per lane scans the maps of 32 chunks at a time
//            with shuffles (Kogge-Stone, composition current∘previous =
//            (Pc*Pp, Pc*Qp + Qc)) and carries the running state across
//            blocks of 32; the exclusive result (each chunk's entry state) is
//            written over Q;
//   phase 3  replay:  each chunk reruns the sequential body from its entry
//            state and writes the outputs.
//
// The backward runs the same three phases on the reverse recurrence
// g_t = fma(a_{t+1}, g_{t+1}, grad_out_t), chunks walked last to first;
// a_{t+1} at the last step of a chunk comes from the next chunk (0 past T)
// and h_{t-1} at a chunk's first step from the previous chunk (0 before 0).
// A short last chunk (T % C != 0) simply has fewer steps, which equals
// padding it with identity steps (a=1, b=0).
//
// P and Q are fp32 [B, Nc, D] in a caller- or library-owned workspace.
//
// Carried state and segment resets (StateArgs, every pointer may be null):
// the forward prefix starts from h0 and a_t is zeroed where segment_pos is 0;
// the backward prefix starts from grad_last, which enters step T-1 through
// a'_T = 1; a'_{t+1} is zeroed where step t+1 starts a segment, grad_a is +0
// where step t does, h_{-1} = h0 and chunk 0 writes grad_h0 = a'_0 * g_0.
#pragma once

#include "scan_common.cuh"
#include "state_args.h"

namespace lrscan {

// Segment start flag of step t of batch row `brow` (false without positions).
__device__ __forceinline__ bool seg_reset(const StateArgs &sx, int brow, int T, int t) {
    return sx.seg != nullptr && __ldg(sx.seg + static_cast<size_t>(brow) * T + t) == 0;
}

// a'_t: the decay of step t, zero where step t starts a segment.
template <typename St, int V>
__device__ __forceinline__ void load_decay(const St *p, const StateArgs &sx, int brow, int T, int t,
                                           float (&x)[V]) {
    load_lanes_global<St, V>(p, x);
    if (seg_reset(sx, brow, T, t)) {
#pragma unroll
        for (int v = 0; v < V; ++v) x[v] = 0.0f;
    }
}

struct ChunkGeom {
    int T, D, Nc;
    int nlb;   // lane blocks per (row, chunk block)
    int lt;    // threads per chunk row: 128, or ceil(D / V) when that is at most 64
    int cpb;   // chunks per CTA: 128 / lt (several chunks share a CTA when D is small)
    int Ncb;   // chunk blocks per row: ceil(Nc / cpb)
};

// Chunk geometry: 128-thread CTAs; when a chunk row needs at most 64 threads
// (D / V <= 64), one CTA takes 128 / lt chunks so that no thread idles.
inline ChunkGeom make_chunk_geom(int64_t T, int64_t D, int C, int V) {
    ChunkGeom g;
    g.T = static_cast<int>(T);
    g.D = static_cast<int>(D);
    g.Nc = static_cast<int>((T + C - 1) / C);
    const int row_threads = static_cast<int>((D + V - 1) / V);
    if (row_threads <= 64) {
        int lt = 1;
        while (lt < row_threads) lt <<= 1;
        g.lt = lt;
        g.cpb = 128 / lt;
        g.nlb = 1;
    } else {
        g.lt = 128;
        g.cpb = 1;
        g.nlb = (row_threads + 127) / 128;
    }
    g.Ncb = (g.Nc + g.cpb - 1) / g.cpb;
    return g;
}

// CTAs of a chunk-parallel launch over B rows.
inline unsigned chunk_blocks(const ChunkGeom &g, int64_t B) {
    return static_cast<unsigned>(static_cast<int64_t>(g.nlb) * g.Ncb * B);
}

// Linear CTA index -> (row, chunk block, lane block); consecutive CTAs take
// neighbouring lanes of the same chunk block.  Within the CTA, thread t works
// on chunk (block * cpb + t / lt) and lanes ((lane block * lt + t % lt) * V ...).
// Returns false for threads with no chunk or lane.
template <int V>
__device__ __forceinline__ bool chunk_thread(const ChunkGeom &g, int &brow, int &c, int &d) {
    const unsigned idx = blockIdx.x;
    const int lb = static_cast<int>(idx % g.nlb);
    const unsigned rc = idx / g.nlb;
    const int cb = static_cast<int>(rc % g.Ncb);
    brow = static_cast<int>(rc / g.Ncb);
    const int sub = static_cast<int>(threadIdx.x) / g.lt;
    if (sub >= g.cpb) return false;
    c = cb * g.cpb + sub;
    d = (lb * g.lt + static_cast<int>(threadIdx.x) - sub * g.lt) * V;
    return c < g.Nc && d < g.D;
}

template <int V>
__device__ __forceinline__ void store_f32_lanes(float *p, const float (&x)[V]) {
    store_lanes<float, V>(p, x);
}

// ---------------------------------------------------------------- phase 1 --
template <typename St, int V, int C>
__global__ void __launch_bounds__(128)
chunk_summary_fwd(const St *__restrict__ a, const St *__restrict__ b, float *__restrict__ P,
                  float *__restrict__ Q, ChunkGeom g, const StateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    float p[V], q[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { p[v] = 1.0f; q[v] = 0.0f; }
    if (n == C) {
#pragma unroll 16
        for (int j = 0; j < C; ++j) {
            float x[V], y[V];
            load_decay<St, V>(a + base + static_cast<size_t>(j) * g.D, sx, brow, g.T, t0 + j, x);
            load_lanes_global<St, V>(b + base + static_cast<size_t>(j) * g.D, y);
#pragma unroll
            for (int v = 0; v < V; ++v) { p[v] = __fmul_rn(x[v], p[v]); q[v] = __fmaf_rn(x[v], q[v], y[v]); }
        }
    } else {
        for (int j = 0; j < n; ++j) {
            float x[V], y[V];
            load_decay<St, V>(a + base + static_cast<size_t>(j) * g.D, sx, brow, g.T, t0 + j, x);
            load_lanes_global<St, V>(b + base + static_cast<size_t>(j) * g.D, y);
#pragma unroll
            for (int v = 0; v < V; ++v) { p[v] = __fmul_rn(x[v], p[v]); q[v] = __fmaf_rn(x[v], q[v], y[v]); }
        }
    }
    const size_t so = (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
    store_f32_lanes<V>(P + so, p);
    store_f32_lanes<V>(Q + so, q);
}

template <typename St, int V, int C>
__global__ void __launch_bounds__(128)
chunk_summary_bwd(const St *__restrict__ a, const St *__restrict__ grad_out, float *__restrict__ P,
                  float *__restrict__ Q, ChunkGeom g, const StateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    float p[V], q[V], x[V];
#pragma unroll
    for (int v = 0; v < V; ++v) { p[v] = 1.0f; q[v] = 0.0f; }
    // a'_{t+1} for the chunk's last step: first step of the next chunk; past
    // T, 1 when grad_last enters there, else 0
    if (t0 + n < g.T) {
        load_decay<St, V>(a + base + static_cast<size_t>(n) * g.D, sx, brow, g.T, t0 + n, x);
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) x[v] = sx.grad_last != nullptr ? 1.0f : 0.0f;
    }
    for (int j = n - 1; j >= 0; --j) {
        float y[V], xn[V];
        load_lanes_global<St, V>(grad_out + base + static_cast<size_t>(j) * g.D, y);
        load_decay<St, V>(a + base + static_cast<size_t>(j) * g.D, sx, brow, g.T, t0 + j, xn);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            p[v] = __fmul_rn(x[v], p[v]);
            q[v] = __fmaf_rn(x[v], q[v], y[v]);
            x[v] = xn[v];
        }
    }
    const size_t so = (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
    store_f32_lanes<V>(P + so, p);
    store_f32_lanes<V>(Q + so, q);
}

// ---------------------------------------------------------------- phase 2 --
// One warp per (row, lane); chunks taken in processing order (ascending for
// the forward, descending for the backward), 32 per step, UNROLL steps of
// loads in flight.  Q is overwritten with each chunk's entry state.
//
// Identity maps (P == 1, Q == 0 exactly, e.g. chunks made only of padding
// steps a=1, b=0) are transparent: a chunk's entry state is the composite up
// to the last non-identity chunk before it, applied to the block's carried
// state, so every run of identity chunks receives bit-for-bit the same state
// (a tree-shaped scan would otherwise round differently per lane).
template <bool REVERSE, int UNROLL>
__global__ void __launch_bounds__(256)
chunk_prefix(const float *__restrict__ P, float *__restrict__ Q, int Nc, int D, long long lanes,
             const float *__restrict__ init) {
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= lanes) return;
    const long long brow = wid / D;
    const int d = static_cast<int>(wid - brow * D);
    const size_t base = static_cast<size_t>(brow) * Nc * D + d;
    // state entering the first processed chunk: h0 (forward) or grad_last (backward)
    float carry = init != nullptr ? __ldg(init + wid) : 0.0f;
    for (int c0 = 0; c0 < Nc; c0 += 32 * UNROLL) {
        float p[UNROLL], q[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int idx = c0 + u * 32 + lane;
            const int c = REVERSE ? Nc - 1 - idx : idx;
            if (idx < Nc) {
                p[u] = __ldcg(P + base + static_cast<size_t>(c) * D);
                q[u] = __ldcg(Q + base + static_cast<size_t>(c) * D);
            } else {
                p[u] = 1.0f;
                q[u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float pu = p[u], qu = q[u];
            const unsigned live = __ballot_sync(0xffffffffu, !(pu == 1.0f && qu == 0.0f));
            // inclusive Kogge-Stone over the 32 maps: current ∘ previous
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float pp = __shfl_up_sync(0xffffffffu, pu, off);
                const float qp = __shfl_up_sync(0xffffffffu, qu, off);
                if (lane >= off) {
                    qu = __fmaf_rn(pu, qp, qu);
                    pu = __fmul_rn(pu, pp);
                }
            }
            // entry state: composite up to the last non-identity chunk before this one
            const unsigned below = live & ((1u << lane) - 1u);
            const int src = below ? 31 - __clz(below) : 0;
            const float pin = __shfl_sync(0xffffffffu, pu, src);
            const float qin = __shfl_sync(0xffffffffu, qu, src);
            const float entry = below ? __fmaf_rn(pin, carry, qin) : carry;
            const int last_live = live ? 31 - __clz(live) : 0;
            const float pall = __shfl_sync(0xffffffffu, pu, last_live);
            const float qall = __shfl_sync(0xffffffffu, qu, last_live);
            const int idx = c0 + u * 32 + lane;
            if (idx < Nc) {
                const int c = REVERSE ? Nc - 1 - idx : idx;
                Q[base + static_cast<size_t>(c) * D] = entry;
            }
            if (live) carry = __fmaf_rn(pall, carry, qall);
        }
    }
}

// ------------------------------------------------- phase 2, grouped form --
// For long chunk sequences with few lanes the prefix above is one warp per
// lane walking all Nc maps.  The grouped form (the three-level scan of chunk
// maps in triton_training_scan.py, _complex_affine_group_local / _outer /
// _correct) splits every lane's chunks into groups of GC (processing order):
//   (a) chunk_group_reduce: one warp per (lane, group) composes the group's
//       maps into one map (P_g = product of P, Q_g = the group's scan from 0);
//   (b) chunk_prefix over the [B, NG, D] group maps gives each group's entry
//       state (from h0 / grad_last);
//   (c) chunk_group_rescan: one warp per (lane, group) rescans its group's
//       maps from that entry state and writes each chunk's entry over Q.
// Group g holds processing-order indices [g*GC, (g+1)*GC); its map is stored
// at group slot g in chunk order (REVERSE: slot NG-1-g), so (b) walks the
// group maps in the same direction as the chunks.

// Scan of the maps at processing-order indices [lo, hi) of one lane from
// `carry`; writes every chunk's entry state over Q when WRITE.  Identity maps
// are transparent (as in chunk_prefix).  Returns the state after the range.
template <bool REVERSE, int UNROLL, bool WRITE>
__device__ __forceinline__ float scan_map_range(const float *__restrict__ P, float *__restrict__ Q, size_t base, int D,
                                                int Nc, int lo, int hi, float carry) {
    const int lane = threadIdx.x & 31;
    for (int c0 = lo; c0 < hi; c0 += 32 * UNROLL) {
        float p[UNROLL], q[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int idx = c0 + u * 32 + lane;
            const int c = REVERSE ? Nc - 1 - idx : idx;
            if (idx < hi) {
                p[u] = __ldcg(P + base + static_cast<size_t>(c) * D);
                q[u] = __ldcg(Q + base + static_cast<size_t>(c) * D);
            } else {
                p[u] = 1.0f;
                q[u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float pu = p[u], qu = q[u];
            const unsigned live = __ballot_sync(0xffffffffu, !(pu == 1.0f && qu == 0.0f));
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float pp = __shfl_up_sync(0xffffffffu, pu, off);
                const float qp = __shfl_up_sync(0xffffffffu, qu, off);
                if (lane >= off) {
                    qu = __fmaf_rn(pu, qp, qu);
                    pu = __fmul_rn(pu, pp);
                }
            }
            if (WRITE) {
                const unsigned below = live & ((1u << lane) - 1u);
                const int src = below ? 31 - __clz(below) : 0;
                const float pin = __shfl_sync(0xffffffffu, pu, src);
                const float qin = __shfl_sync(0xffffffffu, qu, src);
                const float entry = below ? __fmaf_rn(pin, carry, qin) : carry;
                const int idx = c0 + u * 32 + lane;
                if (idx < hi) Q[base + static_cast<size_t>(REVERSE ? Nc - 1 - idx : idx) * D] = entry;
            }
            const int last_live = live ? 31 - __clz(live) : 0;
            const float pall = __shfl_sync(0xffffffffu, pu, last_live);
            const float qall = __shfl_sync(0xffffffffu, qu, last_live);
            if (live) carry = __fmaf_rn(pall, carry, qall);
        }
    }
    return carry;
}

template <bool REVERSE, int UNROLL>
__global__ void __launch_bounds__(256)
chunk_group_reduce(const float *__restrict__ P, const float *__restrict__ Q, float *__restrict__ PG,
                   float *__restrict__ QG, int Nc, int D, int GC, int NG, long long lanes) {
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wid >= lanes * NG) return;
    const int g = static_cast<int>(wid % NG);
    const long long ln = wid / NG;
    const long long brow = ln / D;
    const int d = static_cast<int>(ln - brow * D);
    const size_t base = static_cast<size_t>(brow) * Nc * D + d;
    const int lo = g * GC, hi = min(Nc, lo + GC);
    // Q_g: the group's scan from zero; P_g: the product of its decays
    const float qg = scan_map_range<REVERSE, UNROLL, false>(P, const_cast<float *>(Q), base, D, Nc, lo, hi, 0.0f);
    const int lane = threadIdx.x & 31;
    float pg = 1.0f;
    for (int idx = lo + lane; idx < hi; idx += 32) pg = __fmul_rn(pg, __ldcg(P + base + static_cast<size_t>(REVERSE ? Nc - 1 - idx : idx) * D));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) pg = __fmul_rn(pg, __shfl_xor_sync(0xffffffffu, pg, off));
    if (lane == 0) {
        const size_t gs = (static_cast<size_t>(brow) * NG + (REVERSE ? NG - 1 - g : g)) * D + d;
        PG[gs] = pg;
        QG[gs] = qg;
    }
}

template <bool REVERSE, int UNROLL>
__global__ void __launch_bounds__(256)
chunk_group_rescan(const float *__restrict__ P, float *__restrict__ Q, const float *__restrict__ HG, int Nc, int D,
                   int GC, int NG, long long lanes) {
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wid >= lanes * NG) return;
    const int g = static_cast<int>(wid % NG);
    const long long ln = wid / NG;
    const long long brow = ln / D;
    const int d = static_cast<int>(ln - brow * D);
    const size_t base = static_cast<size_t>(brow) * Nc * D + d;
    const int lo = g * GC, hi = min(Nc, lo + GC);
    const float entry = __ldcg(HG + (static_cast<size_t>(brow) * NG + (REVERSE ? NG - 1 - g : g)) * D + d);
    scan_map_range<REVERSE, UNROLL, true>(P, Q, base, D, Nc, lo, hi, entry);
}

// ---------------------------------------------------------------- phase 3 --
template <typename St, int V, int C>
__global__ void __launch_bounds__(128)
chunk_replay_fwd(const St *__restrict__ a, const St *__restrict__ b, const float *__restrict__ Hin,
                 St *__restrict__ out, float *__restrict__ last, ChunkGeom g, const StateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    float h[V];
    {
        const float *hp = Hin + (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
#pragma unroll
        for (int v = 0; v < V; ++v) h[v] = __ldcg(hp + v);
    }
    if (n == C) {
#pragma unroll 16
        for (int j = 0; j < C; ++j) {
            float x[V], y[V];
            load_decay<St, V>(a + base + static_cast<size_t>(j) * g.D, sx, brow, g.T, t0 + j, x);
            load_lanes_global<St, V>(b + base + static_cast<size_t>(j) * g.D, y);
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(x[v], h[v], y[v]);
            store_lanes<St, V>(out + base + static_cast<size_t>(j) * g.D, h);
        }
    } else {
        for (int j = 0; j < n; ++j) {
            float x[V], y[V];
            load_decay<St, V>(a + base + static_cast<size_t>(j) * g.D, sx, brow, g.T, t0 + j, x);
            load_lanes_global<St, V>(b + base + static_cast<size_t>(j) * g.D, y);
#pragma unroll
            for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(x[v], h[v], y[v]);
            store_lanes<St, V>(out + base + static_cast<size_t>(j) * g.D, h);
        }
    }
    if (last != nullptr && c == g.Nc - 1) {
#pragma unroll
        for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * g.D + d + v] = h[v];
    }
}

template <typename St, int V, int C>
__global__ void __launch_bounds__(128)
chunk_replay_bwd(const St *__restrict__ a, const St *__restrict__ out, const St *__restrict__ grad_out,
                 const float *__restrict__ Gin, St *__restrict__ grad_a, St *__restrict__ grad_b,
                 ChunkGeom g, const StateArgs sx) {
    int brow, c, d;
    if (!chunk_thread<V>(g, brow, c, d)) return;
    const int t0 = c * C;
    const int n = min(C, g.T - t0);
    const size_t base = (static_cast<size_t>(brow) * g.T + t0) * g.D + d;
    float gv[V], x[V];
    {
        const float *gp = Gin + (static_cast<size_t>(brow) * g.Nc + c) * g.D + d;
#pragma unroll
        for (int v = 0; v < V; ++v) gv[v] = __ldcg(gp + v);
    }
    if (t0 + n < g.T) {
        load_decay<St, V>(a + base + static_cast<size_t>(n) * g.D, sx, brow, g.T, t0 + n, x);
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) x[v] = sx.grad_last != nullptr ? 1.0f : 0.0f;
    }
    for (int j = n - 1; j >= 0; --j) {
        float y[V], hp[V], xn[V], ga[V];
        const size_t o = base + static_cast<size_t>(j) * g.D;
        load_lanes_global<St, V>(grad_out + o, y);
        load_decay<St, V>(a + o, sx, brow, g.T, t0 + j, xn);
        if (t0 + j > 0) {
            load_lanes_global<St, V>(out + o - g.D, hp);
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v)
                hp[v] = sx.h0 != nullptr ? sx.h0[static_cast<size_t>(brow) * g.D + d + v] : 0.0f;
        }
        const bool rz = seg_reset(sx, brow, g.T, t0 + j);  // a_t unused: grad_a = +0
#pragma unroll
        for (int v = 0; v < V; ++v) {
            gv[v] = __fmaf_rn(x[v], gv[v], y[v]);
            ga[v] = rz ? 0.0f : __fmul_rn(gv[v], hp[v]);
            x[v] = xn[v];
        }
        store_lanes<St, V>(grad_b + o, gv);
        store_lanes<St, V>(grad_a + o, ga);
    }
    if (c == 0 && sx.grad_h0 != nullptr) {
        // x holds a'_0
#pragma unroll
        for (int v = 0; v < V; ++v) sx.grad_h0[static_cast<size_t>(brow) * g.D + d + v] = __fmul_rn(x[v], gv[v]);
    }
}

// ------------------------------------------------- plain sequential kernels --
// Thread per lane, plain loads, any alignment.  Same operation order as the
// sequential definition (bit-identical results); used when rows are not
// 16-byte aligned, so bulk tensor copies cannot be used.
template <typename St>
__global__ void __launch_bounds__(128)
plain_fwd(const St *__restrict__ a, const St *__restrict__ b, St *__restrict__ out,
          float *__restrict__ last, int T, int D, int nlb, const StateArgs sx) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    size_t i = static_cast<size_t>(brow) * T * D + d;
    float h = sx.h0 != nullptr ? sx.h0[static_cast<size_t>(brow) * D + d] : 0.0f;
#pragma unroll 8
    for (int t = 0; t < T; ++t) {
        float x[1], y[1];
        load_decay<St, 1>(a + i, sx, brow, T, t, x);
        load_lanes_global<St, 1>(b + i, y);
        h = __fmaf_rn(x[0], h, y[0]);
        const float hv[1] = {h};
        store_lanes<St, 1>(out + i, hv);
        i += D;
    }
    if (last != nullptr) last[static_cast<size_t>(brow) * D + d] = h;
}

template <typename St>
__global__ void __launch_bounds__(128)
plain_bwd(const St *__restrict__ a, const St *__restrict__ out, const St *__restrict__ grad_out,
          St *__restrict__ grad_a, St *__restrict__ grad_b, int T, int D, int nlb, const StateArgs sx) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    const size_t row = static_cast<size_t>(brow) * T * D + d;
    const size_t sd = static_cast<size_t>(brow) * D + d;
    // g_T = grad_last enters step T-1 through a'_T = 1 (without it, a'_T = 0)
    float g = sx.grad_last != nullptr ? sx.grad_last[sd] : 0.0f;
    float x = sx.grad_last != nullptr ? 1.0f : 0.0f;
#pragma unroll 8
    for (int t = T - 1; t >= 0; --t) {
        const size_t i = row + static_cast<size_t>(t) * D;
        float y[1], hp[1] = {0.0f}, xn[1];
        load_lanes_global<St, 1>(grad_out + i, y);
        load_decay<St, 1>(a + i, sx, brow, T, t, xn);
        if (t > 0) load_lanes_global<St, 1>(out + i - D, hp);
        else if (sx.h0 != nullptr) hp[0] = sx.h0[sd];
        g = __fmaf_rn(x, g, y[0]);
        const float gb[1] = {g}, ga[1] = {seg_reset(sx, brow, T, t) ? 0.0f : __fmul_rn(g, hp[0])};
        store_lanes<St, 1>(grad_b + i, gb);
        store_lanes<St, 1>(grad_a + i, ga);
        x = xn[0];
    }
    if (sx.grad_h0 != nullptr) sx.grad_h0[sd] = T > 0 ? __fmul_rn(x, g) : g;  // x holds a'_0
}

// ------------------------------------------------ whole-sequence summary --
// Per lane, the affine map of the whole sequence (one chunk of length T):
// forward  h_{T-1} = P * h_{-1} + Q        (Q: the scan of b from zero)
// backward grad_h0 = P * grad_last + Q     (Q: a'_0 * g_0 from grad_last = 0)
// with P = prod_t a'_t in both directions.  One thread per lane, plain
// loads (coalesced along D), nothing stored but P and Q.
template <typename St>
__global__ void __launch_bounds__(128)
summary_fwd(const St *__restrict__ a, const St *__restrict__ b, float *__restrict__ P, float *__restrict__ Q,
            int T, int D, int nlb, const StateArgs sx) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    size_t i = static_cast<size_t>(brow) * T * D + d;
    float p = 1.0f, q = 0.0f;
#pragma unroll 8
    for (int t = 0; t < T; ++t) {
        float x[1], y[1];
        load_decay<St, 1>(a + i, sx, brow, T, t, x);
        load_lanes_global<St, 1>(b + i, y);
        p = __fmul_rn(x[0], p);
        q = __fmaf_rn(x[0], q, y[0]);
        i += D;
    }
    P[static_cast<size_t>(brow) * D + d] = p;
    Q[static_cast<size_t>(brow) * D + d] = q;
}

template <typename St>
__global__ void __launch_bounds__(128)
summary_bwd(const St *__restrict__ a, const St *__restrict__ grad_out, float *__restrict__ P,
            float *__restrict__ Q, int T, int D, int nlb, const StateArgs sx) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    const size_t row = static_cast<size_t>(brow) * T * D + d;
    float p = 1.0f, g = 0.0f, x = 0.0f;  // x: a'_{t+1} (nothing enters past T: grad_last = 0)
#pragma unroll 8
    for (int t = T - 1; t >= 0; --t) {
        const size_t i = row + static_cast<size_t>(t) * D;
        float y[1], xn[1];
        load_lanes_global<St, 1>(grad_out + i, y);
        load_decay<St, 1>(a + i, sx, brow, T, t, xn);
        g = __fmaf_rn(x, g, y[0]);
        p = __fmul_rn(xn[0], p);
        x = xn[0];
    }
    P[static_cast<size_t>(brow) * D + d] = p;
    Q[static_cast<size_t>(brow) * D + d] = T > 0 ? __fmul_rn(x, g) : 0.0f;  // x holds a'_0
}

}  // namespace lrscan
