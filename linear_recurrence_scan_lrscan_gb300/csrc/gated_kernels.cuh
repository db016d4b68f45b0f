// Scan with a generated decay (triton_training_scan.py, _samu_forward and
// _samu_precompute_decay, radius part): the decay of lane d at token t is
// rebuilt in the kernel from one value per token and one per lane,
//
//   nu_d = exp(nu_log_d),  E_t = exp(eta_t),  a_{t,d} = exp(-nu_d * E_t),
//   h_t = a_t * h_{t-1} + b_t                  (one fma per step)
//
// so the forward streams b and out (2 elements per (t, d)) instead of a, b
// and out, and the backward streams out and grad_out in and grad_b out (3
// instead of 5).  Backward, with grad_a = g * out_{t-1} and
// q = grad_a * a * (-nu * E) (= dL / dlog a):
//   grad_eta[b,t] = sum_d q,   grad_nu_log[d] = sum_{b,t} q.
// Exponentials are fast approximations, as the page's tl.exp is: e^x is
// taken as 2^(x log2 e) with 2^y on the multi-function unit.  The rate is kept
// in base-2 units, nu2_d = nu_d log2 e, so each decay costs one multiply and
// one ex2 (a = 2^(-nu2 E)), and the kernels accumulate
// q2 = grad_a * a * log2(a) = q / ln 2; gated_finish scales the sums by ln 2.
//
// Tiled sequential kernels (S = 1, L = 32 rows per window): lane j of each
// warp computes E for row j of the window (its eta loaded two windows ahead)
// and every row takes it with one shuffle.  The backward accumulates q per
// row in registers and reduces the warp's 32 rows x 32 lanes with a
// transpose-sum (31 shuffles per window: afterwards lane j holds row j's sum
// over the warp's lanes), written as one partial per (row, warp); q is also
// summed per thread over time for grad_nu_log, written per (batch row,
// lane).  gated_finish sums both partial sets (fixed order: deterministic).
#pragma once

#include "packed_f32x2.cuh"
#include "window_kernels.cuh"

namespace lrscan {

__device__ __forceinline__ float eta_at(const float *row, int t, int T) {
    return (t >= 0 && t < T) ? __ldg(row + t) : 0.0f;
}

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

// 2^y by the PTX ex2.approx.ftz.f32 instruction (relative error about 2^-22;
// results below the normal range flush to zero, i.e. a decay under 2^-126
// is taken as 0).
__device__ __forceinline__ float ex2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// e^x = 2^(x log2 e)
__device__ __forceinline__ float exp_approx(float x) { return ex2_approx(__fmul_rn(x, kLog2e)); }

// Rate of lane d in base-2 units: nu2 = exp(nu_log) log2 e, so a = 2^(-nu2 E).
__device__ __forceinline__ float rate2(const float *nu_log, int d) {
    return __fmul_rn(exp_approx(__ldg(nu_log + d)), kLog2e);
}

// After the call, lane l holds sum over the warp's lanes of v[l] (v has 32
// entries per lane): halves of the remaining entries are exchanged with the
// partner lane at distance 16, 8, 4, 2, 1.
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = upper ? v[i] : v[i + w];
            const float keep = upper ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

template <class C>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
gwin_fwd_kernel(const __grid_constant__ CUtensorMap tm_b, const float *__restrict__ eta,
                const float *__restrict__ nu_log, typename C::St *__restrict__ out, float *__restrict__ last,
                const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns) {
    static_assert(C::SEQ && C::NIN == 1 && C::L == 32 && C::G % 32 == 0,
                  "generated-decay forward: sequential, one plane, 32-row windows, whole warps");
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
            const CUtensorMap *const maps[1] = {&tm_b};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow, [W](int k, int) { return k * W; }, wc);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int d = d0 + threadIdx.x * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const float *eta_row = eta + row0;
    float nu2[V], h[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        nu2[v] = lane_ok ? rate2(nu_log, d + v) : 0.0f;
        h[v] = 0.0f;
    }
    float eta1 = eta_at(eta_row, lane, T), eta2 = eta_at(eta_row, L + lane, T);  // windows k, k+1
    bool failed = false;
    int stage = 0, use = 0;
    const int off = threadIdx.x * V;
    for (int k = 0; k < sm.nwin; ++k) {
        const float e_lane = exp_approx(eta1);  // E of row k*L + lane
        eta1 = eta2;
        eta2 = eta_at(eta_row, (k + 2) * L + lane, T);
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) { failed = true; break; }
        const St *tb = sm.tile<C>(stage, 0) + off;
        const int rbase = k * L;
        const int n = min(T - rbase, L);
        const size_t o = (row0 + rbase) * D + d;
        auto step = [&](int j, const float (&y)[V]) {
            const float e = __shfl_sync(0xffffffffu, e_lane, j);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float a = ex2_approx(-__fmul_rn(nu2[v], e));
                h[v] = __fmaf_rn(a, h[v], y[v]);
            }
            if (lane_ok) store_lanes<St, V>(out + o + static_cast<size_t>(j) * D, h);
        };
        if (n == L) {
            // phases: the window's inputs to registers, every row's decay
            // (independent of the state), then the dependent chain
            using Raw = typename RawOf<St, V>::T;
            Raw rb[L];
            float av[L][V];
#pragma unroll
            for (int j = 0; j < L; ++j) rb[j] = load_raw<St, V>(tb + j * DT);
#pragma unroll
            for (int j = 0; j < L; ++j) {
                const float e = __shfl_sync(0xffffffffu, e_lane, j);
#pragma unroll
                for (int v = 0; v < V; ++v) av[j][v] = ex2_approx(-__fmul_rn(nu2[v], e));
            }
#pragma unroll
            for (int j = 0; j < L; ++j) {
                float y[V];
                widen_raw(rb[j], y);
#pragma unroll
                for (int v = 0; v < V; ++v) h[v] = __fmaf_rn(av[j][v], h[v], y[v]);
                if (lane_ok) store_lanes<St, V>(out + o + static_cast<size_t>(j) * D, h);
            }
        } else {
            for (int j = 0; j < n; ++j) {
                float y[V];
                unpack_lanes<St, V>(tb + j * DT, y);
                step(j, y);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
    }
    if (!failed && lane_ok && last != nullptr) {
#pragma unroll
        for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
    }
}

// Windowed forward (S > 1 sub-chunks of L rows per window, lane-scan prefix;
// the window kernel's structure with the decay tile replaced by generated
// decays): thread (s, g) loads its L rows of b, builds its L decays from the
// rows' eta (loaded one window ahead) and its lanes' nu, summarizes its
// sub-chunk as h -> P*h + Q, takes its entry state from the lane threads'
// in-order walk over the S maps, and replays.  Splitting time inside the CTA
// keeps several times more warps busy than the sequential form.
template <class C>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
gwinw_fwd_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_out,
                 const float *__restrict__ eta, const float *__restrict__ nu_log, float *__restrict__ last,
                 const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns) {
    static_assert(!C::SEQ && !C::PT && C::NIN == 1 && C::G <= 32 && 32 % C::G == 0 && C::G >= C::L,
                  "generated-decay windowed forward: lane-scan shape, one plane, row groups within a warp");
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
            const CUtensorMap *const maps[1] = {&tm_b};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow, [W](int k, int) { return k * W; }, wc);
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int lane = threadIdx.x & 31;
    const int gbase = lane & ~(G - 1);  // first lane of this sub-chunk's thread group
    const int myrow = lg < L ? lg : L - 1;  // row whose E this thread computes
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const float *eta_row = eta + row0;
    // out tiles: staged in shared memory (two window buffers) and written by
    // one thread outside the lane scan with a bulk tensor store, one window
    // late; the tensor map clips rows past T and lanes past D
    const OutStage<1, St> ost = make_out_stage<1, St>(smem_raw, geom);
    const CUtensorMap *const omaps[1] = {&tm_out};
    const bool issuer = static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    float nnu2[V];  // -nu2: the decay exponent is (-nu2) * E
#pragma unroll
    for (int v = 0; v < V; ++v) nnu2[v] = lane_ok ? -rate2(nu_log, d + v) : -0.0f;
    float ev = eta_at(eta_row, s * L + myrow, T);  // eta of row myrow of the current window's sub-chunk
    float h[V];
    int replayed = 0;
    float carry = 0.0f;  // window-to-window state of lane threadIdx.x (threads < DT)
    int stage = 0, use = 0;
    for (int k = 0; k < sm.nwin; ++k) {
        const int rbase = k * sm.W + s * L;
        const int n = min(max(T - rbase, 0), L);
        const float evn = eta_at(eta_row, rbase + sm.W + myrow, T);  // next window
        // E of the sub-chunk's rows: one exponential per thread, then shuffles
        // within the thread group
        const float e_mine = exp_approx(ev);
        float xa[L][V], xb[L][V];
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const float e = __shfl_sync(0xffffffffu, e_mine, gbase + j);
            float ej[V];
#pragma unroll
            for (int v = 0; v < V; ++v) ej[v] = e;
            vmul(xa[j], nnu2, ej);
#pragma unroll
            for (int v = 0; v < V; ++v) xa[j][v] = ex2_approx(xa[j][v]);
        }
        const bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        const St *tb = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;
        if (ok) {
#pragma unroll
            for (int j = 0; j < L; ++j) unpack_lanes<St, V>(tb + j * DT, xb[j]);
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
        float P[V], Q[V];
#pragma unroll
        for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
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
#pragma unroll
        for (int j = 0; j < L; ++j) {
            vmul(P, xa[j], P);
            vfma(Q, xa[j], Q, xb[j]);
        }
        float2 *pq = sm.sPQ<C>(0);
#pragma unroll
        for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
        if (bar_sync_or(1, NT, !ok)) break;
        if (issuer && k > 0) {
            // every thread's rows of window k-1 are staged (fenced before the
            // barrier above); once this store has been issued, the one before
            // it must have finished reading the buffer window k is about to fill
            ost.store(omaps, k - 1, d0, (k - 1) * sm.W, brow);
            bulk_wait_read<1>();
        }
        // lane threads push the carried state through the sub-chunk maps in order
        float *entry = sm.sEntry<C>();
        if (static_cast<int>(threadIdx.x) < DT) carry = lane_walk<false, DT>(pq, entry, S, threadIdx.x, carry);
        bar_sync_or(1, NT, false);
#pragma unroll
        for (int v = 0; v < V; ++v) h[v] = entry[s * DT + v * G + lg];
        St *op = ost.plane(k, 0) + (s * L) * DT + lg * V;
#pragma unroll
        for (int j = 0; j < L; ++j) {
            vfma(h, xa[j], h, xb[j]);
            store_lanes<St, V>(op + j * DT, h);
        }
        fence_proxy_async_smem();
        replayed = k + 1;
        if (last != nullptr && lane_ok && n > 0 && rbase + n == T) {
#pragma unroll
            for (int v = 0; v < V; ++v) last[static_cast<size_t>(brow) * D + d + v] = h[v];
        }
        ev = evn;
    }
    // the last window's tile (not after an abort), then every store complete
    // before the CTA's shared memory goes away
    const bool aborted = bar_sync_or(1, NT, replayed != sm.nwin);
    if (issuer) {
        if (!aborted && replayed > 0) ost.store(omaps, replayed - 1, d0, (replayed - 1) * sm.W, brow);
        bulk_wait<0>();
    }
}

// Backward.  Tiles: out one row early (h_{t-1}; zero fill before t = 0) and
// grad_out.  part_eta: [ncol][prow] with ncol = gridDim.x * (G / 32) warp
// columns and prow = rows B*T of the whole call; part_nu: [B][D].
template <class C>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
gwin_bwd_kernel(const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_go,
                const float *__restrict__ eta, const float *__restrict__ nu_log, typename C::St *__restrict__ grad_b,
                float *__restrict__ part_eta, long long prow, float *__restrict__ part_nu,
                const __grid_constant__ WinGeom geom, DevStatus *status, uint64_t timeout_ns) {
    static_assert(C::SEQ && C::NIN == 2 && C::L == 32 && C::G % 32 == 0,
                  "generated-decay backward: sequential, two planes, 32-row windows, whole warps");
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
            const CUtensorMap *const maps[2] = {&tm_out, &tm_go};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow,
                            [W, nwin](int k, int i) { return (nwin - 1 - k) * W + (i == 0 ? -1 : 0); }, wc);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    const int d = d0 + threadIdx.x * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const float *eta_row = eta + row0;
    const int col = blockIdx.x * (G / 32) + static_cast<int>(threadIdx.x) / 32;
    float nu2[V], g[V], a_next[V], acc_nu[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        nu2[v] = lane_ok ? rate2(nu_log, d + v) : 0.0f;
        g[v] = 0.0f;
        a_next[v] = 0.0f;  // a_T: nothing enters past the end
        acc_nu[v] = 0.0f;
    }
    float eta1 = eta_at(eta_row, (nwin - 1) * L + lane, T), eta2 = eta_at(eta_row, (nwin - 2) * L + lane, T);
    bool failed = false;
    int stage = 0, use = 0;
    const int off = threadIdx.x * V;
    for (int k = 0; k < nwin; ++k) {
        const float e_lane = exp_approx(eta1);
        eta1 = eta2;
        eta2 = eta_at(eta_row, (nwin - 3 - k) * L + lane, T);
        bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) { failed = true; break; }
        const St *th = sm.tile<C>(stage, 0) + off;  // h_{t-1}
        const St *tg = sm.tile<C>(stage, 1) + off;  // grad_out_t
        const int wbase = (nwin - 1 - k) * L;
        const int n = min(T - wbase, L);
        const size_t o = (row0 + wbase) * D + d;
        float qrow[L];
        // phases: every row's log-decay and decay (independent of the state),
        // then the dependent chain.  Rows past T (only in the sequence's last
        // window) are zero-filled: g stays 0 through them and their q is 0;
        // nothing of theirs is stored
        float lav[L][V], av[L][V];
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const float e = __shfl_sync(0xffffffffu, e_lane, j);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                lav[j][v] = -__fmul_rn(nu2[v], e);  // log2 of the decay
                av[j][v] = ex2_approx(lav[j][v]);
            }
        }
#pragma unroll
        for (int j = L - 1; j >= 0; --j) {
            float hp[V], go[V], gav[V];
            unpack_lanes<St, V>(th + j * DT, hp);
            unpack_lanes<St, V>(tg + j * DT, go);
            float qs = 0.0f;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float la = lav[j][v];
                const float a = av[j][v];
                g[v] = __fmaf_rn(a_next[v], g[v], go[v]);
                gav[v] = __fmul_rn(g[v], hp[v]);
                const float q = __fmul_rn(__fmul_rn(gav[v], a), la);
                acc_nu[v] += q;
                qs += q;
                a_next[v] = a;
            }
            qrow[j] = qs;
            if (lane_ok && (n == L || j < n)) store_lanes<St, V>(grad_b + o + static_cast<size_t>(j) * D, g);
        }
        const float rsum = warp_transpose_sum(qrow);  // row wbase + lane
        if (lane < n) part_eta[col * prow + row0 + wbase + lane] = rsum;
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
    }
    if (!failed && lane_ok) {
#pragma unroll
        for (int v = 0; v < V; ++v) part_nu[static_cast<size_t>(brow) * D + d + v] = acc_nu[v];
    }
}

// Row-sum scratch of the windowed backward: per sub-chunk L rows x (G + 1)
// floats, padded so consecutive sub-chunks start 16 banks apart (the two
// sub-chunks of a warp on opposite bank halves): 144 floats for 8 rows of 16.
template <int L, int G>
__host__ __device__ constexpr int gated_qsub_floats() {
    return L * (G + 1) + (16 - (L * (G + 1)) % 32 + 32) % 32;
}

// Windowed backward (S sub-chunks of L = 8 rows, G = 16 threads per
// sub-chunk row, lane-scan prefix).  Tiles: out one row early and grad_out.
// Thread (s, g) builds the decays of rows rbase .. rbase + L (a_{t+1} for
// its last row comes from the next sub-chunk's first row; 0 past T), takes
// the adjoint entering its sub-chunk from the lane threads' walk over the S
// reverse maps, replays, and sums q2 over its rows.  Row sums over the CTA's
// lanes: each thread stores its 8 row sums in shared memory and thread g < 8
// of the sub-chunk adds row g's 16 values.
// part_eta: [gridDim.x][prow] (prow = rows B*T of the whole call, so the
// eight rows of a sub-chunk land in 32 contiguous bytes); part_nu: [B*S][D]
// (time sums per sub-chunk).
template <class C>
__global__ void __launch_bounds__(C::MAXT, C::MINB)
gwinw_bwd_kernel(const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_go,
                 const __grid_constant__ CUtensorMap tm_gb, const float *__restrict__ eta,
                 const float *__restrict__ nu_log, float *__restrict__ part_eta, long long prow,
                 float *__restrict__ part_nu, const __grid_constant__ WinGeom geom, DevStatus *status,
                 uint64_t timeout_ns) {
    static_assert(!C::SEQ && !C::PT && C::NIN == 2 && C::L <= 8 && C::G == 16,
                  "windowed generated-decay backward: lane-scan shape, two planes, up to 8 rows x 16 threads");
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
    const int nwin = sm.nwin;

    if (static_cast<int>(threadIdx.x) >= NT) {
        if (static_cast<int>(threadIdx.x) == NT) {
            const CUtensorMap *const maps[2] = {&tm_out, &tm_go};
            const int W = sm.W;
            win_producer<C>(sm, maps, d0, brow,
                            [W, nwin](int k, int i) { return (nwin - 1 - k) * W + (i == 0 ? -1 : 0); }, wc);
        }
        return;
    }

    const int s = threadIdx.x / G;
    const int lg = threadIdx.x - s * G;
    const int lane = threadIdx.x & 31;
    const int gbase = lane & ~(G - 1);  // first lane of this sub-chunk's thread group
    const int myrow = lg <= L ? lg : L;  // row (of rbase .. rbase + L) whose E this thread computes
    const int d = d0 + lg * V;
    const bool lane_ok = d < D;
    const size_t row0 = static_cast<size_t>(brow) * T;
    const float *eta_row = eta + row0;
    float nnu2[V], acc_nu[V], g[V];  // nnu2 = -nu2: the decay exponent is (-nu2) * E
#pragma unroll
    for (int v = 0; v < V; ++v) {
        nnu2[v] = lane_ok ? -rate2(nu_log, d + v) : -0.0f;
        acc_nu[v] = 0.0f;
    }
    float ev = eta_at(eta_row, (nwin - 1) * sm.W + s * L + myrow, T);  // current window
    float carry = 0.0f;  // window-to-window adjoint of lane threadIdx.x (threads < DT)
    int stage = 0, use = 0;
    // grad_b tiles staged in shared memory, stored by one thread outside the
    // lane scan a window late (rows past T and lanes past D are clipped)
    const OutStage<1, St> ost = make_out_stage<1, St>(smem_raw, geom);
    const CUtensorMap *const omaps[1] = {&tm_gb};
    const bool issuer = static_cast<int>(threadIdx.x) == (NT > DT ? DT : 0);
    int replayed = 0;
    // per-row q2 sums of this thread's sub-chunk: [L][G + 1] floats (odd row
    // pitch: the 8 summing threads read distinct banks), sub-chunks
    // gated_qsub_floats apart (the two sub-chunks of a warp on opposite bank halves)
    float *const qsub = reinterpret_cast<float *>(smem_raw + win_out_smem(geom)) + s * gated_qsub_floats<L, G>();
    for (int k = 0; k < nwin; ++k) {
        const int wbase = (nwin - 1 - k) * sm.W;
        const int rbase = wbase + s * L;
        const int n = min(max(T - rbase, 0), L);
        const float evn = eta_at(eta_row, rbase - sm.W + myrow, T);  // next processed window
        // decays a[j] of rows rbase + j (j = 0..L), and a[j] * log2 a[j] (j < L)
        const float e_mine = exp_approx(ev);
        float a[L + 1][V], w[L][V];
#pragma unroll
        for (int j = 0; j <= L; ++j) {
            const float e = __shfl_sync(0xffffffffu, e_mine, gbase + j);
            float l[V];
#pragma unroll
            for (int v = 0; v < V; ++v) l[v] = e;
            vmul(l, nnu2, l);
#pragma unroll
            for (int v = 0; v < V; ++v) a[j][v] = ex2_approx(l[v]);
            if (j < L) vmul(w[j], a[j], l);
        }
        // grad_out rows stay packed (storage words) until used: fewer registers
        using Raw = typename RawOf<St, V>::T;
        Raw xg[L];
        const bool ok = mbar_wait(sm.full_bar(stage), use & 1, wc, kSiteConsumerFull);
        const St *th = sm.tile<C>(stage, 0) + (s * L) * DT + lg * V;  // h_{t-1}
        const St *tg = sm.tile<C>(stage, 1) + (s * L) * DT + lg * V;  // grad_out_t
        if (ok) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
                float xh[V];
                unpack_lanes<St, V>(th + j * DT, xh);
                xg[j] = load_raw<St, V>(tg + j * DT);
                // w = h_{t-1} a log2 a, so that q2 = g * w
                vmul(w[j], xh, w[j]);
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sm.empty_bar(stage));
        if (++stage == sm.nstage) { stage = 0; ++use; }
        // a'_{t+1} of row j is a[j + 1]: 0 for the row just before the end of
        // the sequence (nothing enters after the last step), 1 for the
        // identity steps past T in a tail sub-chunk.  Only rows j < n use
        // a[j] for their q, and j + 1 >= tl implies j + 1 >= n, so rewriting
        // a[j + 1] there leaves every used a_t intact.  Rows past T get
        // grad_out = 0 and w = 0.
        const int tl = T - rbase;  // rows of this sub-chunk before the sequence's end (may be <= 0)
        if (tl <= L) {
#pragma unroll
            for (int j = 0; j < L; ++j) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    if (j + 1 >= tl) a[j + 1][v] = (j < n) ? 0.0f : 1.0f;
                    if (j >= n) w[j][v] = 0.0f;
                }
                if (j >= n) xg[j] = Raw{};  // zero bits: grad_out = +0
            }
        }
        float P[V], Q[V];
#pragma unroll
        for (int v = 0; v < V; ++v) { P[v] = 1.0f; Q[v] = 0.0f; }
#pragma unroll
        for (int j = L - 1; j >= 0; --j) {
            float gj[V];
            widen_raw(xg[j], gj);
            vmul(P, a[j + 1], P);
            vfma(Q, a[j + 1], Q, gj);
        }
        float2 *pq = sm.sPQ<C>(0);
#pragma unroll
        for (int v = 0; v < V; ++v) pq[s * DT + v * G + lg] = make_float2(P[v], Q[v]);
        if (bar_sync_or(1, NT, !ok)) break;
        if (issuer && k > 0) {
            // window k-1's rows are staged and fenced; once its store is
            // issued, the one before must have finished reading the buffer
            // window k is about to fill
            ost.store(omaps, k - 1, d0, wbase + sm.W, brow);
            bulk_wait_read<1>();
        }
        float *entry = sm.sEntry<C>();
        if (static_cast<int>(threadIdx.x) < DT) carry = lane_walk<true, DT>(pq, entry, S, threadIdx.x, carry);
        bar_sync_or(1, NT, false);
#pragma unroll
        for (int v = 0; v < V; ++v) g[v] = entry[s * DT + v * G + lg];
        St *gbp = ost.plane(k, 0) + (s * L) * DT + lg * V;
#pragma unroll
        for (int j = L - 1; j >= 0; --j) {
            float qs = 0.0f, gj[V], q[V];
            widen_raw(xg[j], gj);
            vfma(g, a[j + 1], g, gj);
            vmul(q, g, w[j]);  // exactly 0 past T: g and w are 0 there
            vadd(acc_nu, acc_nu, q);
#pragma unroll
            for (int v = 0; v < V; ++v) qs += q[v];
            qsub[j * (G + 1) + lg] = qs;
            store_lanes<St, V>(gbp + j * DT, g);
        }
        fence_proxy_async_smem();
        replayed = k + 1;
        // row sums over the sub-chunk's 16 threads (its half-warp): thread
        // lg < L adds row lg's 16 values in order
        __syncwarp();
        if (lg < L) {
            float t = 0.0f;
#pragma unroll
            for (int i = 0; i < G; ++i) t += qsub[lg * (G + 1) + i];
            if (lg < n) part_eta[blockIdx.x * prow + row0 + rbase + lg] = t;
        }
        ev = evn;
    }
    if (lane_ok) {
#pragma unroll
        for (int v = 0; v < V; ++v) part_nu[(static_cast<size_t>(brow) * S + s) * D + d + v] = acc_nu[v];
    }
    // the last processed window's tile (not after an abort), then every store
    // complete before the CTA's shared memory goes away
    const bool aborted = bar_sync_or(1, NT, replayed != nwin);
    if (issuer) {
        if (!aborted && replayed > 0) ost.store(omaps, replayed - 1, d0, (nwin - replayed) * sm.W, brow);
        bulk_wait<0>();
    }
}

// Both gradients are column sums of a row-major [K][N] matrix of partials,
// scaled by ln 2 (the kernels sum q2 = q / ln 2): grad_eta[r] = ln 2 *
// sum_c part_eta[c][r] (K = partial columns, N = rows B*T) and
// grad_nu_log[d] = ln 2 * sum_b part_nu[b][d] (K = partial rows, N = D).
// Blocks [0, blocks0) take the first, the rest the second.  A block covers 64
// columns with 8 threads each; thread y sums the K range [K y / 8, K (y+1) / 8)
// in order and thread y = 0 adds the eight in order (deterministic).
constexpr int kFinishCols = 64, kFinishSplit = 8;

__global__ void __launch_bounds__(kFinishCols * kFinishSplit)
gated_finish(const float *__restrict__ p0, int K0, long long N0, float *__restrict__ o0,
             const float *__restrict__ p1, int K1, long long N1, float *__restrict__ o1, unsigned blocks0) {
    const bool first = blockIdx.x < blocks0;
    const float *p = first ? p0 : p1;
    const int K = first ? K0 : K1;
    const long long N = first ? N0 : N1;
    float *o = first ? o0 : o1;
    const long long n = static_cast<long long>(first ? blockIdx.x : blockIdx.x - blocks0) * kFinishCols + threadIdx.x;
    const int y = threadIdx.y;
    pdl_wait();  // the partials come from the kernel before this one in the stream
    float sum = 0.0f;
    if (n < N) {
        const int k1 = static_cast<int>(static_cast<long long>(K) * (y + 1) / kFinishSplit);
#pragma unroll 4
        for (int k = static_cast<int>(static_cast<long long>(K) * y / kFinishSplit); k < k1; ++k)
            sum += p[k * N + n];
    }
    __shared__ float part[kFinishSplit][kFinishCols];
    part[y][threadIdx.x] = sum;
    __syncthreads();
    if (y == 0 && n < N) {
        float t = part[0][threadIdx.x];
#pragma unroll
        for (int i = 1; i < kFinishSplit; ++i) t += part[i][threadIdx.x];
        o[n] = __fmul_rn(t, kLn2);
    }
}

// Plain kernels (any alignment): thread per lane.  The backward's per-row
// sums over lanes go through a warp shuffle reduction into the same
// [ncol][B*T] partials (ncol = ceil(D / 32)).
template <typename St>
__global__ void __launch_bounds__(128)
gplain_fwd(const float *__restrict__ eta, const float *__restrict__ nu_log, const St *__restrict__ b,
           St *__restrict__ out, float *__restrict__ last, int T, int D, int nlb) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    if (d >= D) return;
    const float nu2 = rate2(nu_log, d);
    size_t i = static_cast<size_t>(brow) * T * D + d;
    float h = 0.0f;
    for (int t = 0; t < T; ++t) {
        float y[1];
        load_lanes_global<St, 1>(b + i, y);
        const float a = ex2_approx(-__fmul_rn(nu2, exp_approx(__ldg(eta + static_cast<size_t>(brow) * T + t))));
        h = __fmaf_rn(a, h, y[0]);
        const float hv[1] = {h};
        store_lanes<St, 1>(out + i, hv);
        i += D;
    }
    if (last != nullptr) last[static_cast<size_t>(brow) * D + d] = h;
}

template <typename St>
__global__ void __launch_bounds__(128)
gplain_bwd(const float *__restrict__ eta, const float *__restrict__ nu_log, const St *__restrict__ out,
           const St *__restrict__ grad_out, St *__restrict__ grad_b, float *__restrict__ part_eta,
           float *__restrict__ part_nu, int T, int D, int nlb) {
    const int brow = blockIdx.x / nlb;
    const int d = (blockIdx.x - brow * nlb) * 128 + threadIdx.x;
    const bool ok = d < D;  // every lane of a warp takes part in the row sums
    const size_t nrows = static_cast<size_t>(gridDim.x / nlb) * T;  // rows B*T: the partials' column stride
    const int col = d / 32;
    const float nu2 = ok ? rate2(nu_log, d) : 0.0f;
    const size_t row = static_cast<size_t>(brow) * T * D + d;
    float g = 0.0f, a_next = 0.0f, acc = 0.0f;
    for (int t = T - 1; t >= 0; --t) {
        const size_t i = row + static_cast<size_t>(t) * D;
        float go[1] = {0.0f}, hp[1] = {0.0f};
        if (ok) {
            load_lanes_global<St, 1>(grad_out + i, go);
            if (t > 0) load_lanes_global<St, 1>(out + i - D, hp);
        }
        const float la = -__fmul_rn(nu2, exp_approx(__ldg(eta + static_cast<size_t>(brow) * T + t)));
        const float a = ex2_approx(la);
        g = __fmaf_rn(a_next, g, go[0]);
        const float q = ok ? __fmul_rn(__fmul_rn(__fmul_rn(g, hp[0]), a), la) : 0.0f;
        acc += q;
        a_next = a;
        if (ok) {
            const float gv[1] = {g};
            store_lanes<St, 1>(grad_b + i, gv);
        }
        float s = q;
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
        if ((threadIdx.x & 31) == 0 && d < D)  // lane 0's lane is the warp's first: d < D iff the warp has lanes
            part_eta[static_cast<size_t>(col) * nrows + static_cast<size_t>(brow) * T + t] = s;
    }
    if (ok) part_nu[static_cast<size_t>(brow) * D + d] = acc;
}

}  // namespace lrscan
