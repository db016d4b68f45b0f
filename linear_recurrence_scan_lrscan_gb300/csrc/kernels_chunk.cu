// Instantiations and launchers of the three-phase chunked kernels, the plain
// sequential kernels and the bounded-wait self-test.
#include <algorithm>

#include "chunk_kernels.cuh"
#include "launch.h"

namespace lrscan {

namespace {

inline unsigned blocks_for(const ChunkGeom &g, int64_t B) { return chunk_blocks(g, B); }

inline ChunkGeom chunk_geom(const ChunkLaunch &L, int C, int V) { return make_chunk_geom(L.T, L.D, C, V); }

// Phase 2: the flat warp-per-lane prefix, or (when the launch carries group
// scratch) the grouped form: group maps, their prefix, the per-group rescan.
template <bool REVERSE>
void prefix_phase(const ChunkLaunch &L, const ChunkGeom &g, const float *init) {
    const long long lanes = static_cast<long long>(L.B) * L.D;
    if (L.PG == nullptr) {
        const unsigned pb = static_cast<unsigned>((lanes * 32 + 255) / 256);
        chunk_prefix<REVERSE, 4><<<pb, 256, 0, L.stream>>>(L.P, L.Q, g.Nc, g.D, lanes, init);
        return;
    }
    const int NG = (g.Nc + kGroupChunks - 1) / kGroupChunks;
    const unsigned gb = static_cast<unsigned>((lanes * NG * 32 + 255) / 256);
    chunk_group_reduce<REVERSE, 4><<<gb, 256, 0, L.stream>>>(L.P, L.Q, L.PG, L.QG, g.Nc, g.D, kGroupChunks, NG, lanes);
    const unsigned pb = static_cast<unsigned>((lanes * 32 + 255) / 256);
    chunk_prefix<REVERSE, 4><<<pb, 256, 0, L.stream>>>(L.PG, L.QG, NG, g.D, lanes, init);
    chunk_group_rescan<REVERSE, 4><<<gb, 256, 0, L.stream>>>(L.P, L.Q, L.QG, g.Nc, g.D, kGroupChunks, NG, lanes);
}

template <typename St, int V, int C>
int chunk_fwd_t(const ChunkLaunch &L) {
    const ChunkGeom g = chunk_geom(L, C, V);
    const unsigned nb = blocks_for(g, L.B);
    chunk_summary_fwd<St, V, C><<<nb, 128, 0, L.stream>>>(static_cast<const St *>(L.in0),
                                                          static_cast<const St *>(L.in1), L.P, L.Q, g, L.sx);
    prefix_phase<false>(L, g, L.sx.h0);
    chunk_replay_fwd<St, V, C><<<nb, 128, 0, L.stream>>>(static_cast<const St *>(L.in0),
                                                         static_cast<const St *>(L.in1), L.Q,
                                                         static_cast<St *>(L.out0), L.last, g, L.sx);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <typename St, int V, int C>
int chunk_bwd_t(const ChunkLaunch &L) {
    const ChunkGeom g = chunk_geom(L, C, V);
    const unsigned nb = blocks_for(g, L.B);
    chunk_summary_bwd<St, V, C><<<nb, 128, 0, L.stream>>>(static_cast<const St *>(L.in0),
                                                          static_cast<const St *>(L.in2), L.P, L.Q, g, L.sx);
    prefix_phase<true>(L, g, L.sx.grad_last);
    chunk_replay_bwd<St, V, C><<<nb, 128, 0, L.stream>>>(
        static_cast<const St *>(L.in0), static_cast<const St *>(L.in1), static_cast<const St *>(L.in2), L.Q,
        static_cast<St *>(L.out0), static_cast<St *>(L.out1), g, L.sx);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <typename St, int VMAX>
int chunk_dispatch(const ChunkLaunch &L, bool fwd) {
    const bool vec = L.vec == VMAX;
#define LRSCAN_CHUNK_CASE(CC)                                                      \
    if (L.chunk == CC) {                                                           \
        if (vec) return fwd ? chunk_fwd_t<St, VMAX, CC>(L) : chunk_bwd_t<St, VMAX, CC>(L); \
        return fwd ? chunk_fwd_t<St, 1, CC>(L) : chunk_bwd_t<St, 1, CC>(L);        \
    }
    LRSCAN_CHUNK_CASE(16)
    LRSCAN_CHUNK_CASE(32)
    LRSCAN_CHUNK_CASE(64)
    LRSCAN_CHUNK_CASE(128)
    LRSCAN_CHUNK_CASE(256)
    LRSCAN_CHUNK_CASE(512)
#undef LRSCAN_CHUNK_CASE
    return -2;
}

// h = init (0 if null); then h = fma(P_r, h, Q_r) for r = r0, r0+step, ...
// (n maps); maps is [W][2][n_lanes] fp32.
__global__ void compose_maps_kernel(const float *__restrict__ maps, const float *__restrict__ init,
                                    float *__restrict__ out, long long lanes, int r0, int step, int n) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i >= lanes) return;
    float h = init != nullptr ? init[i] : 0.0f;
    for (int k = 0, r = r0; k < n; ++k, r += step) {
        const float *m = maps + static_cast<size_t>(r) * 2 * lanes;
        h = __fmaf_rn(m[i], h, m[lanes + i]);
    }
    out[i] = h;
}

__global__ void fill_f32_kernel(float *p, size_t n, float v) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = v;
}

__global__ void selftest_wait_kernel(DevStatus *status, uint64_t timeout_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx wc{status, &abort_flag, timeout_ns};
        // Nothing arrives on this barrier: the wait has to expire and report.
        (void)mbar_wait(smem_addr(&bar), 0, wc, kSiteSelftest);
    }
}

}  // namespace

int chunk_fwd(const ChunkLaunch &L, int dtype) {
    return dtype == 0 ? chunk_dispatch<float, 4>(L, true) : chunk_dispatch<bf16_t, 8>(L, true);
}

int chunk_bwd(const ChunkLaunch &L, int dtype) {
    return dtype == 0 ? chunk_dispatch<float, 4>(L, false) : chunk_dispatch<bf16_t, 8>(L, false);
}

int plain_fwd_launch(const ChunkLaunch &L, int dtype) {
    const int nlb = static_cast<int>((L.D + 127) / 128);
    const unsigned nb = static_cast<unsigned>(nlb * L.B);
    if (dtype == 0)
        plain_fwd<float><<<nb, 128, 0, L.stream>>>(static_cast<const float *>(L.in0),
                                                   static_cast<const float *>(L.in1),
                                                   static_cast<float *>(L.out0), L.last,
                                                   static_cast<int>(L.T), static_cast<int>(L.D), nlb, L.sx);
    else
        plain_fwd<bf16_t><<<nb, 128, 0, L.stream>>>(static_cast<const bf16_t *>(L.in0),
                                                    static_cast<const bf16_t *>(L.in1),
                                                    static_cast<bf16_t *>(L.out0), L.last,
                                                    static_cast<int>(L.T), static_cast<int>(L.D), nlb, L.sx);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int plain_bwd_launch(const ChunkLaunch &L, int dtype) {
    const int nlb = static_cast<int>((L.D + 127) / 128);
    const unsigned nb = static_cast<unsigned>(nlb * L.B);
    if (dtype == 0)
        plain_bwd<float><<<nb, 128, 0, L.stream>>>(
            static_cast<const float *>(L.in0), static_cast<const float *>(L.in1),
            static_cast<const float *>(L.in2), static_cast<float *>(L.out0), static_cast<float *>(L.out1),
            static_cast<int>(L.T), static_cast<int>(L.D), nlb, L.sx);
    else
        plain_bwd<bf16_t><<<nb, 128, 0, L.stream>>>(
            static_cast<const bf16_t *>(L.in0), static_cast<const bf16_t *>(L.in1),
            static_cast<const bf16_t *>(L.in2), static_cast<bf16_t *>(L.out0), static_cast<bf16_t *>(L.out1),
            static_cast<int>(L.T), static_cast<int>(L.D), nlb, L.sx);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int summary_launch(const ChunkLaunch &L, int dtype, int dir) {
    const int nlb = static_cast<int>((L.D + 127) / 128);
    const unsigned nb = static_cast<unsigned>(nlb * L.B);
    const int T = static_cast<int>(L.T), D = static_cast<int>(L.D);
    if (dtype == 0) {
        auto fn = dir == 0 ? summary_fwd<float> : summary_bwd<float>;
        fn<<<nb, 128, 0, L.stream>>>(static_cast<const float *>(L.in0), static_cast<const float *>(L.in1), L.P, L.Q,
                                     T, D, nlb, L.sx);
    } else {
        auto fn = dir == 0 ? summary_fwd<bf16_t> : summary_bwd<bf16_t>;
        fn<<<nb, 128, 0, L.stream>>>(static_cast<const bf16_t *>(L.in0), static_cast<const bf16_t *>(L.in1), L.P,
                                     L.Q, T, D, nlb, L.sx);
    }
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int compose_maps_launch(const float *maps, const float *init, float *out, long long lanes, int r0, int step, int n,
                        cudaStream_t stream) {
    if (lanes == 0) return 0;
    const unsigned nb = static_cast<unsigned>((lanes + 255) / 256);
    compose_maps_kernel<<<nb, 256, 0, stream>>>(maps, init, out, lanes, r0, step, n);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int fill_f32_launch(float *p, size_t n, float v, cudaStream_t stream) {
    if (n == 0) return 0;
    const unsigned nb = static_cast<unsigned>(std::min<size_t>((n + 255) / 256, 4096));
    fill_f32_kernel<<<nb, 256, 0, stream>>>(p, n, v);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int selftest_wait_launch(DevStatus *status, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lrscan
