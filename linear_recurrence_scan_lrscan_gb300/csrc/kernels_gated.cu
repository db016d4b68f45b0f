// Instantiations and launchers of the generated-decay scan kernels, and their
// tile variant table.
#include <algorithm>
#include <cstdlib>

#include "gated_kernels.cuh"
#include "gated_pipe_kernels.cuh"
#include "gated_warp_kernels.cuh"
#include "window_launch.cuh"

namespace lrscan {

namespace {

template <class C>
int launch_gwin_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gwin_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(1, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    using St = typename C::St;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], L.eta, L.nu_log, static_cast<St *>(L.out0), L.last, g,
                                     L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_gwinw_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gwinw_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), win_out_smem(g),
                                     L.stream, *L.maps[0], *L.maps[1], L.eta, L.nu_log, L.last, g, L.status,
                                     L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_gwinw_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gwinw_bwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads),
                                     win_out_smem(g) + cfg.s * gated_qsub_floats<C::L, C::G>() * 4, L.stream,
                                     *L.maps[0], *L.maps[1],
                                     *L.maps[2], L.eta, L.nu_log, L.part_eta,
                                     static_cast<long long>(L.part_rows), L.part_nu, g, L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_gwin_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gwin_bwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(1, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    using St = typename C::St;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], L.eta, L.nu_log, static_cast<St *>(L.out0),
                                     L.part_eta, static_cast<long long>(L.part_rows), L.part_nu, g, L.status,
                                     L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_gpipe_fwd(const WinLaunch &L, const WinDirCfg &) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gpipe_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const GPipeGeom g = make_gpipe_geom<C>();
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(C::THREADS), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], L.eta, L.nu_log, L.last, static_cast<int>(L.T),
                                     static_cast<int>(L.D), L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_gwarp_fwd(const WinLaunch &L, const WinDirCfg &) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gwarp_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const int nsl = static_cast<int>((L.D + C::LW - 1) / C::LW);
    const cudaError_t e = launch_pdl(fn, dim3(nsl, static_cast<unsigned>(L.B)), dim3(32), gwarp_smem_bytes<C>(),
                                     L.stream, *L.maps[0], *L.maps[1], L.eta, L.nu_log, L.last, static_cast<int>(L.T),
                                     static_cast<int>(L.D), L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_gwarp_bwd(const WinLaunch &L, const WinDirCfg &) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = gwarp_bwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const int nsl = static_cast<int>((L.D + C::LW - 1) / C::LW);
    const cudaError_t e =
        launch_pdl(fn, dim3(nsl, static_cast<unsigned>(L.B)), dim3(32), gwarp_bwd_smem_bytes<C>(), L.stream,
                   *L.maps[0], *L.maps[1], *L.maps[2], L.eta, L.nu_log, L.part_eta,
                   static_cast<long long>(L.part_rows), L.part_nu, static_cast<int>(L.T), static_cast<int>(L.D),
                   L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

// One warp per lane slice (gated_warp_kernels.cuh): a CTA is one warp over LW
// lanes; its tiles are LW lanes by W rows.  The backward's partials: one
// column per slice, one nu row per batch row and thread group.
template <class C>
WinDirCfg gwarp_cfg() {
    WinDirCfg d{};
    d.dt = C::LW;
    d.v = C::V;
    d.l = C::L;
    d.s = C::S;
    d.lane_scan = 1;
    d.exact = 0;
    d.w = C::W;
    d.nstage = C::NST;
    d.threads = 32;
    d.smem = gwarp_smem_bytes<C>();
    d.stage_bytes = C::TILE;
    d.max_resident = 0;
    d.launch = &launch_gwarp_fwd<C>;
    return d;
}
template <class C>
WinDirCfg gwarp_bwd_cfg() {
    WinDirCfg d{};
    d.dt = C::LW;
    d.v = C::V;
    d.l = C::L;
    d.s = C::S;
    d.lane_scan = 1;
    d.exact = 0;
    d.w = C::W;
    d.nstage = C::NST;
    d.threads = 32;
    d.smem = gwarp_bwd_smem_bytes<C>();
    d.stage_bytes = 2 * C::TILE;
    d.max_resident = 0;
    d.launch = &launch_gwarp_bwd<C>;
    return d;
}

// Forward with warp roles (gated_pipe_kernels.cuh): W-row windows, one lane per
// thread, a ring of NST b tiles.
template <class C>
WinDirCfg gpdir_cfg() {
    const GPipeGeom g = make_gpipe_geom<C>();
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = 1;
    d.l = C::W;
    d.s = 1;
    d.lane_scan = 1;
    d.exact = 0;
    d.w = C::W;
    d.nstage = C::NST;
    d.threads = C::THREADS;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.tile_bytes;
    d.max_resident = C::MINB;
    d.launch = &launch_gpipe_fwd<C>;
    return d;
}

template <class C, bool FWD>
WinDirCfg gdir_cfg(int nstage) {
    static_assert(C::NIN == (FWD ? 1 : 2), "generated-decay planes: b forward; out and grad_out backward");
    const WinGeom g = make_win_geom<C>(1, nstage, 1, 1);
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = 1;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = C::G + 32;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) d.launch = &launch_gwin_fwd<C>;
    else d.launch = &launch_gwin_bwd<C>;
    return d;
}

// Windowed generated-decay tiles: S sub-chunks of L = 8 rows, lane scan.
template <class C, bool FWD>
WinDirCfg gwdir_cfg(int S, int nstage) {
    static_assert(!C::SEQ && !C::PT && C::NIN == (FWD ? 1 : 2), "windowed generated-decay shape");
    const WinGeom g = make_win_geom<C>(S, nstage, 1, 1);
    if (S > C::SMAX || (S * C::G) % 32 != 0) std::abort();  // table error: sub-chunk groups fill whole warps
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.lane_scan = 1;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = S * C::G + 32;
    // plus the staging buffers of out (forward) or grad_b (backward) and the
    // backward's row-sum scratch
    d.smem = win_out_smem(g) + (FWD ? 0 : S * gated_qsub_floats<C::L, C::G>() * 4);
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) d.launch = &launch_gwinw_fwd<C>;
    else d.launch = &launch_gwinw_bwd<C>;
    return d;
}

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ>
using GBF_64_1 = WinShape<bf16_t, 64, 1, 32, 1, 96, 1, true>;
using GBB_64_1 = WinShape<bf16_t, 64, 1, 32, 2, 96, 1, true>;
using GBF_64_2 = WinShape<bf16_t, 64, 2, 32, 1, 64, 1, true>;
using GBB_64_2 = WinShape<bf16_t, 64, 2, 32, 2, 64, 1, true>;
using GFF_32_1 = WinShape<float, 32, 1, 32, 1, 64, 1, true>;
using GFB_32_1 = WinShape<float, 32, 1, 32, 2, 64, 1, true>;
using GFF_64_2 = WinShape<float, 64, 2, 32, 1, 64, 1, true>;
using GFB_64_2 = WinShape<float, 64, 2, 32, 2, 64, 1, true>;

using GWF_BF_32_2_8 = WinShape<bf16_t, 32, 2, 8, 1, 160, 5, false>;
using GWF_FF_32_1_8 = WinShape<float, 32, 1, 8, 1, 288, 2, false>;
using GWB_BF_32_2_8 = WinShape<bf16_t, 32, 2, 8, 2, 288, 2, false>;
using GWB_BF_32_2_8_M4 = WinShape<bf16_t, 32, 2, 8, 2, 160, 4, false>;
using GWB_BF_32_2_8_M5 = WinShape<bf16_t, 32, 2, 8, 2, 160, 5, false>;
using GWB_FF_16_1_8 = WinShape<float, 16, 1, 8, 2, 288, 2, false>;

// GPipeShape<St, W, NS, NR, NST, NM, MINB>: two summary and three replay warps
// on 16-row windows, twelve ring stages, eight window slots, five CTAs per SM
// (fp32 only: with bf16 rows the warp handoffs per window, not the bytes, set
// the time).
using GP_FF_16 = GPipeShape<float, 16, 2, 3, 12, 8, 5>;

// GWarpShape<St, LW, V, L, NST>: lanes per warp, lanes per thread, rows per
// sub-chunk, ring stages.
// GWarpShape<St, LW, V, L, NST>: lanes per warp, lanes per thread, rows per
// sub-chunk, ring stages.  Measured on B=8 T=2048 D=2560 forward (CUDA
// events): bf16 33.9 us with 15-row sub-chunks, 33.8 with 23, 35.1 before
// the window was one block of code, 42.6 with 7 (windowed tile 38.1); fp32
// 54.0 us with 15 (tile with warp roles 61.7).  Slower: 32-lane slices with
// four lanes per thread (bf16 46.7 us), 8-lane slices (16-byte rows; 64.2),
// 31-row sub-chunks (38.6), two warps per slice taking windows in turn and
// handing the state over by an mbarrier (36.1) or a polled word (46.2), and a
// software pipeline overlapping window k+1's summary with window k's replay
// (54.2).
using GW_BF_16_15 = GWarpShape<bf16_t, 16, 2, 15, 6>;
using GW_BF_16_23 = GWarpShape<bf16_t, 16, 2, 23, 5>;
using GW_FF_16_15 = GWarpShape<float, 16, 2, 15, 4>;
// backward: two tiles per stage.  B=8 T=2048 D=2560 with the finishing
// reduction: bf16 56.0 us with 15-row sub-chunks (67.7 with 7), fp32 93.7 us.
using GWB_BF_16_15 = GWarpShape<bf16_t, 16, 2, 15, 5>;
using GWB_BF_16_7 = GWarpShape<bf16_t, 16, 2, 7, 8>;
using GWB_FF_16_15 = GWarpShape<float, 16, 2, 15, 3>;

#define F(SH, N) gdir_cfg<SH, true>(N)
#define B(SH, N) gdir_cfg<SH, false>(N)
#define FW(SH, S, N) gwdir_cfg<SH, true>(S, N)
#define BW(SH, S, N) gwdir_cfg<SH, false>(S, N)
const WinVariant kGatedBF16[] = {
    {"gseq_bf16_d64_v1", F(GBF_64_1, 8), B(GBB_64_1, 6)},
    {"gseq_bf16_d64_v2", F(GBF_64_2, 8), B(GBB_64_2, 6)},
    {"gwin_bf16_d32_s8", FW(GWF_BF_32_2_8, 8, 2), BW(GWB_BF_32_2_8_M5, 8, 2)},
    {"gwin_bf16_d32_s8_n3", FW(GWF_BF_32_2_8, 8, 3), BW(GWB_BF_32_2_8_M5, 8, 3)},
    {"gwin_bf16_d32_s8_m4", FW(GWF_BF_32_2_8, 8, 2), BW(GWB_BF_32_2_8_M4, 8, 2)},
    {"gwin_bf16_d32_s16", FW(GWF_BF_32_2_8, 8, 2), BW(GWB_BF_32_2_8, 16, 2)},
    {"gwarp_bf16_l16_r15", gwarp_cfg<GW_BF_16_15>(), gwarp_bwd_cfg<GWB_BF_16_15>()},
    {"gwarp_bf16_l16_r23", gwarp_cfg<GW_BF_16_23>(), gwarp_bwd_cfg<GWB_BF_16_7>()},
};
const WinVariant kGatedF32[] = {
    {"gseq_f32_d32_v1", F(GFF_32_1, 8), B(GFB_32_1, 6)},
    {"gseq_f32_d64_v2", F(GFF_64_2, 6), B(GFB_64_2, 4)},
    {"gwin_f32_d32_s8", FW(GWF_FF_32_1_8, 8, 3), BW(GWB_FF_16_1_8, 16, 2)},
    {"gpipe_f32_w16", gpdir_cfg<GP_FF_16>(), BW(GWB_FF_16_1_8, 16, 2)},
    {"gwarp_f32_l16_r15", gwarp_cfg<GW_FF_16_15>(), gwarp_bwd_cfg<GWB_FF_16_15>()},
};
#undef FW
#undef BW
#undef F
#undef B

}  // namespace

const WinVariant *gwin_variants(int dtype, int *count) {
    if (dtype == 0) {
        *count = sizeof(kGatedF32) / sizeof(kGatedF32[0]);
        return kGatedF32;
    }
    *count = sizeof(kGatedBF16) / sizeof(kGatedBF16[0]);
    return kGatedBF16;
}

int gated_finish_launch(const float *part_eta, int ncol, long long rows, float *grad_eta, const float *part_nu,
                        int nu_rows, int D, float *grad_nu_log, cudaStream_t stream) {
    const unsigned b0 = static_cast<unsigned>((rows + kFinishCols - 1) / kFinishCols);
    const unsigned b1 = static_cast<unsigned>((D + kFinishCols - 1) / kFinishCols);
    if (b0 + b1 == 0) return 0;
    // programmatic dependent launch: the blocks start while the backward
    // drains and wait (griddepcontrol.wait) before reading its partials
    const cudaError_t e = launch_pdl(gated_finish, dim3(b0 + b1), dim3(kFinishCols, kFinishSplit), 0, stream,
                                     part_eta, ncol, rows, grad_eta, part_nu, nu_rows, D, grad_nu_log, b0);
    return e == cudaSuccess ? 0 : -1;
}

int gplain_launch(const WinLaunch &L, int dtype, bool fwd) {
    const int nlb = static_cast<int>((L.D + 127) / 128);
    const unsigned nb = static_cast<unsigned>(nlb * L.B);
    const int T = static_cast<int>(L.T), D = static_cast<int>(L.D);
    if (fwd) {
        if (dtype == 0)
            gplain_fwd<float><<<nb, 128, 0, L.stream>>>(L.eta, L.nu_log, static_cast<const float *>(L.in0),
                                                        static_cast<float *>(L.out0), L.last, T, D, nlb);
        else
            gplain_fwd<bf16_t><<<nb, 128, 0, L.stream>>>(L.eta, L.nu_log, static_cast<const bf16_t *>(L.in0),
                                                         static_cast<bf16_t *>(L.out0), L.last, T, D, nlb);
    } else {
        if (dtype == 0)
            gplain_bwd<float><<<nb, 128, 0, L.stream>>>(L.eta, L.nu_log, static_cast<const float *>(L.in0),
                                                        static_cast<const float *>(L.in1),
                                                        static_cast<float *>(L.out0), L.part_eta, L.part_nu, T, D,
                                                        nlb);
        else
            gplain_bwd<bf16_t><<<nb, 128, 0, L.stream>>>(L.eta, L.nu_log, static_cast<const bf16_t *>(L.in0),
                                                         static_cast<const bf16_t *>(L.in1),
                                                         static_cast<bf16_t *>(L.out0), L.part_eta, L.part_nu, T,
                                                         D, nlb);
    }
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lrscan
