// Launchers of the complex tiled kernels, templated on the compiled shape and
// on EXT (carried state and segment resets).  The plain launchers are
// instantiated in kernels_complex.cu, the EXT ones in kernels_complex_state.cu.
#pragma once

#include "complex_kernels.cuh"
#include "window_launch.cuh"

namespace lrscan {

// rows staged in registers per step of a full window
template <class C> constexpr int kStageRowsFwd = C::L < 16 ? C::L : 16;
template <class C> constexpr int kStageRowsBwd = C::L < 8 ? C::L : 8;

template <class C, bool EXT>
int launch_cwin_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwin_fwd_kernel<C, kStageRowsFwd<C>, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(1, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    using St = typename C::St;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3],
                                     static_cast<St *>(L.out0), static_cast<St *>(L.out1), L.last, L.last_i, g,
                                     L.status, L.timeout_ns, L.csx);
    return e == cudaSuccess ? 0 : -1;
}

template <class C, bool EXT>
int launch_cwinw_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwinw_fwd_kernel<C, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_cwin_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads),
                                     win_out_smem(g, 2), L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3],
                                     *L.maps[4], *L.maps[5], L.last, L.last_i, g, L.status, L.timeout_ns, L.csx);
    return e == cudaSuccess ? 0 : -1;
}

template <class C, bool EXT>
int launch_cwin_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwin_bwd_kernel<C, kStageRowsBwd<C>, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(1, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    using St = typename C::St;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3], *L.maps[4],
                                     *L.maps[5], static_cast<St *>(L.out0), static_cast<St *>(L.out1),
                                     static_cast<St *>(L.out2), static_cast<St *>(L.out3), g, L.status,
                                     L.timeout_ns, L.csx);
    return e == cudaSuccess ? 0 : -1;
}

template <class C, bool EXT>
int launch_cwinw_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwinw_bwd_kernel<C, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_cwin_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads),
                                     win_out_smem(g, 4, 1), L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3],
                                     *L.maps[4], *L.maps[5], *L.maps[6], *L.maps[7], *L.maps[8], *L.maps[9], g,
                                     L.status, L.timeout_ns, L.csx);
    return e == cudaSuccess ? 0 : -1;
}

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ> of the complex tile variants.
// Windowed (S sub-chunks of L rows, lane scan):
using CWF_BF_32_1_8 = WinShape<bf16_t, 32, 1, 8, 4, 288, 2, false>;
using CWF_BF_32_2_8 = WinShape<bf16_t, 32, 2, 8, 4, 288, 2, false>;
using CWF_FF_32_1_8 = WinShape<float, 32, 1, 8, 4, 288, 2, false>;
// 4-row sub-chunks, five CTAs per SM: every CTA of a 640-tile launch resident
using CWF_BF_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 4, 160, 5, false>;
using CWB_BF_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 6, 160, 5, false>;
// Sequential:
using CBF_64_1_32 = WinShape<bf16_t, 64, 1, 32, 4, 96, 1, true>;
using CBB_64_1_32 = WinShape<bf16_t, 64, 1, 32, 6, 96, 1, true>;
using CBF_64_2_32 = WinShape<bf16_t, 64, 2, 32, 4, 64, 1, true>;
using CBB_64_2_16 = WinShape<bf16_t, 64, 2, 16, 6, 64, 1, true>;
using CBF_32_1_32 = WinShape<bf16_t, 32, 1, 32, 4, 64, 1, true>;
using CBB_32_1_32 = WinShape<bf16_t, 32, 1, 32, 6, 64, 1, true>;
using CFF_32_1_32 = WinShape<float, 32, 1, 32, 4, 64, 1, true>;
using CFB_32_1_32 = WinShape<float, 32, 1, 32, 6, 64, 1, true>;
using CFF_64_2_16 = WinShape<float, 64, 2, 16, 4, 64, 1, true>;
using CFB_64_2_16 = WinShape<float, 64, 2, 16, 6, 64, 1, true>;
using CFF_64_1_16 = WinShape<float, 64, 1, 16, 4, 96, 1, true>;
using CFB_64_1_16 = WinShape<float, 64, 1, 16, 6, 96, 1, true>;

#define LRSCAN_CSEQ_FWD_SHAPES(X) X(CBF_64_1_32) X(CBF_64_2_32) X(CBF_32_1_32) X(CFF_32_1_32) X(CFF_64_2_16) X(CFF_64_1_16)
#define LRSCAN_CSEQ_BWD_SHAPES(X) X(CBB_64_1_32) X(CBB_64_2_16) X(CBB_32_1_32) X(CFB_32_1_32) X(CFB_64_2_16) X(CFB_64_1_16)
#define LRSCAN_CWIN_FWD_SHAPES(X) X(CWF_BF_32_1_8) X(CWF_BF_32_2_8) X(CWF_FF_32_1_8) X(CWF_BF_32_2_4_M5)
#define LRSCAN_CWIN_BWD_SHAPES(X) X(CWB_BF_32_2_4_M5)

}  // namespace lrscan
