// Launchers of the time-tiled kernels, templated on the compiled shape and on
// EXT (carried state and segment resets).  The plain launchers are
// instantiated in kernels_window.cu, the EXT ones in kernels_window_state.cu.
#pragma once

#include <mutex>

#include "launch.h"
#include "wavefront_kernels.cuh"
#include "window_kernels.cuh"

namespace lrscan {

// Dynamic shared memory above 48 KB has to be opted into, per kernel and
// device; the largest size any variant asks for is set once.
inline int set_smem_attr(const void *fn, int dev, unsigned long long *mask, std::mutex *mu) {
    std::lock_guard<std::mutex> lk(*mu);
    if (dev < 64 && ((*mask >> dev) & 1ull)) return 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
        return -1;
    if (dev < 64) *mask |= 1ull << dev;
    return 0;
}

template <class C, bool EXT>
int launch_win_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = win_fwd_kernel<C, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const int smem = win_staged<C>() ? win_out_smem(g) : g.smem_bytes;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), smem, L.stream,
                                     *L.maps[0], *L.maps[1], *L.maps[2], static_cast<typename C::St *>(L.out0),
                                     L.last, g, L.status, L.timeout_ns, L.sx);
    return e == cudaSuccess ? 0 : -1;
}

template <class C, bool EXT>
int launch_win_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = win_bwd_kernel<C, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const int smem = win_staged<C>() ? win_out_smem(g, 2) : g.smem_bytes;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), smem, L.stream,
                                     *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3], *L.maps[4],
                                     static_cast<typename C::St *>(L.out0), static_cast<typename C::St *>(L.out1), g,
                                     L.status, L.timeout_ns, L.sx);
    return e == cudaSuccess ? 0 : -1;
}

// Wavefront exact tiles: S consumer warps and a producer warp; forward maps
// a, b, out; backward a, out, grad_out, grad_a, grad_b; three output buffers.
template <class C, bool BWD, bool EXT>
int launch_wfx(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = wfx_kernel<C, BWD, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const CUtensorMap &m3 = BWD ? *L.maps[3] : *L.maps[2];
    const CUtensorMap &m4 = BWD ? *L.maps[4] : *L.maps[2];
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads),
                                     win_out_smem(g, BWD ? 2 : 1, 3), L.stream, *L.maps[0], *L.maps[1], *L.maps[2], m3,
                                     m4, L.last, g, L.status, L.timeout_ns, L.sx);
    return e == cudaSuccess ? 0 : -1;
}

}  // namespace lrscan
