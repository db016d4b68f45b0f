// Instantiations and launchers of the persistent chunk-streaming kernels, and
// their variant table.
#include <cstdlib>
#include <mutex>

#include "launch.h"
#include "stream_kernels.cuh"
#include "stream_split_kernels.cuh"
#include "window_launch.cuh"  // set_smem_attr

namespace lrscan {

namespace {

template <class C, bool BWD>
int launch_stream(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = stream_kernel<C, BWD>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    if (L.grid <= 0) return -1;
    using St = typename C::St;
    const StreamGeom g = make_stream_geom<C, BWD ? 3 : 2>(cfg.nstage);
    const cudaError_t e =
        launch_pdl(fn, dim3(static_cast<unsigned>(L.grid)), dim3(C::THREADS), g.smem_bytes, L.stream, *L.maps[0],
                   *L.maps[1], BWD ? *L.maps[2] : *L.maps[0], static_cast<St *>(L.out0), static_cast<St *>(L.out1),
                   L.last, static_cast<int>(L.T), static_cast<int>(L.D), cfg.nstage, L.status, L.timeout_ns, L.sa);
    return e == cudaSuccess ? 0 : -1;
}

// rows_per_window (w) = rows of one window warp, subchunks (s) = window warps
// per chunk: a chunk is s * w steps.
// nstage is 2 * NWC: window warp w owns stages w (summary tiles) and
// NWC + w (replay tiles), issues their copies itself and alone waits on them,
// so each of its parity waits is one phase past the last one it saw complete.
template <class C, bool FWD>
WinDirCfg sdir_cfg(int nstage) {
    if (nstage != 2 * C::NWC) std::abort();  // table error
    const StreamGeom g = make_stream_geom<C, FWD ? 2 : 3>(nstage);
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::W;
    d.s = C::NWC;
    d.lane_scan = 1;
    d.exact = 0;
    d.w = C::W;
    d.nstage = nstage;
    d.threads = C::THREADS;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.stage_bytes;
    d.max_resident = C::MINB;
    d.launch = &launch_stream<C, !FWD>;
    d.launch_state = nullptr;
    return d;
}

template <class C, bool BWD>
int launch_split(const WinLaunch &L, const WinDirCfg &) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = stream_split_kernel<C, BWD>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    if (L.grid <= 0) return -1;
    const SplitGeom g = make_split_geom<C, BWD>();
    // maps[3], maps[4]: the outputs (out; grad_a, grad_b)
    const cudaError_t e =
        launch_pdl(fn, dim3(static_cast<unsigned>(L.grid)), dim3(C::THREADS), g.smem_bytes, L.stream, *L.maps[0],
                   *L.maps[1], BWD ? *L.maps[2] : *L.maps[0], *L.maps[3], BWD ? *L.maps[4] : *L.maps[3], L.last,
                   static_cast<int>(L.T), static_cast<int>(L.D), L.status, L.timeout_ns, L.sa);
    return e == cudaSuccess ? 0 : -1;
}

// Split-role tiles: rows_per_window (w) = rows of a window, subchunks (s) =
// windows per chunk (a chunk is s * w steps); stages counts both rings.
template <class C, bool FWD>
WinDirCfg split_cfg() {
    const SplitGeom g = make_split_geom<C, !FWD>();
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::W;
    d.s = C::NWIN;
    d.lane_scan = 1;
    d.exact = 0;
    d.w = C::W;
    d.nstage = C::NW * (C::S + C::SR);
    d.threads = C::THREADS;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.rstage_bytes;
    d.max_resident = 1;
    d.ws_unset = 1;
    d.launch = &launch_split<C, !FWD>;
    d.launch_state = nullptr;
    return d;
}

// SplitShape<St, DT, V, W, NW, R, S, SR, NSCAN, NB>: four summary and four
// replay warps over 32-row windows, four windows each per 512-step chunk,
// S summary and SR replay stages per warp, two scan warps, two chunk buffers;
// one CTA per SM.
using PF32_S3R3 = SplitShape<float, 32, 1, 32, 4, 4, 3, 3, 2, 2>;
using PF32_S3R2 = SplitShape<float, 32, 1, 32, 4, 4, 3, 2, 2, 2>;
using PF32_S2R3 = SplitShape<float, 32, 1, 32, 4, 4, 2, 3, 2, 2>;
using PBF64_S3R3 = SplitShape<bf16_t, 64, 2, 32, 4, 4, 3, 3, 2, 2>;
using PBF64_S3R2 = SplitShape<bf16_t, 64, 2, 32, 4, 4, 3, 2, 2, 2>;

// StreamShape<St, DT, V, W, NWC, MINB>: eight window warps (256-step chunks of
// 32-row windows; 128-step chunks of 16-row windows for 64-lane fp32 tiles),
// two ring stages per window warp; one CTA per SM, two for 32-lane bf16
// tiles.  A thread owns V lanes of its warp's rows.
using SF32_32 = StreamShape<float, 32, 1, 32, 8, 1>;
using SF32_64 = StreamShape<float, 64, 2, 16, 8, 1>;
using SBF_32 = StreamShape<bf16_t, 32, 1, 32, 8, 2>;
using SBF_64 = StreamShape<bf16_t, 64, 2, 32, 8, 1>;

const WinVariant kStreamF32[] = {
    {"stream_f32_d32", sdir_cfg<SF32_32, true>(16), sdir_cfg<SF32_32, false>(16)},
    {"stream_f32_d64", sdir_cfg<SF32_64, true>(16), sdir_cfg<SF32_64, false>(16)},
    {"stream_split_f32_d32", split_cfg<PF32_S3R3, true>(), split_cfg<PF32_S3R2, false>()},
    {"stream_split_f32_d32_b", split_cfg<PF32_S3R2, true>(), split_cfg<PF32_S2R3, false>()},
};
const WinVariant kStreamBF16[] = {
    {"stream_bf16_d32", sdir_cfg<SBF_32, true>(16), sdir_cfg<SBF_32, false>(16)},
    {"stream_bf16_d64", sdir_cfg<SBF_64, true>(16), sdir_cfg<SBF_64, false>(16)},
    {"stream_split_bf16_d64", split_cfg<PBF64_S3R3, true>(), split_cfg<PBF64_S3R2, false>()},
};

}  // namespace

const WinVariant *stream_variants(int dtype, int *count) {
    if (dtype == 0) {
        *count = static_cast<int>(sizeof(kStreamF32) / sizeof(kStreamF32[0]));
        return kStreamF32;
    }
    *count = static_cast<int>(sizeof(kStreamBF16) / sizeof(kStreamBF16[0]));
    return kStreamBF16;
}

}  // namespace lrscan
