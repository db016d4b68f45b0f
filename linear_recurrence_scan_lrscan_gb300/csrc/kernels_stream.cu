// Instantiations and launchers of the persistent chunk-streaming kernels, and
// their variant table.
#include <mutex>

#include "launch.h"
#include "stream_kernels.cuh"
#include "window_launch.cuh"  // set_smem_attr

namespace lrscan {

namespace {

template <class C, bool BWD>
int launch_stream(const WinLaunch &L, const WinDirCfg &) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = stream_kernel<C, BWD>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    if (L.grid <= 0) return -1;
    const StreamGeom g = make_stream_geom<C, BWD>();
    // maps[3], maps[4]: the outputs (out; grad_a, grad_b)
    const cudaError_t e =
        launch_pdl(fn, dim3(static_cast<unsigned>(L.grid)), dim3(C::THREADS), g.smem_bytes, L.stream, *L.maps[0],
                   *L.maps[1], BWD ? *L.maps[2] : *L.maps[0], *L.maps[3], BWD ? *L.maps[4] : *L.maps[3], L.last,
                   static_cast<int>(L.T), static_cast<int>(L.D), L.status, L.timeout_ns, L.sa);
    return e == cudaSuccess ? 0 : -1;
}

// rows_per_window (w) = rows of a window, subchunks (s) = windows per chunk
// (a chunk is s * w steps); stages counts both rings of a CTA.
template <class C, bool FWD>
WinDirCfg stream_cfg() {
    const StreamGeom g = make_stream_geom<C, !FWD>();
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
    d.launch = &launch_stream<C, !FWD>;
    d.launch_state = nullptr;
    return d;
}

// StreamShape<St, DT, V, W, NW, R, S, SR, NSCAN, NB>: four summary and four
// replay warps, two scan warps, two chunk buffers, one CTA per SM.  fp32:
// 32-lane tiles of 32-row windows; forward 512-step chunks (three summary /
// two replay stages) or 256-step ones (more lane groups), backward 256-step
// chunks (two / three stages: its replays trail their summaries by less time,
// so more of their tiles are still in L2).  bf16: 32-lane tiles of 64-row
// windows (forward 1024-step chunks, backward 512), or 64-lane tiles of 32-row
// windows in 512- or 256-step chunks.
using SF32_C512_F = StreamShape<float, 32, 1, 32, 4, 4, 3, 2, 2, 2>;
using SF32_C256_F = StreamShape<float, 32, 1, 32, 4, 2, 3, 2, 2, 2>;
using SF32_C256_B = StreamShape<float, 32, 1, 32, 4, 2, 2, 3, 2, 2>;
using SBF_D32_F = StreamShape<bf16_t, 32, 1, 64, 4, 4, 3, 3, 2, 2>;
using SBF_D32_B = StreamShape<bf16_t, 32, 1, 64, 4, 2, 2, 3, 2, 2>;
using SBF_D64_F = StreamShape<bf16_t, 64, 2, 32, 4, 4, 3, 3, 2, 2>;
using SBF_D64_B = StreamShape<bf16_t, 64, 2, 32, 4, 4, 3, 2, 2, 2>;
using SBF_D64_C256_F = StreamShape<bf16_t, 64, 2, 32, 4, 2, 3, 3, 2, 2>;
using SBF_D64_C256_B = StreamShape<bf16_t, 64, 2, 32, 4, 2, 3, 2, 2, 2>;

const WinVariant kStreamF32[] = {
    {"stream_f32_d32", stream_cfg<SF32_C512_F, true>(), stream_cfg<SF32_C256_B, false>()},
    {"stream_f32_d32_c256", stream_cfg<SF32_C256_F, true>(), stream_cfg<SF32_C256_B, false>()},
};
const WinVariant kStreamBF16[] = {
    {"stream_bf16_d32", stream_cfg<SBF_D32_F, true>(), stream_cfg<SBF_D32_B, false>()},
    {"stream_bf16_d64", stream_cfg<SBF_D64_F, true>(), stream_cfg<SBF_D64_B, false>()},
    {"stream_bf16_d64_c256", stream_cfg<SBF_D64_C256_F, true>(), stream_cfg<SBF_D64_C256_B, false>()},
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
