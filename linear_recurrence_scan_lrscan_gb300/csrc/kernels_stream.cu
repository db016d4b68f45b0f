// Instantiations and launchers of the persistent chunk-streaming kernels, and
// their variant table.
#include <mutex>

#include "launch.h"
#include "stream_kernels.cuh"
#include "window_launch.cuh"  // set_smem_attr

namespace lrscan {

namespace {

template <class C, bool BWD, bool EXT>
int launch_stream(const WinLaunch &L, const WinDirCfg &) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = stream_kernel<C, BWD, EXT>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    if (L.grid <= 0) return -1;
    const StreamGeom g = make_stream_geom<C, BWD>();
    // L.maps[0..5]: the inputs in kernel order; L.maps[6..9]: the outputs
    using PL = StreamPlanes<C, BWD>;
    StreamMaps m{};
    for (int i = 0; i < PL::NIN; ++i) m.in[i] = *L.maps[i];
    for (int i = 0; i < PL::NOUT; ++i) m.out[i] = *L.maps[6 + i];
    const cudaError_t e = launch_pdl(fn, dim3(static_cast<unsigned>(L.grid)), dim3(C::THREADS), g.smem_bytes,
                                     L.stream, m, L.last, L.last_i, static_cast<int>(L.T), static_cast<int>(L.D),
                                     L.status, L.timeout_ns, L.sa, L.sx, L.csx);
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
    d.launch = &launch_stream<C, !FWD, false>;
    d.launch_state = &launch_stream<C, !FWD, true>;  // carried state and resets
    return d;
}

// StreamShape<St, DT, V, W, NW, R, S, SR, NSCAN, NB>: two scan warps, two
// chunk buffers, one CTA per SM.  fp32: four summary and four replay warps on
// 32-lane tiles of 32-row windows; forward 512-step chunks (three summary /
// two replay stages) or 256-step ones (more lane groups), backward 256-step
// chunks (two / three stages: its replays trail their summaries by less time,
// so more of their tiles are still in L2).  bf16: eight summary and eight
// replay warps on 32-lane tiles of 32-row windows, forward 1024-step chunks
// (three / two stages), backward 512 (two / three); at B=1 T=2^22 D=64 that
// is 0.30 against 0.32 ms forward and 0.47 against 0.48 ms backward of four
// warps of each kind on 64-row windows, at B=1 T=2^20 D=256 0.29 against 0.32
// and 0.43 against 0.46 ms.  The other bf16 variants keep four of each on
// 64-lane tiles of 32-row windows in 512- or 256-step chunks.
using SF32_C512_F = StreamShape<float, 32, 1, 32, 4, 4, 3, 2, 2, 2>;
using SF32_C256_F = StreamShape<float, 32, 1, 32, 4, 2, 3, 2, 2, 2>;
using SF32_C256_B = StreamShape<float, 32, 1, 32, 4, 2, 2, 3, 2, 2>;
using SBF_D32_F = StreamShape<bf16_t, 32, 1, 32, 8, 4, 3, 2, 2, 2>;
using SBF_D32_B = StreamShape<bf16_t, 32, 1, 32, 8, 2, 2, 3, 2, 2>;
using SBF_D64_F = StreamShape<bf16_t, 64, 2, 32, 4, 4, 3, 3, 2, 2>;
using SBF_D64_B = StreamShape<bf16_t, 64, 2, 32, 4, 4, 3, 2, 2, 2>;
using SBF_D64_C256_F = StreamShape<bf16_t, 64, 2, 32, 4, 2, 3, 3, 2, 2>;
using SBF_D64_C256_B = StreamShape<bf16_t, 64, 2, 32, 4, 2, 3, 2, 2, 2>;

// Complex: four (forward) or six (backward) planes per tile.  The forward
// keeps four summary and four replay warps on 16-row fp32 windows (32-row
// bf16) in 256-step (512) chunks: at B=1 T=2^20 D=64, 256 against 512 steps
// is 0.30 against 0.41 ms, and eight warps of each kind on 8-row windows take
// 0.33 ms.  The backward takes eight of each on 8-row fp32 windows (16-row
// bf16), two summary and two replay stages, in 128-step (256) chunks: at B=1
// T=2^18 D=256, 0.43 against 0.48 ms fp32 and 0.27 against 0.30 ms bf16 of
// four warps of each kind on the forward's windows.
using SC_F32_F = StreamShape<float, 32, 1, 16, 4, 4, 3, 2, 2, 2, true>;
using SC_F32_B = StreamShape<float, 32, 1, 8, 8, 2, 2, 2, 2, 2, true>;
using SC_BF_F = StreamShape<bf16_t, 32, 1, 32, 4, 4, 3, 2, 2, 2, true>;
using SC_BF_B = StreamShape<bf16_t, 32, 1, 16, 8, 2, 2, 2, 2, 2, true>;

const WinVariant kCStreamF32[] = {
    {"cstream_f32_d32", stream_cfg<SC_F32_F, true>(), stream_cfg<SC_F32_B, false>()},
};
const WinVariant kCStreamBF16[] = {
    {"cstream_bf16_d32", stream_cfg<SC_BF_F, true>(), stream_cfg<SC_BF_B, false>()},
};

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

const WinVariant *cstream_variants(int dtype, int *count) {
    *count = 1;
    return dtype == 0 ? kCStreamF32 : kCStreamBF16;
}

const WinVariant *stream_variants(int dtype, int *count) {
    if (dtype == 0) {
        *count = static_cast<int>(sizeof(kStreamF32) / sizeof(kStreamF32[0]));
        return kStreamF32;
    }
    *count = static_cast<int>(sizeof(kStreamBF16) / sizeof(kStreamBF16[0]));
    return kStreamBF16;
}

}  // namespace lrscan
