// Instantiations and launchers of the persistent chunk-streaming kernels, and
// their variant table.
#include <cstdlib>
#include <mutex>

#include "launch.h"
#include "stream_kernels.cuh"
#include "window_launch.cuh"

namespace lrscan {

namespace {

// Dynamic shared memory of one direction: the window kernel's layout (ring,
// barriers, maps, entries, two output buffers) plus one ticket word per stage.
template <class C, bool BWD>
int stream_smem(const WinGeom &g) {
    return win_out_smem(g, BWD ? 2 : 1, 2) + 4 * g.nstage;
}

template <class C, bool BWD>
int launch_stream(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = stream_kernel<C, BWD>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    if (L.grid <= 0) return -1;
    const CUtensorMap &m2 = BWD ? *L.maps[2] : *L.maps[0];
    const CUtensorMap &m3 = BWD ? *L.maps[3] : *L.maps[2];
    const CUtensorMap &m4 = BWD ? *L.maps[4] : *L.maps[2];
    const cudaError_t e = launch_pdl(fn, dim3(static_cast<unsigned>(L.grid)), dim3(cfg.threads),
                                     stream_smem<C, BWD>(g), L.stream, *L.maps[0], *L.maps[1], m2, m3, m4, L.last, g,
                                     L.status, L.timeout_ns, L.sa);
    return e == cudaSuccess ? 0 : -1;
}

template <class C, bool FWD>
WinDirCfg sdir_cfg(int S, int nstage) {
    static_assert(!C::SEQ && !C::PT && !C::EX && C::NIN == (FWD ? 2 : 3), "stream tile shape");
    const WinGeom g = make_win_geom<C>(S, nstage, 1, 1);
    if (S < 2 || S > C::SMAX || S * C::G + 32 > C::MAXT) std::abort();  // table error
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.lane_scan = 1;
    d.exact = 0;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = S * C::G + 32;
    d.smem = stream_smem<C, !FWD>(g);
    d.stage_bytes = g.stage_bytes;
    d.max_resident = C::MINB;  // the register budget of the launch bounds
    d.launch = &launch_stream<C, !FWD>;
    d.launch_state = nullptr;
    return d;
}

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ>: eight sub-chunks of 8 rows
// (64-row windows).  One lane per thread: two CTAs per SM; two lanes per
// thread (64-lane tiles) keep three row tiles in registers and run one CTA per
// SM.
using STF_F32_32 = WinShape<float, 32, 1, 8, 2, 288, 2, false>;
using STB_F32_32 = WinShape<float, 32, 1, 8, 3, 288, 2, false>;
using STF_F32_64 = WinShape<float, 64, 2, 8, 2, 288, 1, false>;
using STB_F32_64 = WinShape<float, 64, 2, 8, 3, 288, 1, false>;
using STF_BF_32 = WinShape<bf16_t, 32, 1, 8, 2, 288, 2, false>;
using STB_BF_32 = WinShape<bf16_t, 32, 1, 8, 3, 288, 2, false>;
using STF_BF_64 = WinShape<bf16_t, 64, 2, 8, 2, 288, 1, false>;
using STB_BF_64 = WinShape<bf16_t, 64, 2, 8, 3, 288, 1, false>;

#define F(SH, S, N) sdir_cfg<SH, true>(S, N)
#define B(SH, S, N) sdir_cfg<SH, false>(S, N)
const WinVariant kStreamF32[] = {
    {"stream_f32_d32_s8", F(STF_F32_32, 8, 4), B(STB_F32_32, 8, 3)},
    {"stream_f32_d64_s8", F(STF_F32_64, 8, 4), B(STB_F32_64, 8, 3)},
};
const WinVariant kStreamBF16[] = {
    {"stream_bf16_d32_s8", F(STF_BF_32, 8, 4), B(STB_BF_32, 8, 3)},
    {"stream_bf16_d64_s8", F(STF_BF_64, 8, 4), B(STB_BF_64, 8, 3)},
};
#undef F
#undef B

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
