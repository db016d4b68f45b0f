// Instantiations and launchers of the single-pass look-back kernels, and
// their tile variant table.
#include <cstdlib>

#include "lookback_kernels.cuh"
#include "window_launch.cuh"

namespace lrscan {

namespace {

template <class C>
int launch_lb_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = lb_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    // one stage: each CTA loads exactly one window
    const WinGeom g = make_win_geom<C>(cfg.s, 1, static_cast<int>(L.T), static_cast<int>(L.D));
    const int lanes_per_row = static_cast<int>((L.D + C::DT - 1) / C::DT);
    LookbackArgs lb{};
    lb.ticket = L.lb_ticket;
    lb.flags = L.lb_flags;
    lb.maps = L.lb_maps;
    lb.incl = L.lb_incl;
    lb.nlt = static_cast<int>(L.B) * lanes_per_row;
    const long long ctas = static_cast<long long>(lb.nlt) * g.nwin;
    const cudaError_t e = launch_pdl(fn, dim3(static_cast<unsigned>(ctas)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], static_cast<typename C::St *>(L.out0), L.last,
                                     g, lb, lanes_per_row, L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
WinDirCfg lb_cfg(int S) {
    static_assert(!C::SEQ && !C::PT && C::DT == 32, "look-back tiles: lane scan, 32 lanes");
    if (S > C::SMAX) std::abort();  // table error
    const WinGeom g = make_win_geom<C>(S, 1, 1, 1);
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.lane_scan = 1;
    d.w = g.W;
    d.nstage = 1;
    d.threads = S * C::G + 32;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.stage_bytes;
    d.launch = &launch_lb_fwd<C>;
    return d;
}

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ>
using LBF_F32 = WinShape<float, 32, 1, 8, 2, 288, 3, false>;
using LBF_BF16 = WinShape<bf16_t, 32, 2, 8, 2, 160, 5, false>;

const WinVariant kLbF32[] = {
    {"lb_f32_d32_s8", lb_cfg<LBF_F32>(8), WinDirCfg{}},
    {"lb_f32_d32_s4", lb_cfg<LBF_F32>(4), WinDirCfg{}},
};
const WinVariant kLbBF16[] = {
    {"lb_bf16_d32_s8", lb_cfg<LBF_BF16>(8), WinDirCfg{}},
    {"lb_bf16_d32_s4", lb_cfg<LBF_BF16>(4), WinDirCfg{}},
};

}  // namespace

const WinVariant *lb_variants(int dtype, int *count) {
    if (dtype == 0) {
        *count = sizeof(kLbF32) / sizeof(kLbF32[0]);
        return kLbF32;
    }
    *count = sizeof(kLbBF16) / sizeof(kLbBF16[0]);
    return kLbBF16;
}

}  // namespace lrscan
