// Instantiations and launchers of the time-tiled (TMA) kernels, and the table
// of tile variants the host dispatcher chooses from.
#include "launch.h"
#include "window_kernels.cuh"

#include <cstdlib>

namespace lrscan {

namespace {

// Dynamic shared memory above 48 KB has to be opted into, per kernel and
// device; the largest size any variant asks for is set once.
int set_smem_attr(const void *fn, int dev, unsigned long long *mask, std::mutex *mu) {
    std::lock_guard<std::mutex> lk(*mu);
    if (dev < 64 && ((*mask >> dev) & 1ull)) return 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
        return -1;
    if (dev < 64) *mask |= 1ull << dev;
    return 0;
}

template <class C>
int launch_win_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = win_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], static_cast<typename C::St *>(L.out0), L.last,
                                     g, L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_win_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = win_bwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], *L.maps[2],
                                     static_cast<typename C::St *>(L.out0), static_cast<typename C::St *>(L.out1), g,
                                     L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C, bool FWD>
WinDirCfg dir_cfg(int S, int nstage) {
    const WinGeom g = make_win_geom<C>(S, nstage, 1, 1);
    if (C::SEQ != (S == 1) || S > C::SMAX) std::abort();  // table error: S out of the shape's range
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.lane_scan = (!C::SEQ && !C::PT) ? 1 : 0;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = S * C::G + 32;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) {
        static_assert(C::NIN == 2, "forward tiles: a, b");
        d.launch = &launch_win_fwd<C>;
    } else {
        static_assert(C::NIN == 3, "backward tiles: a, out, grad_out");
        d.launch = &launch_win_bwd<C>;
    }
    return d;
}

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ>
// Sequential shapes (S = 1): L rows per window streamed from shared memory.
using SBF_64_2_32 = WinShape<bf16_t, 64, 2, 32, 2, 64, 1, true>;
using SBF_128_2_32 = WinShape<bf16_t, 128, 2, 32, 2, 96, 1, true>;
using SBF_128_4_32 = WinShape<bf16_t, 128, 4, 32, 2, 64, 1, true>;
using SBB_64_2_32 = WinShape<bf16_t, 64, 2, 32, 3, 64, 1, true>;
using SBF_32_1_32 = WinShape<bf16_t, 32, 1, 32, 2, 64, 1, true>;
using SBF_64_1_32 = WinShape<bf16_t, 64, 1, 32, 2, 96, 1, true>;
using SBB_32_1_32 = WinShape<bf16_t, 32, 1, 32, 3, 64, 1, true>;
using SBB_64_1_32 = WinShape<bf16_t, 64, 1, 32, 3, 96, 1, true>;
using SBB_128_2_32 = WinShape<bf16_t, 128, 2, 32, 3, 96, 1, true>;
using SBB_128_4_16 = WinShape<bf16_t, 128, 4, 16, 3, 64, 1, true>;
using SFF_32_1_32 = WinShape<float, 32, 1, 32, 2, 64, 1, true>;
using SFF_64_2_16 = WinShape<float, 64, 2, 16, 2, 64, 1, true>;
using SFF_64_1_32 = WinShape<float, 64, 1, 32, 2, 96, 1, true>;
using SFF_128_4_8 = WinShape<float, 128, 4, 8, 2, 64, 1, true>;
using SFB_32_1_32 = WinShape<float, 32, 1, 32, 3, 64, 1, true>;
using SFB_64_2_16 = WinShape<float, 64, 2, 16, 3, 64, 1, true>;
using SFB_64_1_32 = WinShape<float, 64, 1, 32, 3, 96, 1, true>;
using SFB_128_4_8 = WinShape<float, 128, 4, 8, 3, 64, 1, true>;
// Windowed shapes (S > 1): each thread holds L rows of its sub-chunk in registers.
using BF_64_2_8 = WinShape<bf16_t, 64, 2, 8, 2, 288, 3, false>;
using BF_32_2_8 = WinShape<bf16_t, 32, 2, 8, 2, 288, 3, false>;
using BF_128_4_8 = WinShape<bf16_t, 128, 4, 8, 2, 288, 1, false>;
using BF_32_1_8 = WinShape<bf16_t, 32, 1, 8, 2, 544, 1, false>;
using BB_64_2_8 = WinShape<bf16_t, 64, 2, 8, 3, 288, 2, false>;
using BB_32_2_8 = WinShape<bf16_t, 32, 2, 8, 3, 288, 2, false>;
// per-thread-prefix shapes (parallel fold, short critical path)
using PF_32_1_8 = WinShape<float, 32, 1, 8, 2, 544, 1, false, true>;
using PFB_32_1_8 = WinShape<float, 32, 1, 8, 3, 544, 1, false, true>;
using PF_16_1_8 = WinShape<float, 16, 1, 8, 2, 544, 1, false, true>;
using PFB_16_1_8 = WinShape<float, 16, 1, 8, 3, 544, 1, false, true>;
using BB_128_4_4 = WinShape<bf16_t, 128, 4, 4, 3, 288, 2, false>;
using BB_32_1_8 = WinShape<bf16_t, 32, 1, 8, 3, 544, 1, false>;
using FF_16_1_8 = WinShape<float, 16, 1, 8, 2, 544, 1, false>;
using FF_32_1_8 = WinShape<float, 32, 1, 8, 2, 544, 1, false>;
using FF_64_2_8 = WinShape<float, 64, 2, 8, 2, 288, 2, false>;
using FB_16_1_8 = WinShape<float, 16, 1, 8, 3, 544, 1, false>;
using FB_32_1_8 = WinShape<float, 32, 1, 8, 3, 544, 1, false>;
using FB_64_2_8 = WinShape<float, 64, 2, 8, 3, 288, 1, false>;
// L = 16: half the sub-chunks (and half the in-CTA prefix work) per window row
using WF_32_1_16 = WinShape<float, 32, 1, 16, 2, 288, 1, false>;
using WF_16_1_16 = WinShape<float, 16, 1, 16, 2, 288, 1, false>;
using WFB_32_1_16 = WinShape<float, 32, 1, 16, 3, 288, 1, false>;
using WFB_16_1_16 = WinShape<float, 16, 1, 16, 3, 288, 1, false>;
using WBF_32_2_16 = WinShape<bf16_t, 32, 2, 16, 2, 288, 1, false>;
using WBF_64_2_16 = WinShape<bf16_t, 64, 2, 16, 2, 288, 1, false>;
using WBB_32_2_16 = WinShape<bf16_t, 32, 2, 16, 3, 288, 1, false>;
using WBB_64_2_16 = WinShape<bf16_t, 64, 2, 16, 3, 288, 1, false>;

#define F(SH, S, N) dir_cfg<SH, true>(S, N)
#define B(SH, S, N) dir_cfg<SH, false>(S, N)


const WinVariant kSeqBF16[] = {
    {"seq_bf16_d64", F(SBF_64_2_32, 1, 8), B(SBB_64_2_32, 1, 6)},
    {"seq_bf16_d128", F(SBF_128_2_32, 1, 4), B(SBB_128_2_32, 1, 4)},
    {"seq_bf16_d64_s9", F(SBF_64_2_32, 1, 9), B(SBB_64_2_32, 1, 6)},
    {"seq_bf16_d128_v4", F(SBF_128_4_32, 1, 6), B(SBB_128_4_16, 1, 6)},
    {"seq_bf16_d32_v1", F(SBF_32_1_32, 1, 8), B(SBB_32_1_32, 1, 6)},
    {"seq_bf16_d64_v1", F(SBF_64_1_32, 1, 8), B(SBB_64_1_32, 1, 6)},
};
const WinVariant kWinBF16[] = {
    {"win_bf16_d32_s16", F(BF_32_2_8, 16, 3), B(BB_32_2_8, 16, 4)},
    {"win_bf16_d64_s8", F(BF_64_2_8, 8, 4), B(BB_64_2_8, 8, 3)},
    {"win_bf16_d32_s16_n2", F(BF_32_2_8, 16, 2), B(BB_32_2_8, 16, 2)},
    {"win_bf16_d32_s16_n4", F(BF_32_2_8, 16, 4), B(BB_32_2_8, 16, 3)},
    {"win_bf16_d32_l16_s8", F(WBF_32_2_16, 8, 4), B(WBB_32_2_16, 8, 4)},
};
const WinVariant kSeqF32[] = {
    {"seq_f32_d32", F(SFF_32_1_32, 1, 8), B(SFB_32_1_32, 1, 6)},
    {"seq_f32_d64", F(SFF_64_2_16, 1, 8), B(SFB_64_2_16, 1, 6)},
    {"seq_f32_d64_v1", F(SFF_64_1_32, 1, 4), B(SFB_64_1_32, 1, 4)},
    {"seq_f32_d128", F(SFF_128_4_8, 1, 8), B(SFB_128_4_8, 1, 6)},
};
const WinVariant kWinF32[] = {
    {"win_f32_d32_s16_pt", F(PF_32_1_8, 16, 4), B(PFB_32_1_8, 16, 3)},
    {"win_f32_d16_s16", F(FF_16_1_8, 16, 4), B(FB_16_1_8, 16, 4)},
    {"win_f32_d32_s16", F(FF_32_1_8, 16, 4), B(FB_32_1_8, 16, 3)},
    {"win_f32_d16_s16_pt", F(PF_16_1_8, 16, 4), B(PFB_16_1_8, 16, 4)},
    {"win_f32_d64_s8", F(FF_64_2_8, 8, 4), B(FB_64_2_8, 8, 3)},
    {"win_f32_d32_s8_pt", F(PF_32_1_8, 8, 8), B(PFB_32_1_8, 8, 6)},
};

#undef F
#undef B


}  // namespace

const WinVariant *win_variants(int path, int dtype, int *count) {
    if (path == kPathSeq) {
        if (dtype == 0) { *count = sizeof(kSeqF32) / sizeof(kSeqF32[0]); return kSeqF32; }
        *count = sizeof(kSeqBF16) / sizeof(kSeqBF16[0]);
        return kSeqBF16;
    }
    if (dtype == 0) { *count = sizeof(kWinF32) / sizeof(kWinF32[0]); return kWinF32; }
    *count = sizeof(kWinBF16) / sizeof(kWinBF16[0]);
    return kWinBF16;
}

}  // namespace lrscan
