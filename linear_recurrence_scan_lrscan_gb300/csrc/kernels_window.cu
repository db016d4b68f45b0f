// Instantiations and launchers of the time-tiled (TMA) kernels, and the table
// of tile variants the host dispatcher chooses from.
#include "window_launch.cuh"
#include "window_shapes.h"

#include <cstdlib>

namespace lrscan {

#define LRSCAN_EXTERN_FWD(SH) extern template int launch_win_fwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_EXTERN_BWD(SH) extern template int launch_win_bwd<SH, true>(const WinLaunch &, const WinDirCfg &);
LRSCAN_WIN_FWD_SHAPES(LRSCAN_EXTERN_FWD)
LRSCAN_WIN_BWD_SHAPES(LRSCAN_EXTERN_BWD)
#undef LRSCAN_EXTERN_FWD
#undef LRSCAN_EXTERN_BWD
#define LRSCAN_EXTERN_WF(SH) extern template int launch_wfx<SH, false, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_EXTERN_WB(SH) extern template int launch_wfx<SH, true, true>(const WinLaunch &, const WinDirCfg &);
LRSCAN_WFX_FWD_SHAPES(LRSCAN_EXTERN_WF)
LRSCAN_WFX_BWD_SHAPES(LRSCAN_EXTERN_WB)
#undef LRSCAN_EXTERN_WF
#undef LRSCAN_EXTERN_WB

namespace {

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
    d.exact = (C::SEQ || C::EX) ? 1 : 0;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = S * C::G + 32;
    d.smem = win_staged<C>() ? win_out_smem(g, FWD ? 1 : 2) : g.smem_bytes;  // plus the output staging buffers
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) {
        static_assert(C::NIN == 2, "forward tiles: a, b");
        d.launch = &launch_win_fwd<C, false>;
        d.launch_state = &launch_win_fwd<C, true>;
    } else {
        static_assert(C::NIN == 3, "backward tiles: a, out, grad_out");
        d.launch = &launch_win_bwd<C, false>;
        d.launch_state = &launch_win_bwd<C, true>;
    }
    return d;
}

// Wavefront exact tiles: S consumer warps (one per sub-chunk) plus the producer.
template <class C, bool FWD>
WinDirCfg wdir_cfg(int S, int nstage) {
    static_assert(C::EX && C::G == 32, "wavefront shape: one warp per sub-chunk");
    const WinGeom g = make_win_geom<C>(S, nstage, 1, 1);
    if (S < 2 || S * 32 + 32 > C::MAXT) std::abort();  // table error
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.exact = 1;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = S * 32 + 32;
    d.smem = win_out_smem(g, FWD ? 1 : 2, 3);
    d.stage_bytes = g.stage_bytes;
    d.launch = &launch_wfx<C, !FWD, false>;
    d.launch_state = &launch_wfx<C, !FWD, true>;
    return d;
}

#define F(SH, S, N) dir_cfg<SH, true>(S, N)
#define B(SH, S, N) dir_cfg<SH, false>(S, N)
#define WF(SH, S, N) wdir_cfg<SH, true>(S, N)
#define WB(SH, S, N) wdir_cfg<SH, false>(S, N)


const WinVariant kSeqBF16[] = {
    {"seq_bf16_d64", F(SBF_64_2_32, 1, 8), B(SBB_64_2_32, 1, 6)},
    {"seq_bf16_d128", F(SBF_128_2_32, 1, 4), B(SBB_128_2_32, 1, 4)},
    {"seq_bf16_d64_s9", F(SBF_64_2_32, 1, 9), B(SBB_64_2_32, 1, 6)},
    {"seq_bf16_d128_v4", F(SBF_128_4_32, 1, 6), B(SBB_128_4_16, 1, 6)},
    {"seq_bf16_d32_v1", F(SBF_32_1_32, 1, 8), B(SBB_32_1_32, 1, 6)},
    {"seq_bf16_d64_v1", F(SBF_64_1_32, 1, 8), B(SBB_64_1_32, 1, 6)},
    // shallower rings: four 128-lane CTAs resident per SM
    {"seq_bf16_d128_v4_n3", F(SBF_128_4_32, 1, 3), B(SBB_128_4_16, 1, 3)},
    {"seq_bf16_d128_n2", F(SBF_128_2_32, 1, 2), B(SBB_128_2_32, 1, 2)},
    {"seq_bf16_d128_n3", F(SBF_128_2_32, 1, 3), B(SBB_128_2_32, 1, 3)},
};
const WinVariant kWinBF16[] = {
    {"win_bf16_d32_s16", F(BF_32_2_8, 16, 3), B(BB_32_2_8, 16, 4)},
    {"win_bf16_d64_s8", F(BF_64_2_8, 8, 4), B(BB_64_2_8, 8, 3)},
    {"win_bf16_d32_s16_n2", F(BF_32_2_8, 16, 2), B(BB_32_2_8, 16, 2)},
    {"win_bf16_d32_s16_n4", F(BF_32_2_8, 16, 4), B(BB_32_2_8, 16, 3)},
    {"win_bf16_d32_l16_s8", F(WBF_32_2_16, 8, 4), B(WBB_32_2_16, 8, 4)},
    {"win_bf16_d32_s8_m5", F(BF_32_2_8_M5, 8, 3), B(BB_32_2_8_M5, 8, 3)},
    {"win_bf16_d32_s8_m5_n2", F(BF_32_2_8_M5, 8, 2), B(BB_32_2_8_M5, 8, 2)},
    {"win_bf16_d32_s4_m8", F(BF_32_2_8_M8, 4, 4), B(BB_32_2_8_M8, 4, 3)},
    {"win_bf16_d32_s4_m8_n2", F(BF_32_2_8_M8, 4, 2), B(BB_32_2_8_M8, 4, 2)},
    {"win_bf16_d32_l4_s12_m5", F(BF_32_2_4_M5, 12, 2), B(BB_32_2_4_M5, 12, 2)},
    {"win_bf16_d32_l4_s12_m5_n3", F(BF_32_2_4_M5, 12, 3), B(BB_32_2_4_M5, 12, 3)},
    // exact walk (bit-identical to the sequential scan)
    {"xwin_bf16_d32_s8_m5_n2", F(XBF_32_2_8_M5, 8, 2), B(XBB_32_2_8_M5, 8, 2)},
    {"xwin_bf16_d32_l4_s12_m5", F(XBF_32_2_4_M5, 12, 2), B(XBB_32_2_4_M5, 12, 2)},
    {"xwin_bf16_d32_l16_s8", F(XWBF_32_2_16, 8, 4), B(XWBB_32_2_16, 8, 4)},
    {"xwin_bf16_d32_s8_m5_n3", F(XBF_32_2_8_M5, 8, 3), B(XBB_32_2_8_M5, 8, 3)},
    // wavefront exact tiles (the chain runs through one warp per sub-chunk)
    {"wfx_bf16_d32_s4_l16", WF(WFF_BF_32_1_16, 4, 2), WB(WFB_BF_32_1_16, 4, 2)},
    {"wfx_bf16_d32_s4_l16_n3", WF(WFF_BF_32_1_16, 4, 3), WB(WFB_BF_32_1_16, 4, 3)},
    {"wfx_bf16_d32_s8_l8", WF(WFF_BF_32_1_8, 8, 2), WB(WFB_BF_32_1_8, 8, 2)},
    {"wfx_bf16_d64_s4_l16_v2", WF(WFF_BF_64_2_16, 4, 2), WB(WFB_BF_64_2_16, 4, 2)},
    {"wfx_bf16_d32_s2_l32", WF(WFF_BF_32_1_32, 2, 3), WB(WFB_BF_32_1_32, 2, 3)},
    {"wfx_bf16_d32_s2_l16", WF(WFF_BF_32_1_16, 2, 3), WB(WFB_BF_32_1_16, 2, 3)},
    {"wfx_bf16_d32_s3_l16", WF(WFF_BF_32_1_16, 3, 2), WB(WFB_BF_32_1_16, 3, 2)},
};
const WinVariant kSeqF32[] = {
    {"seq_f32_d32", F(SFF_32_1_32, 1, 8), B(SFB_32_1_32, 1, 6)},
    {"seq_f32_d64", F(SFF_64_2_16, 1, 8), B(SFB_64_2_16, 1, 6)},
    {"seq_f32_d64_v1", F(SFF_64_1_32, 1, 4), B(SFB_64_1_32, 1, 4)},
    {"seq_f32_d128", F(SFF_128_4_8, 1, 8), B(SFB_128_4_8, 1, 6)},
    // a shallower ring: more CTAs resident per SM
    {"seq_f32_d64_v1_n3", F(SFF_64_1_32, 1, 3), B(SFB_64_1_32, 1, 2)},
};
const WinVariant kWinF32[] = {
    {"win_f32_d32_s16_pt", F(PF_32_1_8, 16, 4), B(PFB_32_1_8, 16, 3)},
    {"win_f32_d16_s16", F(FF_16_1_8, 16, 4), B(FB_16_1_8, 16, 4)},
    {"win_f32_d32_s16", F(FF_32_1_8, 16, 4), B(FB_32_1_8, 16, 3)},
    {"win_f32_d16_s16_pt", F(PF_16_1_8, 16, 4), B(PFB_16_1_8, 16, 4)},
    {"win_f32_d64_s8", F(FF_64_2_8, 8, 4), B(FB_64_2_8, 8, 3)},
    {"win_f32_d32_s8_pt", F(PF_32_1_8, 8, 8), B(PFB_32_1_8, 8, 6)},
    {"win_f32_d32_s31", F(FF_32_1_8_X, 31, 2), B(FB_32_1_8, 16, 3)},
    // exact walk (bit-identical to the sequential scan)
    {"xwin_f32_d64_s8", F(XFF_64_2_8, 8, 4), B(XFB_64_2_8, 8, 3)},
    {"xwin_f32_d32_s16", F(XFF_32_1_8, 16, 4), B(XFB_32_1_8, 16, 3)},
    // wavefront exact tiles
    {"wfx_f32_d32_s4_l16", WF(WFF_FF_32_1_16, 4, 2), WB(WFB_FF_32_1_16, 4, 2)},
    {"wfx_f32_d64_s8_l8_v2", WF(WFF_FF_64_2_8, 8, 2), WB(WFB_FF_64_2_8, 8, 2)},
};

#undef F
#undef B
#undef WF
#undef WB


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
