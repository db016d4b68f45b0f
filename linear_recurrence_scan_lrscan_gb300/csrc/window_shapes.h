// Compiled tile shapes of the time-tiled kernels, and the lists of the shapes
// the variant tables use (for explicit instantiation across translation
// units).
#pragma once

#include "window_kernels.cuh"

namespace lrscan {

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ, PT>
// Sequential shapes (S = 1): L rows per window streamed from shared memory.
using SBF_64_2_32 = WinShape<bf16_t, 64, 2, 32, 2, 64, 1, true>;
using SBF_128_2_32 = WinShape<bf16_t, 128, 2, 32, 2, 96, 1, true>;
using SBF_128_4_32 = WinShape<bf16_t, 128, 4, 32, 2, 64, 1, true>;
using SBF_32_1_32 = WinShape<bf16_t, 32, 1, 32, 2, 64, 1, true>;
using SBF_64_1_32 = WinShape<bf16_t, 64, 1, 32, 2, 96, 1, true>;
using SBB_64_2_32 = WinShape<bf16_t, 64, 2, 32, 3, 64, 1, true>;
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
using BB_64_2_8 = WinShape<bf16_t, 64, 2, 8, 3, 288, 2, false>;
using BB_32_2_8 = WinShape<bf16_t, 32, 2, 8, 3, 288, 2, false>;
using FF_16_1_8 = WinShape<float, 16, 1, 8, 2, 544, 1, false>;
using FF_32_1_8 = WinShape<float, 32, 1, 8, 2, 544, 1, false>;
using FF_64_2_8 = WinShape<float, 64, 2, 8, 2, 288, 2, false>;
using FB_16_1_8 = WinShape<float, 16, 1, 8, 3, 544, 1, false>;
using FB_32_1_8 = WinShape<float, 32, 1, 8, 3, 544, 1, false>;
using FB_64_2_8 = WinShape<float, 64, 2, 8, 3, 288, 1, false>;
// few threads per CTA and a high residency floor: every CTA of a 640-tile
// launch resident at once (5 or 8 per SM), no tail wave
using BF_32_2_8_M5 = WinShape<bf16_t, 32, 2, 8, 2, 160, 5, false>;
using BB_32_2_8_M5 = WinShape<bf16_t, 32, 2, 8, 3, 160, 5, false>;
using BF_32_2_8_M8 = WinShape<bf16_t, 32, 2, 8, 2, 96, 8, false>;
using BB_32_2_8_M8 = WinShape<bf16_t, 32, 2, 8, 3, 96, 8, false>;
// L = 4 with 12 sub-chunks (7 warps per CTA), five resident per SM: more
// consumer warps on the same 640-tile launch
using BF_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 2, 224, 5, false>;
using BB_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 3, 224, 5, false>;
// fp32, one CTA of 32 warps per lane tile (few lane tiles)
using FF_32_1_8_X = WinShape<float, 32, 1, 8, 2, 1024, 1, false>;
// per-thread-prefix shapes (parallel fold, short critical path)
using PF_32_1_8 = WinShape<float, 32, 1, 8, 2, 544, 1, false, true>;
using PFB_32_1_8 = WinShape<float, 32, 1, 8, 3, 544, 1, false, true>;
using PF_16_1_8 = WinShape<float, 16, 1, 8, 2, 544, 1, false, true>;
using PFB_16_1_8 = WinShape<float, 16, 1, 8, 3, 544, 1, false, true>;
// L = 16: half the sub-chunks (and half the in-CTA prefix work) per window row
using WBF_32_2_16 = WinShape<bf16_t, 32, 2, 16, 2, 288, 1, false>;
using WBB_32_2_16 = WinShape<bf16_t, 32, 2, 16, 3, 288, 1, false>;

// Exact windowed shapes: the lane threads walk the window's rows with the
// sequential step (no sub-chunk maps), so every result is bit-identical to
// the sequential scan.
using XBF_32_2_8_M5 = WinShape<bf16_t, 32, 2, 8, 2, 160, 5, false, false, true>;
using XBB_32_2_8_M5 = WinShape<bf16_t, 32, 2, 8, 3, 160, 5, false, false, true>;
using XBF_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 2, 224, 5, false, false, true>;
using XBB_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 3, 224, 5, false, false, true>;
using XWBF_32_2_16 = WinShape<bf16_t, 32, 2, 16, 2, 288, 1, false, false, true>;
using XWBB_32_2_16 = WinShape<bf16_t, 32, 2, 16, 3, 288, 1, false, false, true>;
using XFF_64_2_8 = WinShape<float, 64, 2, 8, 2, 288, 2, false, false, true>;
using XFB_64_2_8 = WinShape<float, 64, 2, 8, 3, 288, 1, false, false, true>;
using XFF_32_1_8 = WinShape<float, 32, 1, 8, 2, 544, 1, false, false, true>;
using XFB_32_1_8 = WinShape<float, 32, 1, 8, 3, 544, 1, false, false, true>;

// Wavefront exact shapes: one warp per sub-chunk (32 lane groups of V lanes).
using WFF_BF_32_1_16 = WinShape<bf16_t, 32, 1, 16, 2, 160, 5, false, false, true>;
using WFB_BF_32_1_16 = WinShape<bf16_t, 32, 1, 16, 3, 160, 5, false, false, true>;
using WFF_BF_32_1_8 = WinShape<bf16_t, 32, 1, 8, 2, 288, 3, false, false, true>;
using WFB_BF_32_1_8 = WinShape<bf16_t, 32, 1, 8, 3, 288, 3, false, false, true>;
using WFF_BF_64_2_16 = WinShape<bf16_t, 64, 2, 16, 2, 160, 4, false, false, true>;
using WFB_BF_64_2_16 = WinShape<bf16_t, 64, 2, 16, 3, 160, 4, false, false, true>;
using WFF_FF_32_1_16 = WinShape<float, 32, 1, 16, 2, 160, 4, false, false, true>;
using WFB_FF_32_1_16 = WinShape<float, 32, 1, 16, 3, 160, 4, false, false, true>;
using WFF_FF_64_2_8 = WinShape<float, 64, 2, 8, 2, 288, 2, false, false, true>;
using WFB_FF_64_2_8 = WinShape<float, 64, 2, 8, 3, 288, 2, false, false, true>;

using WFF_BF_32_1_32 = WinShape<bf16_t, 32, 1, 32, 2, 96, 6, false, false, true>;
using WFB_BF_32_1_32 = WinShape<bf16_t, 32, 1, 32, 3, 96, 6, false, false, true>;

#define LRSCAN_WFX_FWD_SHAPES(X) \
    X(WFF_BF_32_1_16) X(WFF_BF_32_1_8) X(WFF_BF_64_2_16) X(WFF_FF_32_1_16) X(WFF_FF_64_2_8) X(WFF_BF_32_1_32)
#define LRSCAN_WFX_BWD_SHAPES(X) \
    X(WFB_BF_32_1_16) X(WFB_BF_32_1_8) X(WFB_BF_64_2_16) X(WFB_FF_32_1_16) X(WFB_FF_64_2_8) X(WFB_BF_32_1_32)

#define LRSCAN_WIN_FWD_SHAPES(X)                                                                   \
    X(SBF_64_2_32) X(SBF_128_2_32) X(SBF_128_4_32) X(SBF_32_1_32) X(SBF_64_1_32) X(SFF_32_1_32) \
    X(SFF_64_2_16) X(SFF_64_1_32) X(SFF_128_4_8) X(BF_64_2_8) X(BF_32_2_8) X(FF_16_1_8)          \
    X(FF_32_1_8) X(FF_64_2_8) X(PF_32_1_8) X(PF_16_1_8) X(WBF_32_2_16) X(BF_32_2_8_M5) X(BF_32_2_8_M8) X(BF_32_2_4_M5) X(FF_32_1_8_X)   \
    X(XBF_32_2_8_M5) X(XBF_32_2_4_M5) X(XWBF_32_2_16) X(XFF_64_2_8) X(XFF_32_1_8)

#define LRSCAN_WIN_BWD_SHAPES(X)                                                                   \
    X(SBB_64_2_32) X(SBB_32_1_32) X(SBB_64_1_32) X(SBB_128_2_32) X(SBB_128_4_16) X(SFB_32_1_32) \
    X(SFB_64_2_16) X(SFB_64_1_32) X(SFB_128_4_8) X(BB_64_2_8) X(BB_32_2_8) X(FB_16_1_8)          \
    X(FB_32_1_8) X(FB_64_2_8) X(PFB_32_1_8) X(PFB_16_1_8) X(WBB_32_2_16) X(BB_32_2_8_M5) X(BB_32_2_8_M8) X(BB_32_2_4_M5)                  \
    X(XBB_32_2_8_M5) X(XBB_32_2_4_M5) X(XWBB_32_2_16) X(XFB_64_2_8) X(XFB_32_1_8)

}  // namespace lrscan
