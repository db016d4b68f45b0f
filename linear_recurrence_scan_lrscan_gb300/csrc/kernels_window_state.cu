// EXT instantiations (carried state and segment resets) of the time-tiled
// kernels, one per shape of the variant tables; compiled in parallel with
// kernels_window.cu.
#include "window_launch.cuh"
#include "window_shapes.h"

namespace lrscan {

#define LRSCAN_INST_FWD(SH) template int launch_win_fwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_INST_BWD(SH) template int launch_win_bwd<SH, true>(const WinLaunch &, const WinDirCfg &);
LRSCAN_WIN_FWD_SHAPES(LRSCAN_INST_FWD)
LRSCAN_WIN_BWD_SHAPES(LRSCAN_INST_BWD)
#undef LRSCAN_INST_FWD
#undef LRSCAN_INST_BWD
#define LRSCAN_INST_WF(SH) template int launch_wfx<SH, false, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_INST_WB(SH) template int launch_wfx<SH, true, true>(const WinLaunch &, const WinDirCfg &);
LRSCAN_WFX_FWD_SHAPES(LRSCAN_INST_WF)
LRSCAN_WFX_BWD_SHAPES(LRSCAN_INST_WB)
#undef LRSCAN_INST_WF
#undef LRSCAN_INST_WB

}  // namespace lrscan
