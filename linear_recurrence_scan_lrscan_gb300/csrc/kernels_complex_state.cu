// EXT instantiations (carried state and segment resets) of the complex tiled
// kernels, one per shape of the complex variant table; compiled in parallel
// with kernels_complex.cu.
#include "complex_launch.cuh"

namespace lrscan {

#define LRSCAN_INST_CSF(SH) template int launch_cwin_fwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_INST_CSB(SH) template int launch_cwin_bwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_INST_CWF(SH) template int launch_cwinw_fwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_INST_CWB(SH) template int launch_cwinw_bwd<SH, true>(const WinLaunch &, const WinDirCfg &);
LRSCAN_CSEQ_FWD_SHAPES(LRSCAN_INST_CSF)
LRSCAN_CSEQ_BWD_SHAPES(LRSCAN_INST_CSB)
LRSCAN_CWIN_FWD_SHAPES(LRSCAN_INST_CWF)
LRSCAN_CWIN_BWD_SHAPES(LRSCAN_INST_CWB)
#undef LRSCAN_INST_CSF
#undef LRSCAN_INST_CSB
#undef LRSCAN_INST_CWF
#undef LRSCAN_INST_CWB

}  // namespace lrscan
