// Instantiations of the complex scan kernels (the EXT ones are in
// kernels_complex_state.cu), and their tile variant table.
#include <cstdlib>

#include "complex_launch.cuh"

namespace lrscan {

#define LRSCAN_EXTERN_CSF(SH) extern template int launch_cwin_fwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_EXTERN_CSB(SH) extern template int launch_cwin_bwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_EXTERN_CWF(SH) extern template int launch_cwinw_fwd<SH, true>(const WinLaunch &, const WinDirCfg &);
#define LRSCAN_EXTERN_CWB(SH) extern template int launch_cwinw_bwd<SH, true>(const WinLaunch &, const WinDirCfg &);
LRSCAN_CSEQ_FWD_SHAPES(LRSCAN_EXTERN_CSF)
LRSCAN_CSEQ_BWD_SHAPES(LRSCAN_EXTERN_CSB)
LRSCAN_CWIN_FWD_SHAPES(LRSCAN_EXTERN_CWF)
LRSCAN_CWIN_BWD_SHAPES(LRSCAN_EXTERN_CWB)
#undef LRSCAN_EXTERN_CSF
#undef LRSCAN_EXTERN_CSB
#undef LRSCAN_EXTERN_CWF
#undef LRSCAN_EXTERN_CWB

namespace {

template <class C, bool FWD>
WinDirCfg cdir_cfg(int nstage) {
    static_assert(C::SEQ && C::G % 32 == 0, "complex tiles: sequential, whole consumer warps");
    static_assert(C::NIN == (FWD ? 4 : 6), "complex planes: 4 forward, 6 backward");
    const WinGeom g = make_win_geom<C>(1, nstage, 1, 1);
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = 1;
    d.exact = 1;  // the sequential nested-fma order
    d.w = g.W;
    d.nstage = nstage;
    d.threads = C::G + 32;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) {
        d.launch = &launch_cwin_fwd<C, false>;
        d.launch_state = &launch_cwin_fwd<C, true>;
    } else {
        d.launch = &launch_cwin_bwd<C, false>;
        d.launch_state = &launch_cwin_bwd<C, true>;
    }
    return d;
}

// Windowed complex tiles: S sub-chunks of L rows, lane scan.  Forward: a, b
// in, out_r / out_i staged in two buffers; backward: a, out, grad_out in,
// the four gradient planes staged in one buffer each.
template <class C, bool FWD = true>
WinDirCfg cwdir_cfg(int S, int nstage) {
    static_assert(!C::SEQ && !C::PT && C::NIN == (FWD ? 4 : 6), "windowed complex shape");
    if (S > C::SMAX) std::abort();  // table error
    const WinGeom g = make_cwin_geom<C>(S, nstage, 1, 1);
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.lane_scan = 1;
    d.w = g.W;
    d.nstage = nstage;
    d.threads = S * C::G + 32;
    d.smem = FWD ? win_out_smem(g, 2) : win_out_smem(g, 4, 1);  // plus the output staging
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) {
        d.launch = &launch_cwinw_fwd<C, false>;
        d.launch_state = &launch_cwinw_fwd<C, true>;
    } else {
        d.launch = &launch_cwinw_bwd<C, false>;
        d.launch_state = &launch_cwinw_bwd<C, true>;
    }
    return d;
}

#define F(SH, N) cdir_cfg<SH, true>(N)
#define B(SH, N) cdir_cfg<SH, false>(N)
const WinVariant kCplxBF16[] = {
    {"cseq_bf16_d64_v1", F(CBF_64_1_32, 6), B(CBB_64_1_32, 4)},
    {"cseq_bf16_d64_v2", F(CBF_64_2_32, 6), B(CBB_64_2_16, 6)},
    {"cseq_bf16_d32_v1", F(CBF_32_1_32, 6), B(CBB_32_1_32, 4)},
    {"cseq_bf16_d64_v1_n4", F(CBF_64_1_32, 4), B(CBB_64_1_32, 3)},
    {"cseq_bf16_d64_v2_n4", F(CBF_64_2_32, 4), B(CBB_64_2_16, 5)},
    {"cwin_bf16_d32_s8", cwdir_cfg<CWF_BF_32_1_8>(8, 3), B(CBB_64_1_32, 3)},
    {"cwin_bf16_d32_s16_v2", cwdir_cfg<CWF_BF_32_2_8>(16, 2), B(CBB_64_1_32, 3)},
    {"cwin_bf16_d32_l4_s8_m5", cwdir_cfg<CWF_BF_32_2_4_M5>(8, 2), (cwdir_cfg<CWB_BF_32_2_4_M5, false>(8, 2))},
};
const WinVariant kCplxF32[] = {
    {"cseq_f32_d32_v1", F(CFF_32_1_32, 6), B(CFB_32_1_32, 4)},
    {"cseq_f32_d64_v2", F(CFF_64_2_16, 8), B(CFB_64_2_16, 6)},
    {"cseq_f32_d64_v1", F(CFF_64_1_16, 8), B(CFB_64_1_16, 6)},
    {"cseq_f32_d32_v1_n4", F(CFF_32_1_32, 4), B(CFB_32_1_32, 3)},
    {"cseq_f32_d64_v1_n4", F(CFF_64_1_16, 4), B(CFB_64_1_16, 3)},
    {"cwin_f32_d32_s8", cwdir_cfg<CWF_FF_32_1_8>(8, 3), B(CFB_32_1_32, 4)},
};
#undef F
#undef B

}  // namespace

const WinVariant *cwin_variants(int dtype, int *count) {
    if (dtype == 0) {
        *count = sizeof(kCplxF32) / sizeof(kCplxF32[0]);
        return kCplxF32;
    }
    *count = sizeof(kCplxBF16) / sizeof(kCplxBF16[0]);
    return kCplxBF16;
}

int cplain_fwd_launch(const ChunkLaunch &L, const void *ai, const void *bi, void *out_i, float *last_i, int dtype) {
    const int nlb = static_cast<int>((L.D + 127) / 128);
    const unsigned nb = static_cast<unsigned>(nlb * L.B);
    const int T = static_cast<int>(L.T), D = static_cast<int>(L.D);
    if (dtype == 0)
        cplain_fwd<float><<<nb, 128, 0, L.stream>>>(
            static_cast<const float *>(L.in0), static_cast<const float *>(ai), static_cast<const float *>(L.in1),
            static_cast<const float *>(bi), static_cast<float *>(L.out0), static_cast<float *>(out_i), L.last,
            last_i, T, D, nlb);
    else
        cplain_fwd<bf16_t><<<nb, 128, 0, L.stream>>>(
            static_cast<const bf16_t *>(L.in0), static_cast<const bf16_t *>(ai), static_cast<const bf16_t *>(L.in1),
            static_cast<const bf16_t *>(bi), static_cast<bf16_t *>(L.out0), static_cast<bf16_t *>(out_i), L.last,
            last_i, T, D, nlb);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int cplain_bwd_launch(const void *const in[6], void *const outp[4], int64_t B, int64_t T, int64_t D, int dtype,
                      cudaStream_t stream) {
    const int nlb = static_cast<int>((D + 127) / 128);
    const unsigned nb = static_cast<unsigned>(nlb * B);
    if (dtype == 0) {
        using S = float;
        cplain_bwd<S><<<nb, 128, 0, stream>>>(
            static_cast<const S *>(in[0]), static_cast<const S *>(in[1]), static_cast<const S *>(in[2]),
            static_cast<const S *>(in[3]), static_cast<const S *>(in[4]), static_cast<const S *>(in[5]),
            static_cast<S *>(outp[0]), static_cast<S *>(outp[1]), static_cast<S *>(outp[2]),
            static_cast<S *>(outp[3]), static_cast<int>(T), static_cast<int>(D), nlb);
    } else {
        using S = bf16_t;
        cplain_bwd<S><<<nb, 128, 0, stream>>>(
            static_cast<const S *>(in[0]), static_cast<const S *>(in[1]), static_cast<const S *>(in[2]),
            static_cast<const S *>(in[3]), static_cast<const S *>(in[4]), static_cast<const S *>(in[5]),
            static_cast<S *>(outp[0]), static_cast<S *>(outp[1]), static_cast<S *>(outp[2]),
            static_cast<S *>(outp[3]), static_cast<int>(T), static_cast<int>(D), nlb);
    }
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace lrscan
