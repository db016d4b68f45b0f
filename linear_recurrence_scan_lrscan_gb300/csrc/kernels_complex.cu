// Instantiations and launchers of the complex scan kernels, and their tile
// variant table.
#include <cstdlib>

#include "complex_kernels.cuh"
#include "window_launch.cuh"

namespace lrscan {

namespace {

// rows staged in registers per step of a full window
template <class C> constexpr int kStageRowsFwd = C::L < 16 ? C::L : 16;
template <class C> constexpr int kStageRowsBwd = C::L < 8 ? C::L : 8;

template <class C>
int launch_cwin_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwin_fwd_kernel<C, kStageRowsFwd<C>>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(1, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    using St = typename C::St;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3],
                                     static_cast<St *>(L.out0), static_cast<St *>(L.out1), L.last, L.last_i, g,
                                     L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_cwinw_fwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwinw_fwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_cwin_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads),
                                     win_out_smem(g, 2), L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3],
                                     *L.maps[4], *L.maps[5], L.last, L.last_i, g, L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_cwin_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwin_bwd_kernel<C, kStageRowsBwd<C>>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(1, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    using St = typename C::St;
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads), g.smem_bytes,
                                     L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3], *L.maps[4],
                                     *L.maps[5], static_cast<St *>(L.out0), static_cast<St *>(L.out1),
                                     static_cast<St *>(L.out2), static_cast<St *>(L.out3), g, L.status,
                                     L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
}

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
    d.w = g.W;
    d.nstage = nstage;
    d.threads = C::G + 32;
    d.smem = g.smem_bytes;
    d.stage_bytes = g.stage_bytes;
    if constexpr (FWD) d.launch = &launch_cwin_fwd<C>;
    else d.launch = &launch_cwin_bwd<C>;
    d.launch_state = nullptr;
    return d;
}

template <class C>
int launch_cwinw_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = cwinw_bwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_cwin_geom<C>(cfg.s, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const cudaError_t e = launch_pdl(fn, dim3(ndt, static_cast<unsigned>(L.B)), dim3(cfg.threads),
                                     win_out_smem(g, 4, 1), L.stream, *L.maps[0], *L.maps[1], *L.maps[2], *L.maps[3],
                                     *L.maps[4], *L.maps[5], *L.maps[6], *L.maps[7], *L.maps[8], *L.maps[9], g,
                                     L.status, L.timeout_ns);
    return e == cudaSuccess ? 0 : -1;
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
    if constexpr (FWD) d.launch = &launch_cwinw_fwd<C>;
    else d.launch = &launch_cwinw_bwd<C>;
    return d;
}

// WinShape<St, DT, V, L, NIN, MAXT, MINB, SEQ>
using CWF_BF_32_1_8 = WinShape<bf16_t, 32, 1, 8, 4, 288, 2, false>;
using CWF_BF_32_2_8 = WinShape<bf16_t, 32, 2, 8, 4, 288, 2, false>;
using CWF_FF_32_1_8 = WinShape<float, 32, 1, 8, 4, 288, 2, false>;
// 4-row sub-chunks, five CTAs per SM: every CTA of a 640-tile launch resident
using CWF_BF_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 4, 160, 5, false>;
using CWB_BF_32_2_4_M5 = WinShape<bf16_t, 32, 2, 4, 6, 160, 5, false>;
using CBF_64_1_32 = WinShape<bf16_t, 64, 1, 32, 4, 96, 1, true>;
using CBB_64_1_32 = WinShape<bf16_t, 64, 1, 32, 6, 96, 1, true>;
using CBF_64_2_32 = WinShape<bf16_t, 64, 2, 32, 4, 64, 1, true>;
using CBB_64_2_16 = WinShape<bf16_t, 64, 2, 16, 6, 64, 1, true>;
using CBF_32_1_32 = WinShape<bf16_t, 32, 1, 32, 4, 64, 1, true>;
using CBB_32_1_32 = WinShape<bf16_t, 32, 1, 32, 6, 64, 1, true>;
using CFF_32_1_32 = WinShape<float, 32, 1, 32, 4, 64, 1, true>;
using CFB_32_1_32 = WinShape<float, 32, 1, 32, 6, 64, 1, true>;
using CFF_64_2_16 = WinShape<float, 64, 2, 16, 4, 64, 1, true>;
using CFB_64_2_16 = WinShape<float, 64, 2, 16, 6, 64, 1, true>;
using CFF_64_1_16 = WinShape<float, 64, 1, 16, 4, 96, 1, true>;
using CFB_64_1_16 = WinShape<float, 64, 1, 16, 6, 96, 1, true>;

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
