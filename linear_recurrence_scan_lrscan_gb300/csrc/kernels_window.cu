// Instantiations and launchers of the time-tiled (TMA) kernels, and the table
// of tile variants the host dispatcher chooses from.
#include "launch.h"
#include "window_kernels.cuh"

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
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.r, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    fn<<<dim3(ndt, static_cast<unsigned>(L.B)), cfg.threads, g.smem_bytes, L.stream>>>(
        *L.maps[0], *L.maps[1], static_cast<typename C::St *>(L.out0), L.last, g, L.status, L.timeout_ns);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_win_bwd(const WinLaunch &L, const WinDirCfg &cfg) {
    static unsigned long long mask = 0;
    static std::mutex mu;
    auto fn = win_bwd_kernel<C>;
    if (set_smem_attr(reinterpret_cast<const void *>(fn), L.device, &mask, &mu)) return -1;
    const WinGeom g = make_win_geom<C>(cfg.s, cfg.r, cfg.nstage, static_cast<int>(L.T), static_cast<int>(L.D));
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    fn<<<dim3(ndt, static_cast<unsigned>(L.B)), cfg.threads, g.smem_bytes, L.stream>>>(
        *L.maps[0], *L.maps[1], *L.maps[2], static_cast<typename C::St *>(L.out0),
        static_cast<typename C::St *>(L.out1), g, L.status, L.timeout_ns);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <class C, bool FWD>
WinDirCfg dir_cfg(int S, int R, int nstage) {
    const WinGeom g = make_win_geom<C>(S, R, nstage, 1, 1);
    WinDirCfg d{};
    d.dt = C::DT;
    d.v = C::V;
    d.l = C::L;
    d.s = S;
    d.r = g.R;
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

// WinShape<St, DT, V, L, NIN, MAXT, MINB>
// forward shapes (NIN = 2)
using BF_64_2_16 = WinShape<bf16_t, 64, 2, 16, 2, 64, 8>;
using BF_128_4_8 = WinShape<bf16_t, 128, 4, 8, 2, 288, 1>;
using BF_64_2_8 = WinShape<bf16_t, 64, 2, 8, 2, 288, 3>;
using BF_32_1_8 = WinShape<bf16_t, 32, 1, 8, 2, 288, 3>;
using FF_32_1_16 = WinShape<float, 32, 1, 16, 2, 64, 8>;
using FF_64_2_8 = WinShape<float, 64, 2, 8, 2, 288, 3>;
using FF_128_4_8 = WinShape<float, 128, 4, 8, 2, 64, 4>;
using FF_32_1_8 = WinShape<float, 32, 1, 8, 2, 544, 1>;
using FF_16_1_8 = WinShape<float, 16, 1, 8, 2, 544, 1>;
// backward shapes (NIN = 3)
using BB_64_2_8 = WinShape<bf16_t, 64, 2, 8, 3, 288, 2>;
using BB_128_4_4 = WinShape<bf16_t, 128, 4, 4, 3, 288, 2>;
using BB_128_4_8 = WinShape<bf16_t, 128, 4, 8, 3, 288, 1>;
using BB_32_1_8 = WinShape<bf16_t, 32, 1, 8, 3, 288, 2>;
using FB_32_1_16 = WinShape<float, 32, 1, 16, 3, 64, 8>;
using FB_64_2_8 = WinShape<float, 64, 2, 8, 3, 288, 1>;
using FB_128_4_4 = WinShape<float, 128, 4, 4, 3, 64, 4>;
using FB_32_1_8 = WinShape<float, 32, 1, 8, 3, 544, 1>;
using FB_16_1_8 = WinShape<float, 16, 1, 8, 3, 544, 1>;

#define F(SH, S, R, N) dir_cfg<SH, true>(S, R, N)
#define B(SH, S, R, N) dir_cfg<SH, false>(S, R, N)

const WinVariant kSeqBF16[] = {
    {"seq_bf16_d64", F(BF_64_2_16, 1, 2, 8), B(BB_64_2_8, 1, 4, 6)},
    {"seq_bf16_d128", F(BF_128_4_8, 1, 4, 6), B(BB_128_4_4, 1, 8, 4)},
    {"seq_bf16_d64_deep", F(BF_64_2_8, 1, 4, 8), B(BB_64_2_8, 1, 2, 12)},
    {"seq_bf16_d128_short", F(BF_128_4_8, 1, 2, 8), B(BB_128_4_4, 1, 4, 6)},
};
const WinVariant kWinBF16[] = {
    {"win_bf16_d64_s4", F(BF_64_2_8, 4, 1, 8), B(BB_64_2_8, 4, 1, 6)},
    {"win_bf16_d64_s8", F(BF_64_2_8, 8, 1, 4), B(BB_64_2_8, 8, 1, 3)},
    {"win_bf16_d32_s8", F(BF_32_1_8, 8, 1, 4), B(BB_32_1_8, 8, 1, 3)},
    {"win_bf16_d128_s4", F(BF_128_4_8, 4, 1, 6), B(BB_128_4_4, 8, 1, 4)},
    {"win_bf16_d64_s2", F(BF_64_2_8, 2, 1, 12), B(BB_64_2_8, 2, 1, 10)},
};
const WinVariant kSeqF32[] = {
    {"seq_f32_d32", F(FF_32_1_16, 1, 2, 8), B(FB_32_1_16, 1, 2, 6)},
    {"seq_f32_d64", F(FF_64_2_8, 1, 4, 6), B(FB_64_2_8, 1, 4, 4)},
    {"seq_f32_d128", F(FF_128_4_8, 1, 2, 6), B(FB_128_4_4, 1, 4, 4)},
    {"seq_f32_d64_short", F(FF_64_2_8, 1, 2, 8), B(FB_64_2_8, 1, 2, 6)},
};
const WinVariant kWinF32[] = {
    {"win_f32_d16_s16", F(FF_16_1_8, 16, 1, 4), B(FB_16_1_8, 16, 1, 4)},
    {"win_f32_d32_s16", F(FF_32_1_8, 16, 1, 4), B(FB_32_1_8, 16, 1, 3)},
    {"win_f32_d32_s8", F(FF_32_1_8, 8, 1, 8), B(FB_32_1_8, 8, 1, 6)},
    {"win_f32_d16_s8", F(FF_16_1_8, 8, 1, 8), B(FB_16_1_8, 8, 1, 6)},
    {"win_f32_d32_s4", F(FF_32_1_8, 4, 1, 12), B(FB_32_1_8, 4, 1, 10)},
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
