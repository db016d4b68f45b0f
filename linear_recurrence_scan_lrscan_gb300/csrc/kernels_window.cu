// Instantiations and launchers of the time-tiled (TMA) kernels.  The host
// dispatcher only sees the variant table at the bottom.
#include "launch.h"
#include "window_kernels.cuh"

namespace lrscan {

namespace {

template <class C>
__host__ int set_smem_attr(const void *fn, int dev) {
    // Dynamic shared memory above 48 KB has to be opted into per device.
    static unsigned long long done_mask = 0;  // devices done (up to 64)
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 64 && (done_mask >> dev) & 1ull) return 0;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return -1;
    if (dev < 64) done_mask |= 1ull << dev;
    return 0;
}

template <class C>
int launch_win_fwd(const WinLaunch &L) {
    auto fn = win_fwd_kernel<C>;
    if (set_smem_attr<C>(reinterpret_cast<const void *>(fn), L.device)) return -1;
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const int nwin = static_cast<int>((L.T + C::W - 1) / C::W);
    fn<<<dim3(ndt, static_cast<unsigned>(L.B)), C::THREADS, C::SMEM_BYTES, L.stream>>>(
        *L.maps[0], *L.maps[1], static_cast<typename C::St *>(L.out0), L.last, static_cast<int>(L.T),
        static_cast<int>(L.D), nwin, L.status, L.timeout_ns);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <class C>
int launch_win_bwd(const WinLaunch &L) {
    auto fn = win_bwd_kernel<C>;
    if (set_smem_attr<C>(reinterpret_cast<const void *>(fn), L.device)) return -1;
    const int ndt = static_cast<int>((L.D + C::DT - 1) / C::DT);
    const int nwin = static_cast<int>((L.T + C::W - 1) / C::W);
    fn<<<dim3(ndt, static_cast<unsigned>(L.B)), C::THREADS, C::SMEM_BYTES, L.stream>>>(
        *L.maps[0], *L.maps[1], *L.maps[2], static_cast<typename C::St *>(L.out0),
        static_cast<typename C::St *>(L.out1), static_cast<int>(L.T), static_cast<int>(L.D), nwin,
        L.status, L.timeout_ns);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <class Cf, class Cb>
constexpr WinVariant make_variant(const char *name) {
    return WinVariant{name,
                      Cf::DT,
                      Cf::V,
                      Cf::S,
                      Cf::L,
                      Cf::W,
                      Cf::NSTAGE,
                      Cb::NSTAGE,
                      Cf::THREADS,
                      Cf::SMEM_BYTES,
                      Cb::SMEM_BYTES,
                      Cf::STAGE_BYTES,
                      Cb::STAGE_BYTES,
                      &launch_win_fwd<Cf>,
                      &launch_win_bwd<Cb>};
}

// WinShape<St, DT, V, S, L, NSTAGE, NIN>
// ---- sequential (S = 1) ----
using F32_S1_A_f = WinShape<float, 32, 1, 1, 32, 4, 2>;
using F32_S1_A_b = WinShape<float, 32, 1, 1, 32, 4, 3>;
using F32_S1_B_f = WinShape<float, 64, 2, 1, 16, 4, 2>;
using F32_S1_B_b = WinShape<float, 64, 2, 1, 16, 4, 3>;
using F32_S1_C_f = WinShape<float, 64, 1, 1, 16, 4, 2>;
using F32_S1_C_b = WinShape<float, 64, 1, 1, 16, 4, 3>;
using F32_S1_D_f = WinShape<float, 128, 4, 1, 8, 6, 2>;
using F32_S1_D_b = WinShape<float, 128, 4, 1, 8, 6, 3>;

using B16_S1_A_f = WinShape<bf16_t, 64, 2, 1, 32, 4, 2>;
using B16_S1_A_b = WinShape<bf16_t, 64, 2, 1, 32, 4, 3>;
using B16_S1_B_f = WinShape<bf16_t, 128, 2, 1, 32, 4, 2>;
using B16_S1_B_b = WinShape<bf16_t, 128, 2, 1, 32, 4, 3>;
using B16_S1_C_f = WinShape<bf16_t, 128, 2, 1, 16, 6, 2>;
using B16_S1_C_b = WinShape<bf16_t, 128, 2, 1, 16, 6, 3>;
using B16_S1_D_f = WinShape<bf16_t, 256, 4, 1, 16, 4, 2>;
using B16_S1_D_b = WinShape<bf16_t, 256, 4, 1, 16, 4, 3>;

// ---- windowed (S > 1) ----
using F32_W_A_f = WinShape<float, 16, 1, 16, 8, 4, 2>;
using F32_W_A_b = WinShape<float, 16, 1, 16, 8, 4, 3>;
using F32_W_B_f = WinShape<float, 32, 1, 16, 8, 3, 2>;
using F32_W_B_b = WinShape<float, 32, 1, 16, 8, 3, 3>;
using F32_W_C_f = WinShape<float, 16, 1, 32, 4, 4, 2>;
using F32_W_C_b = WinShape<float, 16, 1, 32, 4, 4, 3>;

using B16_W_A_f = WinShape<bf16_t, 32, 2, 16, 8, 4, 2>;
using B16_W_A_b = WinShape<bf16_t, 32, 2, 16, 8, 4, 3>;
using B16_W_B_f = WinShape<bf16_t, 64, 2, 8, 16, 4, 2>;
using B16_W_B_b = WinShape<bf16_t, 64, 2, 8, 16, 4, 3>;

const WinVariant kSeqF32[] = {
    make_variant<F32_S1_A_f, F32_S1_A_b>("seq_f32_d32_v1_l32"),
    make_variant<F32_S1_B_f, F32_S1_B_b>("seq_f32_d64_v2_l16"),
    make_variant<F32_S1_C_f, F32_S1_C_b>("seq_f32_d64_v1_l16"),
    make_variant<F32_S1_D_f, F32_S1_D_b>("seq_f32_d128_v4_l8"),
};
const WinVariant kSeqBF16[] = {
    make_variant<B16_S1_A_f, B16_S1_A_b>("seq_bf16_d64_v2_l32"),
    make_variant<B16_S1_B_f, B16_S1_B_b>("seq_bf16_d128_v2_l32"),
    make_variant<B16_S1_C_f, B16_S1_C_b>("seq_bf16_d128_v2_l16_s6"),
    make_variant<B16_S1_D_f, B16_S1_D_b>("seq_bf16_d256_v4_l16"),
};
const WinVariant kWinF32[] = {
    make_variant<F32_W_A_f, F32_W_A_b>("win_f32_d16_s16_l8"),
    make_variant<F32_W_B_f, F32_W_B_b>("win_f32_d32_s16_l8"),
    make_variant<F32_W_C_f, F32_W_C_b>("win_f32_d16_s32_l4"),
};
const WinVariant kWinBF16[] = {
    make_variant<B16_W_A_f, B16_W_A_b>("win_bf16_d32_s16_l8"),
    make_variant<B16_W_B_f, B16_W_B_b>("win_bf16_d64_s8_l16"),
};

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
