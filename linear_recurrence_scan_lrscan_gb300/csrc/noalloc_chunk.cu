// lrscan_fwd_chunk_noalloc: the three-phase chunked forward scan with its
// scratch in a fixed block of device memory that the library owns, so that a
// call allocates nothing.
//
// Who needs it: code that must not call cudaMalloc once it is running -- for
// example a caller inside a custom allocator or memory-pool callback (where a
// nested allocation would re-enter the allocator), a latency-critical loop
// that has banned allocation because cudaMalloc can synchronize the device,
// or an embedding that hands the library only pre-sized buffers.  The regular
// entry points grow a library-owned workspace with cudaMalloc on first use of
// the chunked path; this one never does.
//
// The scratch is one file-scope __device__ array: every GPU that loads the
// library holds LRSCAN_NOALLOC_SCRATCH_BYTES of it until the process exits,
// and every call on a device shares it.
#include <mutex>

#include "launch.h"
#include "lrscan.h"

namespace lrscan {
namespace {

// Device-side scratch for the chunk summaries P and Q.  Host code must not
// hand this name to a kernel: on the host it is only a stand-in symbol, so its
// device address is looked up with cudaGetSymbolAddress (per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[LRSCAN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch on the current device; looked up once per
// device, with that device current.
int noalloc_scratch(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return report_error(LRSCAN_ECUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LRSCAN_OK;
}

}  // namespace
}  // namespace lrscan

using namespace lrscan;

extern "C" int lrscan_fwd_chunk_noalloc(const void *a, const void *b, void *out, float *last, int64_t B, int64_t T,
                                        int64_t D, int dtype, int chunk_len, void *stream) {
    if (dtype != LRSCAN_F32 && dtype != LRSCAN_BF16) return report_error(LRSCAN_EDTYPE, "dtype is not f32 or bf16");
    if (B < 0 || T < 0 || D < 0 || T > 0x7fffffffLL || D > 0x7fffffffLL)
        return report_error(LRSCAN_EINVAL, "sizes must be >= 0 with T and D below 2^31");
    const int C = chunk_len ? chunk_len : 64;
    if (C != 16 && C != 32 && C != 64) return report_error(LRSCAN_EINVAL, "chunk_len must be 16, 32 or 64");
    if (B == 0 || D == 0) return LRSCAN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (last && cudaMemsetAsync(last, 0, static_cast<size_t>(B) * D * 4, st) != cudaSuccess)
            return report_error(LRSCAN_ECUDA, "cudaMemsetAsync of last failed");
        return LRSCAN_OK;
    }
    if (!a || !b || !out) return report_error(LRSCAN_EINVAL, "NULL a, b or out");
    // P and Q: fp32 [B, ceil(T/C), D] each, Q starting on a 256-byte boundary
    const unsigned long long nc = static_cast<unsigned long long>((T + C - 1) / C);
    unsigned long long n = 0, bytes = 0;
    const bool overflow = __builtin_mul_overflow(static_cast<unsigned long long>(B), nc, &n) ||
                          __builtin_mul_overflow(n, static_cast<unsigned long long>(D), &n) ||
                          __builtin_mul_overflow(n, 4ull, &bytes);
    const unsigned long long half = overflow ? 0 : (bytes + 255) / 256 * 256;
    if (overflow || half > LRSCAN_NOALLOC_SCRATCH_BYTES / 2)
        return report_error(LRSCAN_ENOMEM,
                            "problem needs more scratch than the no-alloc entry point holds "
                            "(2 * B * ceil(T/chunk_len) * D * 4 bytes > LRSCAN_NOALLOC_SCRATCH_BYTES)");
    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
        minor != 3) {
        cudaGetLastError();
        return report_error(LRSCAN_ENODEVICE, "no sm_103 device is current");
    }
    void *scratch = nullptr;
    int rc = noalloc_scratch(dev, &scratch);
    if (rc) return rc;
    const int es = dtype == LRSCAN_F32 ? 4 : 2;
    const int vmax = dtype == LRSCAN_F32 ? 4 : 8;
    const bool aligned = (reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                          reinterpret_cast<uintptr_t>(out)) % 16 == 0 &&
                         (D * es) % 16 == 0;
    ChunkLaunch L{};
    L.in0 = a;
    L.in1 = b;
    L.out0 = out;
    L.last = last;
    L.P = static_cast<float *>(scratch);
    L.Q = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + half);
    L.B = B;
    L.T = T;
    L.D = D;
    L.chunk = C;
    L.vec = (aligned && D % vmax == 0) ? vmax : 1;
    L.stream = st;
    // Nothing in the scratch has to start at zero: the summary pass writes every
    // P and Q it later reads, so a call never sees the previous call's values.
    rc = chunk_fwd(L, dtype);
    if (rc) {
        return report_error(LRSCAN_ECUDA, cudaGetErrorString(cudaGetLastError()));
    }
    return LRSCAN_OK;
}
