// Device-side building blocks shared by the lrscan kernels (sm_103a):
// storage traits, shared-memory barriers (mbarrier), bulk tensor copies
// (TMA), and bounded waits that report instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace lrscan {

// ----------------------------------------------------------------------------
// Device status word: the first error a kernel records sticks until the host
// reads and clears it (lrscan_sync_check).
// ----------------------------------------------------------------------------
struct DevStatus {
    int code;            // 0 or an LRSCAN_E* code
    int where;           // which wait gave up (see WaitSite)
    unsigned int block;  // linear CTA index that recorded it
    unsigned int pad;
};

enum WaitSite : int {
    kSiteConsumerFull = 1,   // consumer waiting for a tile to land
    kSiteProducerEmpty = 2,  // producer waiting for a stage to be released
    kSiteDrain = 3,          // producer draining copies in flight before exit
    kSiteSelftest = 4,
};

constexpr int kErrTimeout = -5;  // == LRSCAN_ETIMEOUT

// ----------------------------------------------------------------------------
// Storage traits.  bf16 values travel as raw 16-bit patterns; widening is
// exact (bits << 16), narrowing uses the hardware round-to-nearest-even cvt.
// ----------------------------------------------------------------------------
using bf16_t = uint16_t;

template <typename St, int V>
__device__ __forceinline__ void unpack_lanes(const St *p, float (&x)[V]) {
    if constexpr (std::is_same<St, float>::value) {
        if constexpr (V == 1) {
            x[0] = p[0];
        } else if constexpr (V == 2) {
            float2 t = *reinterpret_cast<const float2 *>(p);
            x[0] = t.x; x[1] = t.y;
        } else {
            static_assert(V == 4, "fp32 lanes per thread: 1, 2 or 4");
            float4 t = *reinterpret_cast<const float4 *>(p);
            x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
        }
    } else {
        static_assert(std::is_same<St, bf16_t>::value, "storage is float or bf16 bits");
        if constexpr (V == 1) {
            x[0] = __uint_as_float(static_cast<uint32_t>(p[0]) << 16);
        } else if constexpr (V == 2) {
            uint32_t u = *reinterpret_cast<const uint32_t *>(p);
            x[0] = __uint_as_float(u << 16);
            x[1] = __uint_as_float(u & 0xffff0000u);
        } else if constexpr (V == 4) {
            uint2 u = *reinterpret_cast<const uint2 *>(p);
            x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            static_assert(V == 8, "bf16 lanes per thread: 1, 2, 4 or 8");
            uint4 u = *reinterpret_cast<const uint4 *>(p);
            x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
            x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
            x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
        }
    }
}

// V storage elements as one packed register-sized value, and its widening.
template <typename St, int V> struct RawOf;
template <> struct RawOf<float, 1> { using T = float; };
template <> struct RawOf<float, 2> { using T = float2; };
template <> struct RawOf<float, 4> { using T = float4; };
template <> struct RawOf<bf16_t, 1> { using T = unsigned short; };
template <> struct RawOf<bf16_t, 2> { using T = uint32_t; };
template <> struct RawOf<bf16_t, 4> { using T = uint2; };
template <> struct RawOf<bf16_t, 8> { using T = uint4; };

template <typename St, int V>
__device__ __forceinline__ typename RawOf<St, V>::T load_raw(const St *p) {
    return *reinterpret_cast<const typename RawOf<St, V>::T *>(p);
}

// Widening works on the value (taking its address would force it to memory).
__device__ __forceinline__ void widen2(uint32_t u, float &lo, float &hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
}
__device__ __forceinline__ void widen_raw(float r, float (&x)[1]) { x[0] = r; }
__device__ __forceinline__ void widen_raw(float2 r, float (&x)[2]) { x[0] = r.x; x[1] = r.y; }
__device__ __forceinline__ void widen_raw(float4 r, float (&x)[4]) { x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w; }
__device__ __forceinline__ void widen_raw(unsigned short r, float (&x)[1]) {
    x[0] = __uint_as_float(static_cast<uint32_t>(r) << 16);
}
__device__ __forceinline__ void widen_raw(uint32_t r, float (&x)[2]) { widen2(r, x[0], x[1]); }
__device__ __forceinline__ void widen_raw(uint2 r, float (&x)[4]) { widen2(r.x, x[0], x[1]); widen2(r.y, x[2], x[3]); }
__device__ __forceinline__ void widen_raw(uint4 r, float (&x)[8]) {
    widen2(r.x, x[0], x[1]); widen2(r.y, x[2], x[3]); widen2(r.z, x[4], x[5]); widen2(r.w, x[6], x[7]);
}

// Read-only global variant (non-coherent path, may be cached in L1).
template <typename St, int V>
__device__ __forceinline__ void load_lanes_global(const St *__restrict__ p, float (&x)[V]) {
    if constexpr (std::is_same<St, float>::value) {
        if constexpr (V == 1) {
            x[0] = __ldg(p);
        } else if constexpr (V == 2) {
            float2 t = __ldg(reinterpret_cast<const float2 *>(p));
            x[0] = t.x; x[1] = t.y;
        } else {
            float4 t = __ldg(reinterpret_cast<const float4 *>(p));
            x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
        }
    } else {
        if constexpr (V == 1) {
            x[0] = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
        } else if constexpr (V == 2) {
            uint32_t u = __ldg(reinterpret_cast<const unsigned int *>(p));
            x[0] = __uint_as_float(u << 16);
            x[1] = __uint_as_float(u & 0xffff0000u);
        } else if constexpr (V == 4) {
            uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
            x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
            x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
            x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
            x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    // round-to-nearest-even of both halves; lo lands in the low 16 bits
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <typename St, int V>
__device__ __forceinline__ void store_lanes(St *p, const float (&x)[V]) {
    if constexpr (std::is_same<St, float>::value) {
        if constexpr (V == 1) {
            p[0] = x[0];
        } else if constexpr (V == 2) {
            *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
        } else if constexpr (V == 4) {
            *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
        } else {
            static_assert(V == 8, "fp32 stores of 1, 2, 4 or 8 lanes");
            *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4 *>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
        }
    } else {
        if constexpr (V == 1) {
            __nv_bfloat16 v = __float2bfloat16_rn(x[0]);
            p[0] = *reinterpret_cast<uint16_t *>(&v);
        } else if constexpr (V == 2) {
            *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(x[0], x[1]);
        } else if constexpr (V == 4) {
            *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
        } else {
            *reinterpret_cast<uint4 *>(p) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                                       pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
        }
    }
}

// ----------------------------------------------------------------------------
// PTX: shared-memory barriers and bulk tensor copies
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Programmatic dependent launch: the next kernel in the stream may be launched
// (and run its prologue) once every CTA of this one has triggered; each kernel
// waits for the previous grid's completion, and its memory, before it reads
// or writes any global memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 3-D tiled bulk copy global -> shared; completion is counted in bytes on `bar`.
// Coordinates are element indices {x: lane, y: time, z: batch row}; out-of-range
// parts of the box are filled with zeros.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// 3-D tiled bulk copy shared -> global, tracked by bulk groups.  Parts of the
// box outside the tensor are not written.  x * element size must be a
// multiple of 16 bytes and no coordinate may be negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *m, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed bulk groups still read shared memory.
template <int N> __device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N of this thread's committed bulk groups are incomplete.
template <int N> __device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Orders this thread's earlier shared-memory writes before later async-proxy
// (bulk copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (ids other than 0 are free for subsets),
// with an OR-reduction of a predicate: every participant learns whether any
// participant passed `flag` = true.
__device__ __forceinline__ bool bar_sync_or(int id, int count, bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(flag ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ----------------------------------------------------------------------------
// Bounded wait.  Spins on try_wait; every few tries it checks the CTA's abort
// flag and the elapsed global time.  On expiry it records the error once in
// the device status word, raises the CTA abort flag and returns false.
// ----------------------------------------------------------------------------
struct WaitCtx {
    DevStatus *status;
    volatile int *abort_flag;  // shared memory, per CTA
    uint64_t timeout_ns;
};

__device__ __forceinline__ void record_error(const WaitCtx &w, int code, int site) {
    if (atomicCAS(&w.status->code, 0, code) == 0) {
        w.status->where = site;
        w.status->block = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    }
    *w.abort_flag = 1;
}

static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const WaitCtx &w, int site) {
    const uint64_t start = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 15u) == 0) {
            if (*w.abort_flag) return false;
            if (global_timer_ns() - start > w.timeout_ns) {
                record_error(w, kErrTimeout, site);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx &w, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, w, site);
}

}  // namespace lrscan
