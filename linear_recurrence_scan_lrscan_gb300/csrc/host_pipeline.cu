// Host-buffer entry points (lrscan_fwd_host, lrscan_bwd_host,
// lrscan_fwd_bwd_host).  The [B, T, D] operands live in host memory; the call
// moves them through device memory in chunks of whole batch rows.  Each chunk
// runs the device entry points (lrscan_fwd_ex / lrscan_bwd_ex) on its rows.
// Copies in, kernels and copies out run on three streams, so chunk c's
// kernels overlap chunk c+1's copy in and chunk c-1's copy out.  Device
// staging is a set of slots; a slot is refilled only after its previous
// chunk's results have left the device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "lrscan.h"

namespace lrscan {
namespace {

constexpr int kSlots = 3;
constexpr int kMaxDev = 64;
constexpr int kTargetChunks = 16;            // chunks per call when the batch allows
constexpr size_t kSlotCap = size_t(1) << 30;  // staging per slot, unless one row needs more

struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, cmp = nullptr, out = nullptr;
    cudaEvent_t ev_in[kSlots], ev_cmp[kSlots], ev_out[kSlots];
    void *buf = nullptr;
    size_t bytes = 0;
    std::mutex mu;  // one host-buffer call at a time per device
};
Pipe g_pipe[kMaxDev];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

int pipe_ready(Pipe &p) {
    if (p.ready) return LRSCAN_OK;
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.cmp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < kSlots; ++i)
        ok = cudaEventCreateWithFlags(&p.ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.ev_cmp[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return report_error(LRSCAN_ECUDA, "creating the host-pipeline streams failed");
    }
    p.ready = true;
    return LRSCAN_OK;
}

// Device pointers of one slot handed to the per-chunk work: planes in the
// order the entry point lists them, then the fp32 [rows, D] final state.
struct SlotView {
    char *plane[7];
    float *last;
};

// What one call moves: `nplanes` [B, T, D] planes per slot, each copied in
// from host_in[i], out to host_out[i], both or neither; an optional fp32
// [B, D] last copied out; `run` launches one chunk's kernels.
struct Job {
    int nplanes;
    const void *host_in[7];   // host source per plane (nullptr: not copied in)
    void *host_out[7];        // host destination per plane (nullptr: not copied out)
    float *host_last;         // [B, D] (nullptr: none)
    int (*run)(const Job &, const SlotView &, int64_t rows, cudaStream_t st);
    int64_t T, D;
    int dtype;
    const lrscan_opts *opts;
};

int drain(Pipe &p) {
    const bool ok = cudaStreamSynchronize(p.in) == cudaSuccess && cudaStreamSynchronize(p.cmp) == cudaSuccess &&
                    cudaStreamSynchronize(p.out) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return report_error(LRSCAN_ECUDA, "a host-pipeline stream failed");
    }
    return LRSCAN_OK;
}

int run_job(const Job &job, int64_t B) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return report_error(LRSCAN_ENODEVICE, "no CUDA device");
    }
    Pipe &p = g_pipe[dev];
    std::lock_guard<std::mutex> lk(p.mu);
    int rc = pipe_ready(p);
    if (rc) return rc;
    const size_t es = job.dtype == LRSCAN_F32 ? 4 : 2;
    const size_t row_plane = static_cast<size_t>(job.T) * job.D * es;  // one batch row of one plane
    const size_t row_bytes = row_plane * job.nplanes + (job.host_last ? job.D * 4 : 0);
    int64_t rows = std::max<int64_t>(1, (B + kTargetChunks - 1) / kTargetChunks);
    rows = std::max<int64_t>(1, std::min<int64_t>(rows, static_cast<int64_t>(kSlotCap / std::max<size_t>(row_bytes, 1))));
    const int64_t nchunks = (B + rows - 1) / rows;
    const int nslots = static_cast<int>(std::min<int64_t>(kSlots, nchunks));
    const size_t plane_bytes = round256(row_plane * rows);
    const size_t last_bytes = job.host_last ? round256(static_cast<size_t>(job.D) * 4 * rows) : 0;
    const size_t slot_bytes = plane_bytes * job.nplanes + last_bytes;
    if (p.bytes < slot_bytes * nslots) {
        if (p.buf) cudaFree(p.buf);
        p.buf = nullptr;
        p.bytes = 0;
        if (cudaMalloc(&p.buf, slot_bytes * nslots) != cudaSuccess) {
            cudaGetLastError();
            return report_error(LRSCAN_ENOMEM, "cudaMalloc of the host-pipeline staging failed");
        }
        p.bytes = slot_bytes * nslots;
    }
    for (int64_t c = 0; c < nchunks; ++c) {
        const int s = static_cast<int>(c % nslots);
        const int64_t r0 = c * rows, nr = std::min<int64_t>(rows, B - r0);
        SlotView v{};
        char *base = static_cast<char *>(p.buf) + slot_bytes * s;
        for (int i = 0; i < job.nplanes; ++i) v.plane[i] = base + plane_bytes * i;
        v.last = job.host_last ? reinterpret_cast<float *>(base + plane_bytes * job.nplanes) : nullptr;
        const size_t n = row_plane * nr, off = row_plane * r0;
        bool ok = true;
        if (c >= nslots) ok = cudaStreamWaitEvent(p.in, p.ev_out[s], 0) == cudaSuccess;  // slot drained
        for (int i = 0; ok && i < job.nplanes; ++i)
            if (job.host_in[i])
                ok = cudaMemcpyAsync(v.plane[i], static_cast<const char *>(job.host_in[i]) + off, n,
                                     cudaMemcpyDefault, p.in) == cudaSuccess;
        ok = ok && cudaEventRecord(p.ev_in[s], p.in) == cudaSuccess &&
             cudaStreamWaitEvent(p.cmp, p.ev_in[s], 0) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            drain(p);
            return report_error(LRSCAN_ECUDA, "host-to-device copy failed");
        }
        if ((rc = job.run(job, v, nr, p.cmp))) {
            drain(p);
            return rc;
        }
        ok = cudaEventRecord(p.ev_cmp[s], p.cmp) == cudaSuccess &&
             cudaStreamWaitEvent(p.out, p.ev_cmp[s], 0) == cudaSuccess;
        for (int i = 0; ok && i < job.nplanes; ++i)
            if (job.host_out[i])
                ok = cudaMemcpyAsync(static_cast<char *>(job.host_out[i]) + off, v.plane[i], n, cudaMemcpyDefault,
                                     p.out) == cudaSuccess;
        if (ok && job.host_last)
            ok = cudaMemcpyAsync(job.host_last + r0 * job.D, v.last, static_cast<size_t>(nr) * job.D * 4,
                                 cudaMemcpyDefault, p.out) == cudaSuccess;
        ok = ok && cudaEventRecord(p.ev_out[s], p.out) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            drain(p);
            return report_error(LRSCAN_ECUDA, "device-to-host copy failed");
        }
    }
    if ((rc = drain(p))) return rc;
    return take_device_status(p.out);
}

int run_fwd_chunk(const Job &j, const SlotView &v, int64_t rows, cudaStream_t st) {
    return lrscan_fwd_ex(v.plane[0], v.plane[1], v.plane[2], v.last, rows, j.T, j.D, j.dtype, st, j.opts);
}

int run_bwd_chunk(const Job &j, const SlotView &v, int64_t rows, cudaStream_t st) {
    return lrscan_bwd_ex(v.plane[0], v.plane[1], v.plane[2], v.plane[3], v.plane[4], rows, j.T, j.D, j.dtype, st,
                         j.opts);
}

// planes: a, b, grad_out, out, grad_a, grad_b
int run_fwd_bwd_chunk(const Job &j, const SlotView &v, int64_t rows, cudaStream_t st) {
    const int rc = lrscan_fwd_ex(v.plane[0], v.plane[1], v.plane[3], v.last, rows, j.T, j.D, j.dtype, st, j.opts);
    if (rc) return rc;
    return lrscan_bwd_ex(v.plane[0], v.plane[3], v.plane[2], v.plane[4], v.plane[5], rows, j.T, j.D, j.dtype, st,
                         j.opts);
}

// Shared argument checks; returns 1 in *nothing when there is no work.
int host_checks(int64_t B, int64_t T, int64_t D, int dtype, float *last, int *nothing) {
    *nothing = 0;
    if (dtype != LRSCAN_F32 && dtype != LRSCAN_BF16) return report_error(LRSCAN_EDTYPE, "dtype is not f32 or bf16");
    if (B < 0 || T < 0 || D < 0 || T > 0x7fffffffLL || D > 0x7fffffffLL)
        return report_error(LRSCAN_EINVAL, "sizes must be >= 0 with T and D below 2^31");
    if (B == 0 || D == 0) {
        *nothing = 1;
        return LRSCAN_OK;
    }
    if (T == 0) {  // no steps: the final state is the zero initial state
        if (last) std::memset(last, 0, static_cast<size_t>(B) * D * sizeof(float));
        *nothing = 1;
    }
    return LRSCAN_OK;
}

}  // namespace
}  // namespace lrscan

using namespace lrscan;

extern "C" {

int lrscan_fwd_host(const void *a, const void *b, void *out, float *last, int64_t B, int64_t T, int64_t D,
                    int dtype, const lrscan_opts *opts) {
    int nothing = 0;
    int rc = host_checks(B, T, D, dtype, last, &nothing);
    if (rc || nothing) return rc;
    if (!a || !b || !out) return report_error(LRSCAN_EINVAL, "NULL a, b or out");
    Job j{};
    j.nplanes = 3;
    j.host_in[0] = a;
    j.host_in[1] = b;
    j.host_out[2] = out;
    j.host_last = last;
    j.run = run_fwd_chunk;
    j.T = T; j.D = D; j.dtype = dtype; j.opts = opts;
    return run_job(j, B);
}

int lrscan_bwd_host(const void *a, const void *out, const void *grad_out, void *grad_a, void *grad_b, int64_t B,
                    int64_t T, int64_t D, int dtype, const lrscan_opts *opts) {
    int nothing = 0;
    int rc = host_checks(B, T, D, dtype, nullptr, &nothing);
    if (rc || nothing) return rc;
    if (!a || !out || !grad_out || !grad_a || !grad_b)
        return report_error(LRSCAN_EINVAL, "NULL a, out, grad_out, grad_a or grad_b");
    Job j{};
    j.nplanes = 5;
    j.host_in[0] = a;
    j.host_in[1] = out;
    j.host_in[2] = grad_out;
    j.host_out[3] = grad_a;
    j.host_out[4] = grad_b;
    j.run = run_bwd_chunk;
    j.T = T; j.D = D; j.dtype = dtype; j.opts = opts;
    return run_job(j, B);
}

int lrscan_fwd_bwd_host(const void *a, const void *b, const void *grad_out, void *out, float *last, void *grad_a,
                        void *grad_b, int64_t B, int64_t T, int64_t D, int dtype, const lrscan_opts *opts) {
    int nothing = 0;
    int rc = host_checks(B, T, D, dtype, last, &nothing);
    if (rc || nothing) return rc;
    if (!a || !b || !grad_out || !out || !grad_a || !grad_b)
        return report_error(LRSCAN_EINVAL, "NULL a, b, grad_out, out, grad_a or grad_b");
    Job j{};
    j.nplanes = 6;
    j.host_in[0] = a;
    j.host_in[1] = b;
    j.host_in[2] = grad_out;
    j.host_out[3] = out;
    j.host_out[4] = grad_a;
    j.host_out[5] = grad_b;
    j.host_last = last;
    j.run = run_fwd_bwd_chunk;
    j.T = T; j.D = D; j.dtype = dtype; j.opts = opts;
    return run_job(j, B);
}

}  // extern "C"
