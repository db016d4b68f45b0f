// Internal interface between the host dispatcher (lrscan_abi.cu) and the
// translation units that instantiate and launch the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "state_args.h"
#include "stream_args.h"

namespace lrscan {

// Launches a kernel that may overlap the tail of the previous kernel in the
// stream (programmatic dependent launch); the kernel itself calls pdl_wait()
// before touching global memory, so stream order is kept for the data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct DevStatus;

enum PathId : int { kPathAuto = 0, kPathSeq = 1, kPathChunk = 2, kPathWindow = 3, kPathPlain = 4, kPathStream = 5 };

// Arguments of one time-tiled launch (forward: maps a,b / out0=out;
// backward: maps a,out,grad_out / out0=grad_a, out1=grad_b).
struct WinLaunch {
    const CUtensorMap *maps[10];  // planes in kernel order (complex backward: 6 in, 4 out)
    void *out0;
    void *out1;
    void *out2, *out3;            // complex backward: grad_br, grad_bi
    float *last;
    float *last_i;                // complex forward: Im of the final state
    int64_t B, T, D;
    DevStatus *status;
    uint64_t timeout_ns;
    cudaStream_t stream;
    int device;
    StateArgs sx;  // carried state and resets (used by the EXT launchers only)
    CStateArgs csx;  // the complex scan's carried state (complex EXT launchers)
    // generated-decay scan: per-token / per-lane parameters, backward partial
    // sums, and the plain kernels' tensor inputs (in0 = b or out, in1 = grad_out)
    const float *eta, *nu_log;
    float *part_eta, *part_nu;
    int64_t part_rows;            // column stride of part_eta: rows B*T of the whole call
    const void *in0, *in1;
    StreamArgs sa;                // persistent chunk-streaming kernels: publication workspace
    int grid;                     // persistent chunk-streaming kernels: CTAs to launch
};

// One direction of a tile variant: compiled shape (DT, V, L) plus the
// launch-time sub-chunk count S and pipeline depth.
struct WinDirCfg {
    int dt;          // lanes per CTA
    int v;           // lanes per thread
    int l;           // steps per sub-chunk (registers)
    int s;           // sub-chunks per window
    int lane_scan;   // windowed prefix by lane threads (1) or per thread (0)
    int exact;       // results bit-identical to the sequential definition (1)
    int w;           // rows per window = s*l
    int nstage;      // pipeline depth
    int threads;     // s*(dt/v) + 32
    int smem;        // dynamic shared memory bytes
    int stage_bytes;
    int max_resident;  // CTAs per SM the registers allow (0: not limited beyond threads and shared memory)
    int (*launch)(const WinLaunch &, const WinDirCfg &);        // plain scan
    int (*launch_state)(const WinLaunch &, const WinDirCfg &);  // with carried state / resets
};

struct WinVariant {
    const char *name;
    WinDirCfg fwd, bwd;
};

// path: kPathSeq or kPathWindow; dtype 0 = f32, 1 = bf16
const WinVariant *win_variants(int path, int dtype, int *count);

// Persistent chunk-streaming variants (kernels_stream.cu); dtype 0 = f32,
// 1 = bf16.
const WinVariant *stream_variants(int dtype, int *count);
// The same kernels on the complex scan's re / im planes.
const WinVariant *cstream_variants(int dtype, int *count);

// Complex scan tile variants (kernels_complex.cu); dtype 0 = f32, 1 = bf16.
const WinVariant *cwin_variants(int dtype, int *count);

// Generated-decay scan (kernels_gated.cu): tile variants, the plain
// kernels, and the partial-sum reduction (part_eta [ncol][rows], part_nu
// [nu_rows][D]; both column sums are scaled by ln 2).
const WinVariant *gwin_variants(int dtype, int *count);
int gplain_launch(const WinLaunch &L, int dtype, bool fwd);
int gated_finish_launch(const float *part_eta, int ncol, long long rows, float *grad_eta, const float *part_nu,
                        int nu_rows, int D, float *grad_nu_log, cudaStream_t stream);
// Most sub-chunks a windowed generated-decay backward tile uses (rows of its
// grad_nu_log partials per batch row).
constexpr int kGatedMaxS = 16;

// Three-phase chunked path and plain kernels (kernels_chunk.cu).
struct ChunkLaunch {
    const void *in0, *in1, *in2;  // fwd: a, b; bwd: a, out, grad_out
    void *out0, *out1;            // fwd: out; bwd: grad_a, grad_b
    float *last;
    float *P, *Q;                 // workspace [B, Nc, D] each
    float *PG, *QG;               // grouped prefix: [B, ceil(Nc / kGroupChunks), D] each, or null (flat prefix)
    int64_t B, T, D;
    int chunk;                    // 16, 32, 64
    int vec;                      // lanes per thread: 1, 2, 4 (f32) / 1, 2, 4, 8 (bf16)
    cudaStream_t stream;
    StateArgs sx;                 // carried state and resets (all null: plain scan)
};
// Chunks per group of the grouped chunk prefix.
constexpr int kGroupChunks = 512;
int chunk_fwd(const ChunkLaunch &L, int dtype);
int chunk_bwd(const ChunkLaunch &L, int dtype);
int plain_fwd_launch(const ChunkLaunch &L, int dtype);
int plain_bwd_launch(const ChunkLaunch &L, int dtype);
// Complex plain kernels: forward in0 = ar, in1 = br, out0 = out_r, last = last_r
// plus the imaginary planes; backward in = {ar, ai, out_r, out_i, go_r, go_i},
// out = {grad_ar, grad_ai, grad_br, grad_bi}.
int cplain_fwd_launch(const ChunkLaunch &L, const void *ai, const void *bi, void *out_i, float *last_i, int dtype);
int cplain_bwd_launch(const void *const in[6], void *const out[4], int64_t B, int64_t T, int64_t D, int dtype,
                      cudaStream_t stream);
// Complex chunked path.  Forward: in = {ar, ai, br, bi}, out = {out_r,
// out_i}, last_r / last_i (may be null); backward: in = {ar, ai, out_r,
// out_i, go_r, go_i}, out = {grad_ar, grad_ai, grad_br, grad_bi}.  maps: P re,
// P im, Q re, Q im [B, Nc, D] each; gmaps: the grouped prefix's group maps
// [B, ceil(Nc / kGroupChunks), D] each, or all null (flat prefix).
struct CChunkLaunch {
    const void *in[6];
    void *out[4];
    float *last_r, *last_i;
    float *maps[4];
    float *gmaps[4];
    int64_t B, T, D;
    int chunk;
    int vec;  // lanes per thread: 4 on 16-byte aligned rows, else 1
    cudaStream_t stream;
    CStateArgs sx;
};
int cchunk_fwd_launch(const CChunkLaunch &L, int dtype);
int cchunk_bwd_launch(const CChunkLaunch &L, int dtype);
// Whole-sequence affine summary per lane (dir 0: forward, 1: backward);
// in0 = a, in1 = b or grad_out, P and Q = [B, D] outputs.
int summary_launch(const ChunkLaunch &L, int dtype, int dir);
int fill_f32_launch(float *p, size_t n, float v, cudaStream_t stream);
// out = fold of h -> P_r*h + Q_r over n maps r = r0, r0+step, ... of maps [W][2][lanes].
int compose_maps_launch(const float *maps, const float *init, float *out, long long lanes, int r0, int step, int n,
                        cudaStream_t stream);
int selftest_wait_launch(DevStatus *status, uint64_t timeout_ns, cudaStream_t stream);

// Records the detail text lrscan_last_error() returns and passes code through.
int report_error(int code, const char *msg);
// Reads and clears the device status word after `st` drains (lrscan_abi.cu).
int take_device_status(cudaStream_t st);

}  // namespace lrscan
