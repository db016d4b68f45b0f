// Host side of liblrscan.so: argument checks, the occupancy rule that picks
// a path, tensor-map encoding, workspace management and the exported C ABI
// declared in include/lrscan.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <map>
#include <mutex>

#include "launch.h"
#include "lrscan.h"
#include "scan_common.cuh"

namespace lrscan {

// One status word per device (module globals are instantiated per device).
__device__ DevStatus g_status;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceCtx {
    bool ready = false;
    int sm_count = 0;
    int smem_per_sm = 0;
    int smem_optin = 0;
    int max_threads_per_sm = 2048;
    DevStatus *status = nullptr;
    std::map<cudaStream_t, std::pair<void *, size_t>> workspace;  // library-owned, per stream
};

std::mutex g_mu;
DeviceCtx g_dev[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
thread_local cudaStream_t t_stream = nullptr;
thread_local char t_detail[256] = "";

// Records why a call failed (read back by lrscan_last_error) and returns code.
int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(t_detail, sizeof t_detail, fmt, ap);
    va_end(ap);
    return code;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Description used when no device is visible (plans only): one GB300.
constexpr int kRefSMs = 152, kRefSmemPerSM = 233472, kRefSmemOptin = 232448;

thread_local int t_ctx_dev = -1;

int device_ctx(DeviceCtx **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return LRSCAN_ENODEVICE;
    }
    if (t_ctx_dev != dev) {
        // A thread that has not touched the runtime yet (e.g. an autograd
        // worker) has no current context; the tensor-map encoder needs one.
        if (cudaSetDevice(dev) != cudaSuccess) {
            cudaGetLastError();
            return LRSCAN_ENODEVICE;
        }
        t_ctx_dev = dev;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceCtx &c = g_dev[dev];
    if (!c.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return LRSCAN_ENODEVICE;
        }
        if (major != 10 || minor != 3) return LRSCAN_ENODEVICE;  // kernels are built for sm_103a only
        cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&c.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&c.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&c.max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
            cudaGetLastError();
            return LRSCAN_ECUDA;
        }
        c.status = static_cast<DevStatus *>(p);
        if (g_encode == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                cudaGetLastError();
                return LRSCAN_ECUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        c.ready = true;
    }
    *out = &c;
    return LRSCAN_OK;
}

struct Geometry {
    int sm_count, smem_per_sm, smem_optin, max_threads_per_sm;
};

Geometry geometry_of(const DeviceCtx *c) {
    if (c) return {c->sm_count, c->smem_per_sm, c->smem_optin, c->max_threads_per_sm};
    return {kRefSMs, kRefSmemPerSM, kRefSmemOptin, 2048};
}

int esize(int dtype) { return dtype == LRSCAN_F32 ? 4 : 2; }

// -------------------------------------------------------------------------
// Occupancy rule
// -------------------------------------------------------------------------
struct Choice {
    int path = kPathSeq;
    int vidx = 0;                 // index into the path's variant table
    const WinVariant *var = nullptr;
    int chunk = 64;
    int vec = 1;
    size_t workspace = 0;
    long long ctas = 0;
    int threads = 0, smem = 0, stages = 0, kernels = 1;
    int dir = 0;
};

struct Occ {
    long long ctas;
    int resident;    // CTAs per SM that fit
    bool one_wave;
    double inflight; // bytes in flight per SM, estimated
};

const WinDirCfg &dir_of(const WinVariant &v, int dir) { return dir == 0 ? v.fwd : v.bwd; }

Occ occupancy(const WinVariant &var, int dir, int64_t B, int64_t D, const Geometry &g) {
    const WinDirCfg &v = dir_of(var, dir);
    const int smem = v.smem;
    const int nst = v.nstage;
    const int stage = v.stage_bytes;
    Occ o{};
    o.ctas = B * ((D + v.dt - 1) / v.dt);
    // the kernels' named barriers and mbarrier arrival counts take whole
    // warps: a table entry whose threads are not whole warps never launches
    if (v.threads < 32 || v.threads % 32 != 0) return o;
    int r_smem = smem > g.smem_optin ? 0 : g.smem_per_sm / (smem + 1024);
    int r_thr = g.max_threads_per_sm / v.threads;
    o.resident = std::min(std::min(r_smem, r_thr), 32);
    o.one_wave = o.resident > 0 && o.ctas <= static_cast<long long>(o.resident) * g.sm_count;
    const double per_sm = std::min<double>(static_cast<double>(o.ctas) / g.sm_count, o.resident);
    o.inflight = per_sm * (nst - 1) * stage;
    return o;
}

// Chunk scratch: P and Q [B, Nc, D] fp32, then (grouped prefix) the group
// maps PG and QG [B, NG, D]; each array rounded up to 256 bytes.
struct ChunkScratch {
    size_t pq;      // bytes of P (= of Q)
    size_t group;   // bytes of PG (= of QG), 0 without groups
    size_t total() const { return 2 * pq + 2 * group; }
};
ChunkScratch chunk_scratch(int64_t B, int64_t T, int64_t D, int C, bool grouped) {
    const int64_t nc = (T + C - 1) / C;
    const int64_t ng = (nc + kGroupChunks - 1) / kGroupChunks;
    auto pad = [](size_t x) { return (x + 255) / 256 * 256; };
    ChunkScratch s;
    s.pq = pad(static_cast<size_t>(B) * nc * D * 4);
    s.group = grouped ? pad(static_cast<size_t>(B) * ng * D * 4) : 0;
    return s;
}
size_t chunk_workspace(int64_t B, int64_t T, int64_t D, int C, bool grouped = true) {
    return chunk_scratch(B, T, D, C, grouped).total();
}

// Chunk-streaming workspace: the ticket word (first 256 bytes), then the
// chunk maps (float2 per lane) and leaving states (float per lane); before
// every launch the ticket is zeroed and the maps and states are filled with
// all-ones words (nothing published).
struct StreamScratch {
    size_t agg, incl;  // byte sizes, padded to 256
    size_t head() const { return 256; }
    size_t total() const { return head() + agg + incl; }
};
StreamScratch stream_scratch(int64_t ng, int64_t nc, int dt, int k = 1) {  // k = 2: complex maps and states
    auto pad = [](size_t x) { return (x + 255) / 256 * 256; };
    StreamScratch s;
    s.agg = pad(static_cast<size_t>(ng) * nc * dt * 8 * k);
    s.incl = pad(static_cast<size_t>(ng) * nc * dt * 4 * k);
    return s;
}

// The plan of a chunk-streaming call on variant vi of tab (k = 2: the
// complex scan's maps and states).
int plan_stream_variant(const WinVariant *tab, int vi, int dir, int64_t B, int64_t T, int64_t D, int k,
                        const Geometry &g, Choice *ch) {
    const WinDirCfg &v = dir_of(tab[vi], dir);
    const Occ o = occupancy(tab[vi], dir, B, D, g);
    if (o.resident == 0) return fail(LRSCAN_EINVAL, "stream variant %s does not fit on an SM", tab[vi].name);
    const int64_t ng = B * ((D + v.dt - 1) / v.dt);
    const int64_t rows = static_cast<int64_t>(v.s) * v.w;  // windows x rows each
    const int64_t nc = (T + rows - 1) / rows;
    if (ng * nc > 0x7fffffffLL) return fail(LRSCAN_EINVAL, "too many chunks for the streaming path");
    ch->vidx = vi;
    ch->var = &tab[vi];
    ch->chunk = static_cast<int>(rows);
    // One CTA per SM (no more than there are chunk tickets).  A chunk's tiles
    // must still be in L2 when its replay reads them: with two chunk buffers a
    // CTA holds at most about two and a half chunks of input planes between
    // summaries and replays (512-step fp32 chunks: 40 MB over 152 SMs).
    const int resident = v.max_resident > 0 ? std::min(o.resident, v.max_resident) : o.resident;
    ch->ctas = std::min<long long>(ng * nc, static_cast<long long>(resident) * g.sm_count);
    ch->threads = v.threads;
    ch->smem = v.smem;
    ch->stages = v.nstage;
    ch->dir = dir;
    ch->kernels = 1;
    ch->workspace = stream_scratch(ng, nc, v.dt, k).total();
    return LRSCAN_OK;
}

// The grouped prefix pays when every lane has many chunks and the lanes alone
// give the GPU few warps to run the flat per-lane prefix.
bool use_grouped_prefix(int64_t B, int64_t T, int64_t D, int C, const Geometry &g) {
    const int64_t nc = (T + C - 1) / C;
    return nc >= 4 * kGroupChunks && B * D < 32LL * g.sm_count;
}

int pick_from_table(const WinVariant *tab, int n, int dir, int64_t B, int64_t D, const Geometry &g, int *vidx) {
    int best = -1;
    double best_score = -1;
    for (int i = 0; i < n; ++i) {
        Occ o = occupancy(tab[i], dir, B, D, g);
        if (o.resident == 0) continue;
        if (o.ctas < static_cast<long long>(0.9 * g.sm_count)) continue;
        // Prefer a single wave (every CTA resident: no tail); past one wave,
        // prefer the fullest last wave.  Then more bytes in flight per SM, then
        // wider rows (longer DRAM bursts).
        const double slots = static_cast<double>(o.resident) * g.sm_count;
        const double waves = std::ceil(static_cast<double>(o.ctas) / slots);
        const double fill = static_cast<double>(o.ctas) / (waves * slots);
        const double score = (o.one_wave ? 2e6 : 1e6 * fill) + std::min(o.inflight, 96.0 * 1024) +
                             dir_of(tab[i], dir).dt * sizeof(float);
        if (score > best_score) {
            best_score = score;
            best = i;
        }
    }
    *vidx = best;
    return best >= 0;
}

int pick_window_variant(int path, int dtype, int dir, int64_t B, int64_t D, const Geometry &g, int *vidx) {
    int n = 0;
    const WinVariant *tab = win_variants(path, dtype, &n);
    return pick_from_table(tab, n, dir, B, D, g, vidx);
}

// The occupancy rule.  For each (dtype, direction), tile variants in order of
// preference, each with the range of CTAs per SM (as multiples of the SM
// count) in which it is the fastest measured choice; the first that
// qualifies (and fits on an SM) wins.  The order comes from timing every
// variant on the five named workloads on GB300: where the lanes alone give
// each SM too little to do, the windowed path splits time inside the CTA and
// keeps far more warps busy on the same lanes (the high-residency bf16
// forward tile puts all 640 CTAs of the gated workload in one wave); the
// fp32 forward prefers the sequential path, bit-identical to the sequential
// definition and as fast wherever the lanes give each SM two CTAs.
struct Pref {
    int path;
    const char *name;
    double min_ctas_per_sm;
    double max_ctas_per_sm;
};
constexpr double kAny = 1e30;
// Exact tiles come first wherever they hold the rate: the sequential tiles,
// and the windowed tiles whose lane threads walk the window's rows with the
// sequential step (xwin_*), reproduce the sequential definition bit for bit.
// fp32 forward with few lane tiles: one 32-warp CTA per tile (31 sub-chunks
// of 8 rows): 333.6 us on the long fp32 workload against 372.5 us for 16
// sub-chunks.
// With many lane tiles, the 64-lane one-lane-per-thread tile with a three-stage
// ring (61.4 us on the padded workload against 63.4 us for the 32-lane tile).
const Pref kPrefF32Fwd[] = {{kPathSeq, "seq_f32_d64_v1_n3", 3.0, kAny},
                            {kPathSeq, "seq_f32_d32", 1.5, kAny},
                            {kPathWindow, "win_f32_d32_s31", 0.45, kAny}};
// fp32 backward with many lane tiles: the exact 64-lane window tile (102.1 us
// on the padded workload against 100.0 us for the re-associating one and
// 105.7 us for the fastest sequential tile)
const Pref kPrefF32Bwd[] = {{kPathWindow, "xwin_f32_d64_s8", 3.0, kAny},
                            {kPathWindow, "win_f32_d64_s8", 3.0, kAny},
                            {kPathWindow, "win_f32_d32_s16", 0.45, kAny}};
// bf16 forward: the sequential 128-lane tile with a three-stage ring (four
// CTAs resident per SM, so 512 tiles run in one wave) from two CTAs per SM
// (245.9 us on the near-unit workload, exact, against 241.0 us for the
// re-associating window tile and 259.2 us for the six-stage four-lane tile,
// 1.68 waves); fewer lanes: the one-wave window tile (42.1 us on the gated
// workload against 49.3 us for the fastest sequential tile and 56.0 us for the
// exact window tile).
const Pref kPrefBF16Fwd[] = {{kPathSeq, "seq_bf16_d128_n3", 2.0, kAny},
                             {kPathWindow, "win_bf16_d32_s8_m5_n2", 0.9, kAny},
                             {kPathSeq, "seq_bf16_d64_v1", 1.5, kAny},
                             {kPathWindow, "win_bf16_d32_s16", 0.9, kAny}};
// bf16 backward: from five 64-lane tiles per SM the wavefront exact tile (one
// warp per 16-row sub-chunk, the chain handed from warp to warp: 407.9 us on
// the near-unit workload, exact, against 404.0 us re-associating); from two
// 128-lane tiles per SM the sequential tile with a two-stage ring (417.1 us
// there, exact, four CTAs per SM, one wave); up to 5 CTAs per SM the
// wavefront tile with three 16-row sub-chunks of 32 lanes, five CTAs per SM
// (70.7 us on the gated workload, exact, against 73.4 us for the fastest
// re-associating tile and 73.7 us for the exact walk-and-replay tile).
const Pref kPrefBF16Bwd[] = {{kPathWindow, "wfx_bf16_d64_s4_l16_v2", 5.0, kAny},
                             {kPathSeq, "seq_bf16_d128_n2", 2.0, kAny},
                             {kPathWindow, "wfx_bf16_d32_s3_l16", 0.9, 5.0},
                             {kPathWindow, "xwin_bf16_d32_s8_m5_n2", 0.9, 5.0},
                             {kPathWindow, "win_bf16_d32_l4_s12_m5", 0.9, 5.0},
                             {kPathWindow, "win_bf16_d32_l16_s8", 0.9, kAny},
                             {kPathWindow, "win_bf16_d64_s8", 0.45, kAny}};
// With carried state / resets: the 16-sub-chunk tiles (80.7 us on the gated
// workload against 81.3 us for the 12-sub-chunk tile and 93.5 us for the
// five-CTA 8-row tile, whose reset masks and grad_last / grad_h0 work spill).
const Pref kPrefBF16BwdState[] = {{kPathWindow, "win_bf16_d32_s16_n4", 0.9, 5.0},
                                  {kPathWindow, "win_bf16_d32_s16_n2", 0.9, kAny},
                                  {kPathWindow, "win_bf16_d64_s8", 0.45, kAny}};

bool auto_candidate(int dtype, int dir, bool ext, int64_t B, int64_t D, const Geometry &g, int *path, int *vidx) {
    const Pref *list;
    int n;
    if (dtype == LRSCAN_F32) {
        list = dir == 0 ? kPrefF32Fwd : kPrefF32Bwd;
        n = dir == 0 ? static_cast<int>(std::size(kPrefF32Fwd)) : static_cast<int>(std::size(kPrefF32Bwd));
    } else if (dir == 0) {
        list = kPrefBF16Fwd;
        n = static_cast<int>(std::size(kPrefBF16Fwd));
    } else {
        list = ext ? kPrefBF16BwdState : kPrefBF16Bwd;
        n = ext ? static_cast<int>(std::size(kPrefBF16BwdState)) : static_cast<int>(std::size(kPrefBF16Bwd));
    }
    for (int i = 0; i < n; ++i) {
        int cnt = 0;
        const WinVariant *tab = win_variants(list[i].path, dtype, &cnt);
        for (int v = 0; v < cnt; ++v) {
            if (std::strcmp(tab[v].name, list[i].name) != 0) continue;
            const Occ o = occupancy(tab[v], dir, B, D, g);
            const double per_sm = static_cast<double>(o.ctas) / g.sm_count;
            if (o.resident > 0 && per_sm >= list[i].min_ctas_per_sm && per_sm <= list[i].max_ctas_per_sm) {
                *path = list[i].path;
                *vidx = v;
                return true;
            }
        }
    }
    return false;
}

// ext: the call carries state or resets (lrscan_fwd_state / lrscan_bwd_state).
int plan_call(int64_t B, int64_t T, int64_t D, int dtype, int dir, bool aligned16, const lrscan_opts *opts,
              const Geometry &g, Choice *ch, bool ext = false) {
    const int want = opts ? opts->path : 0;
    const int force_v = opts ? opts->tile_variant : 0;
    int chunk = opts && opts->chunk_len ? opts->chunk_len : 64;
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128 && chunk != 256 && chunk != 512)
        return fail(LRSCAN_EINVAL, "chunk_len %d is not 16, 32, 64, 128, 256 or 512", chunk);
    ch->chunk = chunk;
    const int vmax = dtype == LRSCAN_F32 ? 4 : 8;
    ch->vec = (aligned16 && D % vmax == 0) ? vmax : 1;

    int path = want;
    if (want < kPathAuto || want > kPathStream) return fail(LRSCAN_EINVAL, "unknown path %d", want);

    if ((path == kPathSeq || path == kPathWindow || path == kPathStream) && !aligned16)
        return fail(LRSCAN_EINVAL, "path %d needs 16-byte aligned pointers and rows (D*elem %% 16 == 0)", path);
    int auto_vi = -1;
    if (path == kPathAuto) {
        if (!aligned16) {
            path = (B * D < 32LL * g.sm_count * 32 && T >= 16LL * chunk) ? kPathChunk : kPathPlain;
        } else if (auto_candidate(dtype, dir, ext, B, D, g, &path, &auto_vi)) {
            // measured preference list (see auto_candidate)
        } else if (T >= 16LL * chunk) {
            // too few lanes for a lane-tiled walk to fill the GPU: parallelize
            // over time chunks instead, in one pass (chunk streaming) from 32
            // chunks of 512 steps per lane group (measured against the three
            // chunked phases, fp32 forward / backward: B=1 T=2^22 D=64 0.52 /
            // 0.97 against 0.87 / 1.25 ms; B=1 T=2^14 D=64 26 / 23 against
            // 33 / 54 us; B=4 T=2^16 D=256 0.16 / 0.26 against 0.27 / 0.39 ms),
            // else (or with a chunk length asked for) in three chunked phases
            path = kPathChunk;
            const bool long_seq = T >= 32LL * 512;
            if (long_seq && !(opts && opts->chunk_len)) path = kPathStream;
        } else {
            path = kPathSeq;  // small problem: latency-bound whatever runs it
        }
    }
    ch->path = path;
    if (path == kPathSeq || path == kPathWindow) {
        int n = 0;
        const WinVariant *tab = win_variants(path, dtype, &n);
        int vi = -1;
        if (force_v > 0) {
            if (force_v > n) return fail(LRSCAN_EINVAL, "tile_variant %d > %d variants", force_v, n);
            vi = force_v - 1;
        } else if (auto_vi >= 0) {
            vi = auto_vi;
        } else if (!pick_window_variant(path, dtype, dir, B, D, g, &vi)) {
            // too few lanes to fill the GPU (or too many for one wave): take the
            // variant with the most CTAs that still fits on an SM
            long long most = -1;
            for (int i = 0; i < n; ++i) {
                Occ o = occupancy(tab[i], dir, B, D, g);
                if (o.resident == 0) continue;
                if (o.ctas > most) { most = o.ctas; vi = i; }
            }
        }
        if (vi < 0) return fail(LRSCAN_EINVAL, "no tile variant fits this device");
        ch->vidx = vi;
        ch->var = &tab[vi];
        Occ o = occupancy(tab[vi], dir, B, D, g);
        if (o.resident == 0) return fail(LRSCAN_EINVAL, "tile variant %s does not fit on an SM", tab[vi].name);
        ch->ctas = o.ctas;
        ch->threads = dir_of(tab[vi], dir).threads;
        ch->smem = dir_of(tab[vi], dir).smem;
        ch->stages = dir_of(tab[vi], dir).nstage;
        ch->dir = dir;
        ch->kernels = 1;
        ch->workspace = 0;
    } else if (path == kPathStream) {
        int n = 0;
        const WinVariant *tab = stream_variants(dtype, &n);
        if (force_v > n) return fail(LRSCAN_EINVAL, "tile_variant %d > %d variants", force_v, n);
        // Measured on few-lane long sequences (fraction of the copy rate):
        // fp32 forward, 512- against 256-step chunks: 0.92 / 0.73 at two 32-lane
        // groups (B=1 D=64), 0.89 / 0.81 at four, 0.89 / 0.89 and 0.80 / 0.88 at
        // eight (B=1 D=256, B=4 D=64), 0.77 / 0.89 at sixteen; the fp32 backward
        // takes 256-step chunks in both variants.  bf16: the first variant
        // (eight summary and eight replay warps on 32-lane tiles) in both
        // directions, 0.78-0.81 forward and 0.84-0.93 backward at B=1 D=64,
        // B=1 D=256 and B=8 D=64 against at most 0.75 and 0.88 for the 64-lane
        // variants; with carried state and resets bf16 takes the 64-lane tile
        // in 512-step chunks (B=1 T=2^22 D=64: forward 0.36 against 0.38 ms,
        // backward 0.53 against 0.58 ms; B=1 T=2^20 D=256: 0.34 / 0.52
        // against 0.38 / 0.57 ms)
        // The bf16 forward from four 64-lane groups takes the 64-lane tile, its
        // two lanes per thread stepping in packed fp32x2 instructions (B=1
        // T=2^20 D=256: 0.279 against 0.294 ms; B=8 T=2^18 D=64: 0.151 against
        // 0.160 ms; one group, B=1 D=64: 0.323 against 0.304 ms).
        int vi = force_v > 0 ? force_v - 1 : 0;
        if (force_v == 0 && dtype == LRSCAN_F32) vi = dir == 0 && B * ((D + 31) / 32) >= 8 ? 1 : 0;
        if (force_v == 0 && dtype == LRSCAN_BF16 && (ext || (dir == 0 && B * ((D + 63) / 64) >= 4))) vi = 1;
        return plan_stream_variant(tab, vi, dir, B, T, D, 1, g, ch);
    } else if (path == kPathChunk) {
        // variant 1: flat per-lane prefix; variant 2: grouped prefix
        if (force_v > 2) return fail(LRSCAN_EINVAL, "the chunked path has two variants (1 flat, 2 grouped prefix)");
        bool grouped = force_v ? force_v == 2 : use_grouped_prefix(B, T, D, chunk, g);
        if (grouped && !(opts && opts->chunk_len)) {
            // Long sequences on few lanes: longer chunks shrink the map walk.
            // Measured on B=1 T=2^22 D=64 fp32 against 64-step chunks: the
            // forward is fastest at 512 (0.86 ms against 0.92 at 128; 1024 is
            // slower), the backward at 128 (its data phases slow down past 128).
            const int want_c = dir == 0 ? 512 : 128;
            for (int c = want_c; c > chunk; c >>= 1)
                if (use_grouped_prefix(B, T, D, c, g)) {
                    chunk = c;
                    break;
                }
            ch->chunk = chunk;
        }
        const int64_t nc = (T + chunk - 1) / chunk;
        ch->vidx = grouped ? 1 : 0;
        // 128-thread CTAs; several chunks per CTA when a chunk row needs <= 64 threads
        const int64_t row_threads = (D + ch->vec - 1) / ch->vec;
        int64_t lt = 1;
        while (lt < row_threads && lt < 128) lt <<= 1;
        const int64_t cpb = row_threads <= 64 ? 128 / lt : 1;
        const int64_t nlb = row_threads <= 64 ? 1 : (row_threads + 127) / 128;
        ch->ctas = B * ((nc + cpb - 1) / cpb) * nlb;
        ch->threads = 128;
        ch->kernels = grouped ? 5 : 3;
        ch->workspace = chunk_workspace(B, T, D, chunk, grouped);
    } else {  // plain
        if (force_v > 1) return fail(LRSCAN_EINVAL, "the plain path has one variant");
        ch->ctas = B * ((D + 127) / 128);
        ch->threads = 128;
        ch->kernels = 1;
        ch->vec = 1;
    }
    return LRSCAN_OK;
}

void fill_info(const Choice &c, lrscan_plan_info *info) {
    std::memset(info, 0, sizeof *info);
    info->path = c.path;
    info->tile_variant = c.vidx + 1;
    info->ctas = static_cast<int>(std::min<long long>(c.ctas, 0x7fffffff));
    info->threads_per_cta = c.threads;
    info->smem_bytes = c.smem;
    info->stages = c.stages;
    info->kernels = c.kernels;
    info->workspace_bytes = c.workspace;
    info->subchunks = 1;
    info->exact = c.var ? dir_of(*c.var, c.dir).exact : (c.path == kPathPlain ? 1 : 0);
    if (c.var) {
        const WinDirCfg &d = dir_of(*c.var, c.dir);
        info->lanes_per_cta = d.dt;
        info->rows_per_window = d.w;
        info->subchunks = d.s;
        std::snprintf(info->name, sizeof info->name, "%s", c.var->name);
    } else if (c.path == kPathChunk) {
        info->lanes_per_cta = 128 * c.vec;
        info->rows_per_window = c.chunk;
        std::snprintf(info->name, sizeof info->name, "chunk%d_v%d%s", c.chunk, c.vec, c.vidx == 1 ? "_grouped" : "");
    } else {
        info->lanes_per_cta = 128;
        std::snprintf(info->name, sizeof info->name, "plain");
    }
}

// -------------------------------------------------------------------------
// Tensor maps: a [B][T][D] tensor viewed as 3-D {D, T, B}; box {DT, W, 1}.
// -------------------------------------------------------------------------
int encode_map(CUtensorMap *m, const void *ptr, int dtype, int64_t B, int64_t T, int64_t D, int dt, int w) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esize(dtype),
                                   static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(D) * esize(dtype)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(dt), static_cast<cuuint32_t>(w), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dtype == LRSCAN_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(LRSCAN_EINVAL, "cuTensorMapEncodeTiled failed (%d) for ptr %p dims {%lld,%lld,%lld} box {%d,%d}",
                    static_cast<int>(r), ptr, static_cast<long long>(D), static_cast<long long>(T),
                    static_cast<long long>(B), dt, w);
    return LRSCAN_OK;
}

int check_shape(int64_t B, int64_t T, int64_t D, int dtype) {
    if (dtype != LRSCAN_F32 && dtype != LRSCAN_BF16) return fail(LRSCAN_EDTYPE, "dtype %d", dtype);
    if (B < 0 || T < 0 || D < 0)
        return fail(LRSCAN_EINVAL, "negative size B=%lld T=%lld D=%lld", static_cast<long long>(B),
                    static_cast<long long>(T), static_cast<long long>(D));
    if (T > 0x7fffffffLL || D > 0x7fffffffLL) return fail(LRSCAN_EINVAL, "T or D above 2^31-1");
    int64_t e = 0, bytes = 0;
    if (__builtin_mul_overflow(B, T, &e) || __builtin_mul_overflow(e, D, &e) ||
        __builtin_mul_overflow(e, static_cast<int64_t>(esize(dtype)), &bytes))
        return fail(LRSCAN_EINVAL, "B*T*D*elem overflows int64");
    return LRSCAN_OK;
}

bool aligned16(std::initializer_list<const void *> ps, int64_t D, int dtype) {
    if ((D * esize(dtype)) % 16 != 0) return false;
    for (const void *p : ps)
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return false;
    return true;
}

int workspace_for(DeviceCtx *ctx, cudaStream_t st, size_t need, const lrscan_opts *opts, void **ws) {
    if (opts && opts->workspace) {
        if (opts->workspace_bytes < need || reinterpret_cast<uintptr_t>(opts->workspace) % 256 != 0)
            return fail(LRSCAN_ENOMEM, "caller workspace of %zu bytes (need %zu, 256-byte aligned)",
                        opts->workspace_bytes, need);
        *ws = opts->workspace;
        return LRSCAN_OK;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    auto &slot = ctx->workspace[st];
    if (slot.second < need) {
        // growing synchronizes the stream and allocates: neither may happen
        // while the stream is being captured into a graph (nothing has been
        // enqueued yet, so the capture stays valid)
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
            cudaGetLastError();
            return fail(LRSCAN_ECUDA, "cudaStreamIsCapturing failed");
        }
        if (cs != cudaStreamCaptureStatusNone)
            return fail(LRSCAN_ENOMEM,
                        "the library-owned workspace must grow to %zu bytes, which cannot happen during stream "
                        "capture: make one call of this size before capturing, or pass opts->workspace",
                        need);
        if (slot.first) {
            cudaStreamSynchronize(st);  // the old buffer may still be in use by this stream
            cudaFree(slot.first);
            slot.first = nullptr;
            slot.second = 0;
        }
        void *p = nullptr;
        if (cudaMalloc(&p, need) != cudaSuccess) {
            cudaGetLastError();
            return fail(LRSCAN_ENOMEM, "cudaMalloc of %zu workspace bytes failed", need);
        }
        slot.first = p;
        slot.second = need;
    }
    *ws = slot.first;
    return LRSCAN_OK;
}

cudaStream_t pick_stream(void *stream) { return stream ? static_cast<cudaStream_t>(stream) : t_stream; }

void set_chunk_scratch(ChunkLaunch *L, void *ws, const Choice &ch) {
    const ChunkScratch sc = chunk_scratch(L->B, L->T, L->D, ch.chunk, ch.vidx == 1);
    char *base = static_cast<char *>(ws);
    L->P = reinterpret_cast<float *>(base);
    L->Q = reinterpret_cast<float *>(base + sc.pq);
    L->PG = sc.group ? reinterpret_cast<float *>(base + 2 * sc.pq) : nullptr;
    L->QG = sc.group ? reinterpret_cast<float *>(base + 2 * sc.pq + sc.group) : nullptr;
}

// Complex chunked scratch views: P re, P im, Q re, Q im, then (grouped
// prefix) the four group-map arrays, each rounded up to 256 bytes.
void set_cchunk_scratch(CChunkLaunch *L, void *ws, int64_t B, int64_t T, int64_t D, const Choice &ch) {
    const ChunkScratch sc = chunk_scratch(B, T, D, ch.chunk, ch.vidx == 1);
    char *base = static_cast<char *>(ws);
    for (int i = 0; i < 4; ++i) {
        L->maps[i] = reinterpret_cast<float *>(base + i * sc.pq);
        L->gmaps[i] = sc.group ? reinterpret_cast<float *>(base + 4 * sc.pq + i * sc.group) : nullptr;
    }
}

// The state members a direction uses, checked: fp32 / int32 device pointers
// must be 4-byte aligned.  *any is set when the call carries state.
int check_state(const lrscan_state *s, bool bwd, bool *any) {
    *any = false;
    if (!s) return LRSCAN_OK;
    const void *ps[4] = {s->h0, s->segment_pos, bwd ? s->grad_last : nullptr, bwd ? s->grad_h0 : nullptr};
    for (const void *p : ps) {
        if (!p) continue;
        if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return fail(LRSCAN_EINVAL, "state pointer %p is not 4-byte aligned", p);
        *any = true;
    }
    return LRSCAN_OK;
}

// Kernel view of the state for batch rows [b0, ...).
StateArgs state_slice(const lrscan_state *s, bool bwd, const void *a, int64_t b0, int64_t T, int64_t D, size_t es) {
    StateArgs x{};
    if (!s) return x;
    const size_t sd = static_cast<size_t>(b0) * D;
    x.h0 = s->h0 ? s->h0 + sd : nullptr;
    x.seg = s->segment_pos ? s->segment_pos + static_cast<size_t>(b0) * T : nullptr;
    if (bwd) {
        x.grad_last = s->grad_last ? s->grad_last + sd : nullptr;
        x.grad_h0 = s->grad_h0 ? s->grad_h0 + sd : nullptr;
        x.a = static_cast<const char *>(a) + static_cast<size_t>(b0) * T * D * es;
    }
    return x;
}

// T == 0: the final state is h0 (forward) and the initial-state gradient is
// grad_last (backward); zeros without them.
int copy_or_zero(float *dst, const float *src, int64_t B, int64_t D, cudaStream_t st) {
    if (!dst) return LRSCAN_OK;
    const size_t bytes = static_cast<size_t>(B) * D * 4;
    const cudaError_t e = src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st)
                              : cudaMemsetAsync(dst, 0, bytes, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(LRSCAN_ECUDA, "T == 0 state copy: %s", cudaGetErrorString(e));
    }
    return LRSCAN_OK;
}

// The persistent chunk-streaming path: tensor maps of the inputs (forward a,
// b; backward a, out, grad_out) and outputs (forward out; backward grad_a,
// grad_b), the publication workspace reset (ticket zeroed, maps and states
// all-ones), one launch.
int run_stream(const Choice &ch, std::initializer_list<const void *> ins, std::initializer_list<void *> outs,
               float *last, float *last_i, int64_t B, int64_t T, int64_t D, int dtype, cudaStream_t st, int dev,
               DeviceCtx *ctx, const lrscan_opts *opts, bool bwd, bool cplx, const StateArgs *sx = nullptr,
               const CStateArgs *csx = nullptr) {
    const WinDirCfg &v = dir_of(*ch.var, bwd ? 1 : 0);
    const int64_t ndt = (D + v.dt - 1) / v.dt;
    const int64_t ng = B * ndt;
    const int64_t nc = (T + ch.chunk - 1) / ch.chunk;
    const StreamScratch sc = stream_scratch(ng, nc, v.dt, cplx ? 2 : 1);
    void *ws = nullptr;
    int rc = workspace_for(ctx, st, ch.workspace, opts, &ws);
    if (rc) return rc;
    CUtensorMap maps[10];  // inputs in kernel order from 0, outputs from 6
    WinLaunch L{};
    int k = 0;
    for (const void *p : ins) {
        if (encode_map(&maps[k], p, dtype, B, T, D, v.dt, v.w)) return LRSCAN_EINVAL;
        L.maps[k] = &maps[k];
        ++k;
    }
    k = 6;
    for (void *p : outs) {
        if (encode_map(&maps[k], p, dtype, B, T, D, v.dt, v.w)) return LRSCAN_EINVAL;
        L.maps[k] = &maps[k];
        ++k;
    }
    L.last = last;
    L.last_i = last_i;
    L.B = B; L.T = T; L.D = D;
    L.status = ctx->status;
    L.timeout_ns = g_timeout_ns.load();
    L.stream = st;
    L.device = dev;
    char *base = static_cast<char *>(ws);
    L.sa.ticket = reinterpret_cast<unsigned int *>(base);
    L.sa.agg = reinterpret_cast<float2 *>(base + sc.head());
    L.sa.incl = reinterpret_cast<float *>(base + sc.head() + sc.agg);
    L.sa.nc = static_cast<int>(nc);
    L.sa.ndt = static_cast<int>(ndt);
    L.sa.ng = static_cast<int>(ng);
    L.grid = static_cast<int>(ch.ctas);
    if (cudaMemsetAsync(ws, 0, sc.head(), st) != cudaSuccess ||
        cudaMemsetAsync(base + sc.head(), 0xff, sc.agg + sc.incl, st) != cudaSuccess) {
        cudaGetLastError();
        return fail(LRSCAN_ECUDA, "clearing the streaming workspace failed");
    }
    if (sx) L.sx = *sx;
    if (csx) L.csx = *csx;
    if ((sx || csx ? v.launch_state : v.launch)(L, v))
        return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
    return LRSCAN_OK;
}

int run_fwd(const void *a, const void *b, void *out, float *last, int64_t B, int64_t T, int64_t D, int dtype,
            void *stream, const lrscan_opts *opts, const lrscan_state *state = nullptr) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    bool ext = false;
    if ((rc = check_state(state, false, &ext))) return rc;
    if (B == 0 || D == 0) return LRSCAN_OK;
    cudaStream_t st = pick_stream(stream);
    if (T == 0) return copy_or_zero(last, ext ? state->h0 : nullptr, B, D, st);
    if (!a || !b || !out) return fail(LRSCAN_EINVAL, "NULL a, b or out");
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool al = aligned16({a, b, out}, D, dtype);
    Choice ch;
    if ((rc = plan_call(B, T, D, dtype, 0, al, opts, geometry_of(ctx), &ch, ext))) return rc;
    const size_t es = esize(dtype);
    if (ch.path == kPathSeq || ch.path == kPathWindow) {
        const WinDirCfg &v = ch.var->fwd;
        for (int64_t b0 = 0; b0 < B; b0 += 65535) {
            const int64_t nb = std::min<int64_t>(65535, B - b0);
            const size_t off = static_cast<size_t>(b0) * T * D * es;
            CUtensorMap ma, mb, mo;  // mo: lane-scan tiles write out through bulk tensor stores
            if (encode_map(&ma, static_cast<const char *>(a) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mb, static_cast<const char *>(b) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mo, static_cast<char *>(out) + off, dtype, nb, T, D, v.dt, v.w))
                return LRSCAN_EINVAL;
            WinLaunch L{};
            L.maps[0] = &ma;
            L.maps[1] = &mb;
            L.maps[2] = &mo;
            L.out0 = static_cast<char *>(out) + off;
            L.last = last ? last + b0 * D : nullptr;
            L.B = nb; L.T = T; L.D = D;
            L.status = ctx->status;
            L.timeout_ns = g_timeout_ns.load();
            L.stream = st;
            L.device = dev;
            L.sx = state_slice(ext ? state : nullptr, false, a, b0, T, D, es);
            if ((ext ? v.launch_state : v.launch)(L, v))
                return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
        }
        return LRSCAN_OK;
    }
    if (ch.path == kPathStream) {
        const StateArgs sx = state_slice(ext ? state : nullptr, false, a, 0, T, D, es);
        return run_stream(ch, {a, b}, {out}, last, nullptr, B, T, D, dtype, st, dev, ctx, opts, false, false,
                          ext ? &sx : nullptr);
    }
    ChunkLaunch L{};
    L.in0 = a; L.in1 = b; L.out0 = out; L.last = last;
    L.B = B; L.T = T; L.D = D;
    L.chunk = ch.chunk; L.vec = ch.vec; L.stream = st;
    L.sx = state_slice(ext ? state : nullptr, false, a, 0, T, D, es);
    if (ch.path == kPathPlain) return plain_fwd_launch(L, dtype) ? LRSCAN_ECUDA : LRSCAN_OK;
    void *ws = nullptr;
    if ((rc = workspace_for(ctx, st, ch.workspace, opts, &ws))) return rc;
    set_chunk_scratch(&L, ws, ch);
    rc = chunk_fwd(L, dtype);
    return rc == 0 ? LRSCAN_OK : (rc == -2 ? LRSCAN_EINVAL : LRSCAN_ECUDA);
}

int run_bwd(const void *a, const void *out, const void *grad_out, void *grad_a, void *grad_b, int64_t B, int64_t T,
            int64_t D, int dtype, void *stream, const lrscan_opts *opts, const lrscan_state *state = nullptr) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    bool ext = false;
    if ((rc = check_state(state, true, &ext))) return rc;
    if (B == 0 || D == 0) return LRSCAN_OK;
    cudaStream_t st = pick_stream(stream);
    if (T == 0) return ext ? copy_or_zero(state->grad_h0, state->grad_last, B, D, st) : LRSCAN_OK;
    if (!a || !out || !grad_out || !grad_a || !grad_b) return fail(LRSCAN_EINVAL, "NULL a, out, grad_out, grad_a or grad_b");
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool al = aligned16({a, out, grad_out, grad_a, grad_b}, D, dtype);
    Choice ch;
    if ((rc = plan_call(B, T, D, dtype, 1, al, opts, geometry_of(ctx), &ch, ext))) return rc;
    const size_t es = esize(dtype);
    if (ch.path == kPathSeq || ch.path == kPathWindow) {
        const WinDirCfg &v = ch.var->bwd;
        for (int64_t b0 = 0; b0 < B; b0 += 65535) {
            const int64_t nb = std::min<int64_t>(65535, B - b0);
            const size_t off = static_cast<size_t>(b0) * T * D * es;
            CUtensorMap ma, mo, mg, mga, mgb;  // mga, mgb: lane-scan tiles write through bulk tensor stores
            if (encode_map(&ma, static_cast<const char *>(a) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mo, static_cast<const char *>(out) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mg, static_cast<const char *>(grad_out) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mga, static_cast<char *>(grad_a) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mgb, static_cast<char *>(grad_b) + off, dtype, nb, T, D, v.dt, v.w))
                return LRSCAN_EINVAL;
            WinLaunch L{};
            L.maps[0] = &ma;
            L.maps[1] = &mo;
            L.maps[2] = &mg;
            L.maps[3] = &mga;
            L.maps[4] = &mgb;
            L.out0 = static_cast<char *>(grad_a) + off;
            L.out1 = static_cast<char *>(grad_b) + off;
            L.B = nb; L.T = T; L.D = D;
            L.status = ctx->status;
            L.timeout_ns = g_timeout_ns.load();
            L.stream = st;
            L.device = dev;
            L.sx = state_slice(ext ? state : nullptr, true, a, b0, T, D, es);
            if ((ext ? v.launch_state : v.launch)(L, v))
                return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
        }
        return LRSCAN_OK;
    }
    if (ch.path == kPathStream) {
        const StateArgs sx = state_slice(ext ? state : nullptr, true, a, 0, T, D, es);
        return run_stream(ch, {a, out, grad_out}, {grad_a, grad_b}, nullptr, nullptr, B, T, D, dtype, st, dev, ctx, opts,
                          true, false, ext ? &sx : nullptr);
    }
    ChunkLaunch L{};
    L.in0 = a; L.in1 = out; L.in2 = grad_out; L.out0 = grad_a; L.out1 = grad_b;
    L.B = B; L.T = T; L.D = D;
    L.chunk = ch.chunk; L.vec = ch.vec; L.stream = st;
    L.sx = state_slice(ext ? state : nullptr, true, a, 0, T, D, es);
    if (ch.path == kPathPlain) return plain_bwd_launch(L, dtype) ? LRSCAN_ECUDA : LRSCAN_OK;
    void *ws = nullptr;
    if ((rc = workspace_for(ctx, st, ch.workspace, opts, &ws))) return rc;
    set_chunk_scratch(&L, ws, ch);
    rc = chunk_bwd(L, dtype);
    return rc == 0 ? LRSCAN_OK : (rc == -2 ? LRSCAN_EINVAL : LRSCAN_ECUDA);
}

// ---------------------------------------------------------------- complex --
// Index of the named variant when it fits on an SM and gives at least 0.9
// CTAs per SM, else -1.
int find_variant(const WinVariant *tab, int n, const char *name, int dir, int64_t B, int64_t D, const Geometry &g) {
    for (int i = 0; i < n; ++i) {
        if (std::strcmp(tab[i].name, name) != 0) continue;
        const Occ o = occupancy(tab[i], dir, B, D, g);
        if (o.resident > 0 && static_cast<double>(o.ctas) >= 0.9 * g.sm_count) return i;
    }
    return -1;
}

// Index of the named variant when all its CTAs are resident at once (and
// they are at least 0.9 per SM), else -1.
int find_one_wave(const WinVariant *tab, int n, const char *name, int dir, int64_t B, int64_t D, const Geometry &g) {
    for (int i = 0; i < n; ++i) {
        if (std::strcmp(tab[i].name, name) != 0) continue;
        const Occ o = occupancy(tab[i], dir, B, D, g);
        if (o.one_wave && static_cast<double>(o.ctas) >= 0.9 * g.sm_count) return i;
    }
    return -1;
}

// Complex scan: the tiled sequential kernels when every plane's rows are
// 16-byte aligned, else the plain kernels.  The tile variant is chosen by the
// window-variant rule (a single wave first, then the fullest last wave, then
// bytes in flight), else the variant with the most CTAs.
// Complex chunked-path scratch: P and Q, re and im ([B, Nc, D] fp32 each),
// then the grouped prefix's four group-map arrays: twice the real path's.
size_t cchunk_workspace(int64_t B, int64_t T, int64_t D, int C, bool grouped) {
    return 2 * chunk_workspace(B, T, D, C, grouped);
}

// ext: the call carries state or resets (chunked path only).
int plan_complex(int64_t B, int64_t T, int64_t D, int dtype, int dir, bool aligned16, const lrscan_opts *opts,
                 const Geometry &g, Choice *ch, bool ext = false) {
    const int want = opts ? opts->path : 0;
    if (ext && want == kPathPlain)
        return fail(LRSCAN_EINVAL, "the plain complex kernels carry no state (path %d)", want);
    const int force_v = opts ? opts->tile_variant : 0;
    if (want != kPathAuto && want != kPathSeq && want != kPathWindow && want != kPathPlain && want != kPathChunk &&
        want != kPathStream)
        return fail(LRSCAN_EINVAL, "unknown complex scan path %d", want);
    if ((want == kPathSeq || want == kPathWindow || want == kPathStream) && !aligned16)
        return fail(LRSCAN_EINVAL, "tiled paths need 16-byte aligned pointers and rows (D*elem %% 16 == 0)");
    // default chunk: 64 steps fp32, 128 bf16 (the same bytes per chunk row;
    // measured on few-lane complex scans: bf16 10-13 % faster than at 64)
    const int chunk = opts && opts->chunk_len ? opts->chunk_len : (dtype == LRSCAN_BF16 ? 128 : 64);
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128 && chunk != 256 && chunk != 512)
        return fail(LRSCAN_EINVAL, "chunk_len %d is not 16, 32, 64, 128, 256 or 512", chunk);
    int path;
    if (want == kPathAuto) {
        // too few lanes for lane tiles of 32 to give the SMs work (fewer than
        // 0.45 tiles per SM; the plain kernels' bound without alignment) and
        // a long sequence: parallelize over time chunks
        // With carried state the tiled kernels (EXT instantiations) run as
        // they would without it; unaligned rows take the chunked kernels,
        // which carry state at any alignment.
        // In one pass (chunk streaming) from 32 chunks of 512 steps per lane
        // group, with or without carried state, unless a chunk length is asked for.
        const long long few = aligned16 ? static_cast<long long>(0.45 * g.sm_count * 32) : 32LL * g.sm_count * 32;
        if (B * D < few && T >= 16LL * chunk)
            path = (aligned16 && T >= 32LL * 512 && !(opts && opts->chunk_len)) ? kPathStream : kPathChunk;
        else path = aligned16 ? kPathSeq : (ext ? kPathChunk : kPathPlain);
    } else {
        // seq and window both name the tiled variant table (sequential and windowed tiles)
        path = (want == kPathPlain || want == kPathChunk || want == kPathStream) ? want : kPathSeq;
    }
    ch->path = path;
    ch->dir = dir;
    ch->kernels = 1;
    ch->vec = 1;
    if (path == kPathStream) {
        int n = 0;
        const WinVariant *tab = cstream_variants(dtype, &n);
        if (force_v > n) return fail(LRSCAN_EINVAL, "tile_variant %d > %d variants", force_v, n);
        return plan_stream_variant(tab, force_v > 0 ? force_v - 1 : 0, dir, B, T, D, 2, g, ch);
    }
    if (path == kPathChunk) {
        // variant 1: flat per-lane prefix; variant 2: grouped prefix
        if (force_v > 2) return fail(LRSCAN_EINVAL, "the chunked path has two variants (1 flat, 2 grouped prefix)");
        const bool grouped = force_v ? force_v == 2 : use_grouped_prefix(B, T, D, chunk, g);
        const int64_t nc = (T + chunk - 1) / chunk;
        // four lanes per thread when the rows are 16-byte aligned (D is then a
        // multiple of 4): 4-11 % faster backward than two on few-lane scans
        ch->vec = aligned16 && D % 4 == 0 ? 4 : 1;
        const int64_t row_threads = (D + ch->vec - 1) / ch->vec;
        int64_t lt = 1;
        while (lt < row_threads && lt < 128) lt <<= 1;
        const int64_t cpb = row_threads <= 64 ? 128 / lt : 1;
        const int64_t nlb = row_threads <= 64 ? 1 : (row_threads + 127) / 128;
        ch->chunk = chunk;
        ch->vidx = grouped ? 1 : 0;
        ch->ctas = B * ((nc + cpb - 1) / cpb) * nlb;
        ch->threads = 128;
        ch->kernels = grouped ? 5 : 3;
        ch->workspace = cchunk_workspace(B, T, D, chunk, grouped);
        return LRSCAN_OK;
    }
    if (path == kPathPlain) {
        if (force_v > 1) return fail(LRSCAN_EINVAL, "the plain path has one variant");
        ch->ctas = B * ((D + 127) / 128);
        ch->threads = 128;
        return LRSCAN_OK;
    }
    int n = 0;
    const WinVariant *tab = cwin_variants(dtype, &n);
    int vi = -1;
    if (force_v > 0) {
        if (force_v > n) return fail(LRSCAN_EINVAL, "tile_variant %d > %d variants", force_v, n);
        vi = force_v - 1;
    } else if (dtype == LRSCAN_BF16 && dir == 0 &&
               ((vi = find_one_wave(tab, n, "cwin_bf16_d32_l4_s8_m5", dir, B, D, g)) >= 0 ||
                (vi = find_variant(tab, n, "cwin_bf16_d32_s16_v2", dir, B, D, g)) >= 0)) {
        // measured best complex bf16 forward: the windowed tiles (time split
        // inside the CTA); 4-row sub-chunks with five CTAs per SM when all the
        // CTAs fit one wave (84.5 us on the complex workload against 93.1 us)
    } else if (dtype == LRSCAN_BF16 && dir == 1 &&
               (vi = find_one_wave(tab, n, "cwin_bf16_d32_l4_s8_m5", dir, B, D, g)) >= 0) {
        // measured best complex bf16 backward: the windowed tile with 4-row
        // sub-chunks, five CTAs per SM, when all its CTAs fit one wave (152.3 us
        // on the complex workload against 157.4 us for the sequential tile)
    } else if (dtype == LRSCAN_BF16 && (vi = find_one_wave(tab, n, "cseq_bf16_d64_v1_n4", dir, B, D, g)) >= 0) {
        // else the sequential tile whenever all its CTAs fit one wave
    } else if (!pick_from_table(tab, n, dir, B, D, g, &vi)) {
        long long most = -1;
        for (int i = 0; i < n; ++i) {
            const Occ o = occupancy(tab[i], dir, B, D, g);
            if (o.resident > 0 && o.ctas > most) { most = o.ctas; vi = i; }
        }
    }
    if (vi < 0) return fail(LRSCAN_EINVAL, "no complex tile variant fits this device");
    const Occ o = occupancy(tab[vi], dir, B, D, g);
    if (o.resident == 0) return fail(LRSCAN_EINVAL, "tile variant %s does not fit on an SM", tab[vi].name);
    ch->vidx = vi;
    ch->var = &tab[vi];
    ch->path = dir_of(tab[vi], dir).s > 1 ? kPathWindow : kPathSeq;
    ch->ctas = o.ctas;
    ch->threads = dir_of(tab[vi], dir).threads;
    ch->smem = dir_of(tab[vi], dir).smem;
    ch->stages = dir_of(tab[vi], dir).nstage;
    return LRSCAN_OK;
}

// Complex carried state, checked (fp32 / int32 pointers 4-byte aligned);
// *any is set when the call carries state.
int check_cstate(const lrscan_cstate *s, bool bwd, CStateArgs *sx, bool *any) {
    *sx = CStateArgs{};
    *any = false;
    if (!s) return LRSCAN_OK;
    sx->h0_r = s->h0_r;
    sx->h0_i = s->h0_i;
    sx->seg = s->segment_pos;
    if (bwd) {
        sx->gl_r = s->grad_last_r;
        sx->gl_i = s->grad_last_i;
        sx->gh0_r = s->grad_h0_r;
        sx->gh0_i = s->grad_h0_i;
    }
    const void *ps[7] = {sx->h0_r, sx->h0_i, sx->seg, sx->gl_r, sx->gl_i, sx->gh0_r, sx->gh0_i};
    for (const void *p : ps) {
        if (!p) continue;
        if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return fail(LRSCAN_EINVAL, "state pointer %p is not 4-byte aligned", p);
        *any = true;
    }
    return LRSCAN_OK;
}

// The complex state of batch rows b0.. of a tiled launch (planes ar / ai:
// the backward's decays, for grad_h0).
CStateArgs cstate_slice(const CStateArgs &s, const void *ar, const void *ai, int64_t b0, int64_t T, int64_t D,
                        size_t es) {
    CStateArgs x = s;
    const size_t sd = static_cast<size_t>(b0) * D;
    auto f = [sd](const float *p) { return p ? p + sd : nullptr; };
    x.h0_r = f(s.h0_r);
    x.h0_i = f(s.h0_i);
    x.gl_r = f(s.gl_r);
    x.gl_i = f(s.gl_i);
    x.gh0_r = s.gh0_r ? s.gh0_r + sd : nullptr;
    x.gh0_i = s.gh0_i ? s.gh0_i + sd : nullptr;
    x.seg = s.seg ? s.seg + static_cast<size_t>(b0) * T : nullptr;
    const size_t po = static_cast<size_t>(b0) * T * D * es;
    x.ar = ar ? static_cast<const char *>(ar) + po : nullptr;
    x.ai = ai ? static_cast<const char *>(ai) + po : nullptr;
    return x;
}

int run_cfwd(const void *const in[4], void *out_r, void *out_i, float *last_r, float *last_i, int64_t B, int64_t T,
             int64_t D, int dtype, void *stream, const lrscan_opts *opts, const lrscan_cstate *state = nullptr) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    CStateArgs sx;
    bool ext = false;
    if ((rc = check_cstate(state, false, &sx, &ext))) return rc;
    if (B == 0 || D == 0) return LRSCAN_OK;
    cudaStream_t st = pick_stream(stream);
    if (T == 0) {
        if ((rc = copy_or_zero(last_r, sx.h0_r, B, D, st)) || (rc = copy_or_zero(last_i, sx.h0_i, B, D, st)))
            return rc;
        return LRSCAN_OK;
    }
    if (!in[0] || !in[1] || !in[2] || !in[3] || !out_r || !out_i)
        return fail(LRSCAN_EINVAL, "NULL ar, ai, br, bi, out_r or out_i");
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool al = aligned16({in[0], in[1], in[2], in[3], out_r, out_i}, D, dtype);
    Choice ch;
    if ((rc = plan_complex(B, T, D, dtype, 0, al, opts, geometry_of(ctx), &ch, ext))) return rc;
    const size_t es = esize(dtype);
    if (ch.path == kPathStream) {
        const CStateArgs xs = cstate_slice(sx, nullptr, nullptr, 0, T, D, es);
        return run_stream(ch, {in[0], in[1], in[2], in[3]}, {out_r, out_i}, last_r, last_i, B, T, D, dtype, st, dev,
                          ctx, opts, false, true, nullptr, ext ? &xs : nullptr);
    }
    if (ch.path == kPathChunk) {
        void *ws = nullptr;
        if ((rc = workspace_for(ctx, st, ch.workspace, opts, &ws))) return rc;
        CChunkLaunch L{};
        for (int i = 0; i < 4; ++i) L.in[i] = in[i];
        L.out[0] = out_r;
        L.out[1] = out_i;
        L.last_r = last_r;
        L.last_i = last_i;
        L.sx = sx;
        set_cchunk_scratch(&L, ws, B, T, D, ch);
        L.B = B; L.T = T; L.D = D; L.chunk = ch.chunk; L.vec = ch.vec; L.stream = st;
        return cchunk_fwd_launch(L, dtype)
                   ? fail(LRSCAN_ECUDA, "complex chunked launch: %s", cudaGetErrorString(cudaGetLastError()))
                   : LRSCAN_OK;
    }
    if (ch.path == kPathPlain) {
        ChunkLaunch L{};
        L.in0 = in[0]; L.in1 = in[2]; L.out0 = out_r; L.last = last_r;
        L.B = B; L.T = T; L.D = D; L.stream = st;
        return cplain_fwd_launch(L, in[1], in[3], out_i, last_i, dtype)
                   ? fail(LRSCAN_ECUDA, "complex plain launch: %s", cudaGetErrorString(cudaGetLastError()))
                   : LRSCAN_OK;
    }
    const WinDirCfg &v = ch.var->fwd;
    for (int64_t b0 = 0; b0 < B; b0 += 65535) {
        const int64_t nb = std::min<int64_t>(65535, B - b0);
        const size_t off = static_cast<size_t>(b0) * T * D * es;
        CUtensorMap m[6];  // ar, ai, br, bi; out_r, out_i (the windowed tiles write through bulk tensor stores)
        const void *planes[6] = {in[0], in[1], in[2], in[3], out_r, out_i};
        for (int i = 0; i < 6; ++i)
            if (encode_map(&m[i], static_cast<const char *>(planes[i]) + off, dtype, nb, T, D, v.dt, v.w))
                return LRSCAN_EINVAL;
        WinLaunch L{};
        for (int i = 0; i < 6; ++i) L.maps[i] = &m[i];
        L.out0 = static_cast<char *>(out_r) + off;
        L.out1 = static_cast<char *>(out_i) + off;
        L.last = last_r ? last_r + b0 * D : nullptr;
        L.last_i = last_i ? last_i + b0 * D : nullptr;
        L.B = nb; L.T = T; L.D = D;
        L.status = ctx->status;
        L.timeout_ns = g_timeout_ns.load();
        L.stream = st;
        L.device = dev;
        if (ext) L.csx = cstate_slice(sx, nullptr, nullptr, b0, T, D, es);
        if ((ext ? v.launch_state : v.launch)(L, v))
            return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
    }
    return LRSCAN_OK;
}

int run_cbwd(const void *const in[6], void *const outp[4], int64_t B, int64_t T, int64_t D, int dtype, void *stream,
             const lrscan_opts *opts, const lrscan_cstate *state = nullptr) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    CStateArgs sx;
    bool ext = false;
    if ((rc = check_cstate(state, true, &sx, &ext))) return rc;
    if (B == 0 || D == 0) return LRSCAN_OK;
    if (T == 0) {
        cudaStream_t st0 = pick_stream(stream);
        if ((rc = copy_or_zero(sx.gh0_r, sx.gl_r, B, D, st0)) || (rc = copy_or_zero(sx.gh0_i, sx.gl_i, B, D, st0)))
            return rc;
        return LRSCAN_OK;
    }
    for (int i = 0; i < 6; ++i)
        if (!in[i]) return fail(LRSCAN_EINVAL, "NULL complex backward input %d", i);
    for (int i = 0; i < 4; ++i)
        if (!outp[i]) return fail(LRSCAN_EINVAL, "NULL complex gradient output %d", i);
    cudaStream_t st = pick_stream(stream);
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool al = aligned16({in[0], in[1], in[2], in[3], in[4], in[5], outp[0], outp[1], outp[2], outp[3]}, D, dtype);
    Choice ch;
    if ((rc = plan_complex(B, T, D, dtype, 1, al, opts, geometry_of(ctx), &ch, ext))) return rc;
    if (ch.path == kPathStream) {
        const CStateArgs xs = cstate_slice(sx, in[0], in[1], 0, T, D, esize(dtype));
        return run_stream(ch, {in[0], in[1], in[2], in[3], in[4], in[5]}, {outp[0], outp[1], outp[2], outp[3]},
                          nullptr, nullptr, B, T, D, dtype, st, dev, ctx, opts, true, true, nullptr,
                          ext ? &xs : nullptr);
    }
    if (ch.path == kPathChunk) {
        void *ws = nullptr;
        if ((rc = workspace_for(ctx, st, ch.workspace, opts, &ws))) return rc;
        CChunkLaunch L{};
        for (int i = 0; i < 6; ++i) L.in[i] = in[i];
        for (int i = 0; i < 4; ++i) L.out[i] = outp[i];
        L.sx = sx;
        set_cchunk_scratch(&L, ws, B, T, D, ch);
        L.B = B; L.T = T; L.D = D; L.chunk = ch.chunk; L.vec = ch.vec; L.stream = st;
        return cchunk_bwd_launch(L, dtype)
                   ? fail(LRSCAN_ECUDA, "complex chunked launch: %s", cudaGetErrorString(cudaGetLastError()))
                   : LRSCAN_OK;
    }
    if (ch.path == kPathPlain)
        return cplain_bwd_launch(in, outp, B, T, D, dtype, st)
                   ? fail(LRSCAN_ECUDA, "complex plain launch: %s", cudaGetErrorString(cudaGetLastError()))
                   : LRSCAN_OK;
    const size_t es = esize(dtype);
    const WinDirCfg &v = ch.var->bwd;
    for (int64_t b0 = 0; b0 < B; b0 += 65535) {
        const int64_t nb = std::min<int64_t>(65535, B - b0);
        const size_t off = static_cast<size_t>(b0) * T * D * es;
        CUtensorMap m[10];  // 6 inputs, then the 4 gradients (windowed tiles store them with bulk copies)
        for (int i = 0; i < 10; ++i) {
            const char *base = i < 6 ? static_cast<const char *>(in[i]) : static_cast<const char *>(outp[i - 6]);
            if (encode_map(&m[i], base + off, dtype, nb, T, D, v.dt, v.w)) return LRSCAN_EINVAL;
        }
        WinLaunch L{};
        for (int i = 0; i < 10; ++i) L.maps[i] = &m[i];
        L.out0 = static_cast<char *>(outp[0]) + off;
        L.out1 = static_cast<char *>(outp[1]) + off;
        L.out2 = static_cast<char *>(outp[2]) + off;
        L.out3 = static_cast<char *>(outp[3]) + off;
        L.B = nb; L.T = T; L.D = D;
        L.status = ctx->status;
        L.timeout_ns = g_timeout_ns.load();
        L.stream = st;
        L.device = dev;
        if (ext) L.csx = cstate_slice(sx, in[0], in[1], b0, T, D, es);
        if ((ext ? v.launch_state : v.launch)(L, v))
            return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
    }
    return LRSCAN_OK;
}

// ------------------------------------------------------- generated decay --
// Partial-sum columns per row of the backward: one per CTA of a windowed
// tile (at least 16 lanes each) or per warp of a sequential tile (32 lanes),
// plus the ragged last CTA's extra warps.
int64_t gated_ncol_bound(int64_t D) { return (D + 15) / 16 + 4; }

// Backward scratch: grad_eta partials [B*T][ncol], then grad_nu_log partials
// [B * kGatedMaxS][D] (one row per batch row and sub-chunk).
size_t gated_workspace(int64_t B, int64_t T, int64_t D) {
    auto pad = [](size_t x) { return (x + 255) / 256 * 256; };
    return pad(static_cast<size_t>(B) * T * gated_ncol_bound(D) * 4) +
           pad(static_cast<size_t>(B) * kGatedMaxS * D * 4);
}

// Tiled sequential kernels for 16-byte aligned rows, else plain kernels.
int plan_gated(int64_t B, int64_t D, int dtype, int dir, bool aligned, const lrscan_opts *opts, const Geometry &g,
               Choice *ch) {
    const int want = opts ? opts->path : 0;
    const int force_v = opts ? opts->tile_variant : 0;
    if (want != kPathAuto && want != kPathSeq && want != kPathPlain)
        return fail(LRSCAN_EINVAL, "the generated-decay scan has the seq and plain paths only (path %d)", want);
    if (want == kPathSeq && !aligned)
        return fail(LRSCAN_EINVAL, "path seq needs 16-byte aligned pointers and rows (D*elem %% 16 == 0)");
    const int path = want == kPathAuto ? (aligned ? kPathSeq : kPathPlain) : want;
    ch->path = path;
    ch->dir = dir;
    ch->kernels = dir == 0 ? 1 : 2;
    ch->vec = 1;
    if (path == kPathPlain) {
        if (force_v > 1) return fail(LRSCAN_EINVAL, "the plain path has one variant");
        ch->ctas = B * ((D + 127) / 128);
        ch->threads = 128;
        return LRSCAN_OK;
    }
    int n = 0;
    const WinVariant *tab = gwin_variants(dtype, &n);
    int vi = -1;
    if (force_v > 0) {
        if (force_v > n) return fail(LRSCAN_EINVAL, "tile_variant %d > %d variants", force_v, n);
        vi = force_v - 1;
    } else if (B * ((D + 15) / 16) >= 8LL * g.sm_count &&
               (vi = find_variant(tab, n, dtype == LRSCAN_BF16 ? "gwarp_bf16_l16_r15" : "gwarp_f32_l16_r15", dir, B,
                                  D, g)) >= 0) {
        // from eight 16-lane slices per SM: one warp per slice (B=8 T=2048
        // D=2560: bf16 forward 33.9 us against 38.1 us for the windowed tile,
        // backward 56.0 against 64.3 us; fp32 forward 54.0 us against 61.7 us
        // for the tile with warp roles, backward 93.7 against 118.0 us)
    } else if ((vi = find_variant(tab, n, dtype == LRSCAN_BF16 ? "gwin_bf16_d32_s8" : "gwin_f32_d32_s8", dir, B, D,
                                  g)) >= 0) {
        // the windowed tiles (time split inside the CTA): the measured fastest in both
        // directions wherever the lanes give the GPU at least 0.9 CTAs per SM
    } else if (!pick_from_table(tab, n, dir, B, D, g, &vi)) {
        long long most = -1;
        for (int i = 0; i < n; ++i) {
            const Occ o = occupancy(tab[i], dir, B, D, g);
            if (o.resident > 0 && o.ctas > most) { most = o.ctas; vi = i; }
        }
    }
    if (vi < 0) return fail(LRSCAN_EINVAL, "no generated-decay tile variant fits this device");
    const Occ o = occupancy(tab[vi], dir, B, D, g);
    if (o.resident == 0) return fail(LRSCAN_EINVAL, "tile variant %s does not fit on an SM", tab[vi].name);
    ch->vidx = vi;
    ch->var = &tab[vi];
    ch->ctas = o.ctas;
    ch->threads = dir_of(tab[vi], dir).threads;
    ch->smem = dir_of(tab[vi], dir).smem;
    ch->stages = dir_of(tab[vi], dir).nstage;
    return LRSCAN_OK;
}

int check_params(const float *eta, const float *nu_log) {
    if (!eta || !nu_log) return fail(LRSCAN_EINVAL, "NULL eta or nu_log");
    if (reinterpret_cast<uintptr_t>(eta) % 4 || reinterpret_cast<uintptr_t>(nu_log) % 4)
        return fail(LRSCAN_EINVAL, "eta and nu_log must be 4-byte aligned");
    return LRSCAN_OK;
}

int run_gfwd(const float *eta, const float *nu_log, const void *b, void *out, float *last, int64_t B, int64_t T,
             int64_t D, int dtype, void *stream, const lrscan_opts *opts) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    if (B == 0 || D == 0) return LRSCAN_OK;
    cudaStream_t st = pick_stream(stream);
    if (T == 0) return copy_or_zero(last, nullptr, B, D, st);
    if (!b || !out) return fail(LRSCAN_EINVAL, "NULL b or out");
    if ((rc = check_params(eta, nu_log))) return rc;
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool al = aligned16({b, out}, D, dtype);
    Choice ch;
    if ((rc = plan_gated(B, D, dtype, 0, al, opts, geometry_of(ctx), &ch))) return rc;
    WinLaunch L{};
    L.eta = eta;
    L.nu_log = nu_log;
    L.status = ctx->status;
    L.timeout_ns = g_timeout_ns.load();
    L.stream = st;
    L.device = dev;
    if (ch.path == kPathPlain) {
        L.in0 = b; L.out0 = out; L.last = last;
        L.B = B; L.T = T; L.D = D;
        return gplain_launch(L, dtype, true) ? fail(LRSCAN_ECUDA, "generated-decay plain launch failed") : LRSCAN_OK;
    }
    const size_t es = esize(dtype);
    const WinDirCfg &v = ch.var->fwd;
    for (int64_t b0 = 0; b0 < B; b0 += 65535) {
        const int64_t nb = std::min<int64_t>(65535, B - b0);
        const size_t off = static_cast<size_t>(b0) * T * D * es;
        CUtensorMap mb, mo;  // mo: the windowed tile writes out through a bulk tensor store
        if (encode_map(&mb, static_cast<const char *>(b) + off, dtype, nb, T, D, v.dt, v.w) ||
            encode_map(&mo, static_cast<char *>(out) + off, dtype, nb, T, D, v.dt, v.w))
            return LRSCAN_EINVAL;
        L.maps[0] = &mb;
        L.maps[1] = &mo;
        L.eta = eta + b0 * T;
        L.out0 = static_cast<char *>(out) + off;
        L.last = last ? last + b0 * D : nullptr;
        L.B = nb; L.T = T; L.D = D;
        if (v.launch(L, v))
            return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
    }
    return LRSCAN_OK;
}

int run_gbwd(const float *eta, const float *nu_log, const void *out, const void *grad_out, void *grad_b,
             float *grad_eta, float *grad_nu_log, int64_t B, int64_t T, int64_t D, int dtype, void *stream,
             const lrscan_opts *opts) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    if (B == 0 || D == 0) {
        if (D > 0 && grad_nu_log)  // no tokens: the rate gradient is zero
            return copy_or_zero(grad_nu_log, nullptr, 1, D, pick_stream(stream));
        return LRSCAN_OK;
    }
    cudaStream_t st = pick_stream(stream);
    if (T == 0) return copy_or_zero(grad_nu_log, nullptr, 1, D, st);  // no tokens: zero rate gradient
    if (!grad_eta || !grad_nu_log) return fail(LRSCAN_EINVAL, "NULL grad_eta or grad_nu_log");
    if (!out || !grad_out || !grad_b) return fail(LRSCAN_EINVAL, "NULL out, grad_out or grad_b");
    if ((rc = check_params(eta, nu_log))) return rc;
    if (reinterpret_cast<uintptr_t>(grad_eta) % 4 || reinterpret_cast<uintptr_t>(grad_nu_log) % 4)
        return fail(LRSCAN_EINVAL, "grad_eta and grad_nu_log must be 4-byte aligned");
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool al = aligned16({out, grad_out, grad_b}, D, dtype);
    Choice ch;
    if ((rc = plan_gated(B, D, dtype, 1, al, opts, geometry_of(ctx), &ch))) return rc;
    const size_t need = gated_workspace(B, T, D);
    void *ws = nullptr;
    if ((rc = workspace_for(ctx, st, need, opts, &ws))) return rc;
    float *part_eta = static_cast<float *>(ws);
    const size_t eta_bytes = (static_cast<size_t>(B) * T * gated_ncol_bound(D) * 4 + 255) / 256 * 256;
    float *part_nu = reinterpret_cast<float *>(static_cast<char *>(ws) + eta_bytes);
    WinLaunch L{};
    L.eta = eta;
    L.nu_log = nu_log;
    L.status = ctx->status;
    L.timeout_ns = g_timeout_ns.load();
    L.stream = st;
    L.device = dev;
    int ncol, nu_rows = static_cast<int>(B);
    if (ch.path == kPathPlain) {
        ncol = static_cast<int>((D + 31) / 32);
        L.in0 = out; L.in1 = grad_out; L.out0 = grad_b;
        L.part_eta = part_eta; L.part_nu = part_nu;
        L.B = B; L.T = T; L.D = D;
        if (gplain_launch(L, dtype, false)) return fail(LRSCAN_ECUDA, "generated-decay plain launch failed");
    } else {
        const WinDirCfg &v = ch.var->bwd;
        // windowed tile: one partial per (row, CTA) and per (batch row,
        // sub-chunk); sequential tile: one per (row, warp) and per batch row
        const bool win = v.s > 1;
        if (win && v.s > kGatedMaxS) return fail(LRSCAN_EINVAL, "internal: too many sub-chunks for the workspace");
        ncol = static_cast<int>(win ? (D + v.dt - 1) / v.dt : ((D + v.dt - 1) / v.dt) * (v.threads - 32) / 32);
        nu_rows = static_cast<int>(win ? B * v.s : B);
        const size_t es = esize(dtype);
        for (int64_t b0 = 0; b0 < B; b0 += 65535) {
            const int64_t nb = std::min<int64_t>(65535, B - b0);
            const size_t off = static_cast<size_t>(b0) * T * D * es;
            CUtensorMap mo, mg, mgb;  // mgb: the windowed tile writes grad_b through bulk tensor stores
            if (encode_map(&mo, static_cast<const char *>(out) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mg, static_cast<const char *>(grad_out) + off, dtype, nb, T, D, v.dt, v.w) ||
                encode_map(&mgb, static_cast<char *>(grad_b) + off, dtype, nb, T, D, v.dt, v.w))
                return LRSCAN_EINVAL;
            L.maps[0] = &mo;
            L.maps[1] = &mg;
            L.maps[2] = &mgb;
            L.eta = eta + b0 * T;
            L.out0 = static_cast<char *>(grad_b) + off;
            L.part_eta = part_eta + static_cast<size_t>(b0) * T;  // [ncol][B*T]: row offset of this slice
            L.part_rows = B * T;
            L.part_nu = part_nu + static_cast<size_t>(b0) * (win ? v.s : 1) * D;
            L.B = nb; L.T = T; L.D = D;
            if (v.launch(L, v))
                return fail(LRSCAN_ECUDA, "launch of %s: %s", ch.var->name, cudaGetErrorString(cudaGetLastError()));
        }
    }
    if (ncol > gated_ncol_bound(D)) return fail(LRSCAN_EINVAL, "internal: partial columns exceed the workspace");
    if (gated_finish_launch(part_eta, ncol, B * T, grad_eta, part_nu, nu_rows, static_cast<int>(D), grad_nu_log,
                            st))
        return fail(LRSCAN_ECUDA, "generated-decay reduction launch failed");
    return LRSCAN_OK;
}

}  // namespace

// Lets other translation units of the library report why a call failed.
int report_error(int code, const char *msg) { return fail(code, "%s", msg); }

// After `st` has drained: the first error a kernel recorded on the current
// device since the last check (cleared), else LRSCAN_OK.
int take_device_status(cudaStream_t st) {
    DeviceCtx *ctx = nullptr;
    int rc = device_ctx(&ctx);
    if (rc) return rc;
    DevStatus s{};
    if (cudaMemcpyAsync(&s, ctx->status, sizeof s, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return fail(LRSCAN_ECUDA, "reading the device status failed");
    }
    if (s.code != 0) {
        cudaMemsetAsync(ctx->status, 0, sizeof s, st);
        cudaStreamSynchronize(st);
        return fail(s.code, "a kernel reported error %d (wait site %d, block %u)", s.code, s.where, s.block);
    }
    return LRSCAN_OK;
}

}  // namespace lrscan

using namespace lrscan;

extern "C" {

int lrscan_fwd(const void *a, const void *b, void *out, float *last, int64_t B, int64_t T, int64_t D, int dtype) {
    return run_fwd(a, b, out, last, B, T, D, dtype, nullptr, nullptr);
}

int lrscan_bwd(const void *a, const void *out, const void *grad_out, void *grad_a, void *grad_b, int64_t B,
               int64_t T, int64_t D, int dtype) {
    return run_bwd(a, out, grad_out, grad_a, grad_b, B, T, D, dtype, nullptr, nullptr);
}

int lrscan_fwd_ex(const void *a, const void *b, void *out, float *last, int64_t B, int64_t T, int64_t D, int dtype,
                  void *stream, const lrscan_opts *opts) {
    return run_fwd(a, b, out, last, B, T, D, dtype, stream, opts);
}

int lrscan_bwd_ex(const void *a, const void *out, const void *grad_out, void *grad_a, void *grad_b, int64_t B,
                  int64_t T, int64_t D, int dtype, void *stream, const lrscan_opts *opts) {
    return run_bwd(a, out, grad_out, grad_a, grad_b, B, T, D, dtype, stream, opts);
}

int lrscan_fwd_state(const void *a, const void *b, void *out, float *last, const lrscan_state *state, int64_t B,
                     int64_t T, int64_t D, int dtype, void *stream, const lrscan_opts *opts) {
    return run_fwd(a, b, out, last, B, T, D, dtype, stream, opts, state);
}

int lrscan_bwd_state(const void *a, const void *out, const void *grad_out, void *grad_a, void *grad_b,
                     const lrscan_state *state, int64_t B, int64_t T, int64_t D, int dtype, void *stream,
                     const lrscan_opts *opts) {
    return run_bwd(a, out, grad_out, grad_a, grad_b, B, T, D, dtype, stream, opts, state);
}

int lrscan_summary(const void *a, const void *x, float *P, float *Q, const int32_t *segment_pos, int64_t B,
                   int64_t T, int64_t D, int dtype, int dir, void *stream) {
    t_detail[0] = 0;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    if (dir != 0 && dir != 1) return fail(LRSCAN_EINVAL, "dir %d is not 0 (forward) or 1 (backward)", dir);
    lrscan_state st{};
    st.segment_pos = segment_pos;
    bool ext = false;
    if ((rc = check_state(&st, false, &ext))) return rc;
    if (B == 0 || D == 0) return LRSCAN_OK;
    if (!P || !Q) return fail(LRSCAN_EINVAL, "NULL P or Q");
    if (reinterpret_cast<uintptr_t>(P) % 4 || reinterpret_cast<uintptr_t>(Q) % 4)
        return fail(LRSCAN_EINVAL, "P and Q must be 4-byte aligned");
    cudaStream_t s = pick_stream(stream);
    if (T == 0) {
        // the identity map h -> 1*h + 0
        if (cudaMemsetAsync(Q, 0, static_cast<size_t>(B) * D * 4, s) != cudaSuccess ||
            fill_f32_launch(P, static_cast<size_t>(B) * D, 1.0f, s)) {
            cudaGetLastError();
            return fail(LRSCAN_ECUDA, "T == 0 summary fill failed");
        }
        return LRSCAN_OK;
    }
    if (!a || !x) return fail(LRSCAN_EINVAL, "NULL a or x");
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx))) return rc;
    ChunkLaunch L{};
    L.in0 = a; L.in1 = x; L.P = P; L.Q = Q;
    L.B = B; L.T = T; L.D = D; L.stream = s;
    L.sx = state_slice(&st, false, a, 0, T, D, esize(dtype));
    if (summary_launch(L, dtype, dir))
        return fail(LRSCAN_ECUDA, "summary launch: %s", cudaGetErrorString(cudaGetLastError()));
    return LRSCAN_OK;
}

int lrscan_compose_maps(const float *maps, int64_t W, int64_t rank, const float *init, float *out, int64_t B,
                        int64_t D, int dir, void *stream) {
    t_detail[0] = 0;
    if (W < 1 || rank < 0 || rank >= W || B < 0 || D < 0 || W > 0x7fffffffLL)
        return fail(LRSCAN_EINVAL, "W=%lld rank=%lld B=%lld D=%lld", static_cast<long long>(W),
                    static_cast<long long>(rank), static_cast<long long>(B), static_cast<long long>(D));
    if (dir != 0 && dir != 1) return fail(LRSCAN_EINVAL, "dir %d is not 0 (forward) or 1 (backward)", dir);
    int64_t lanes = 0, total = 0;
    if (__builtin_mul_overflow(B, D, &lanes) || __builtin_mul_overflow(lanes, 2 * W, &total) ||
        __builtin_mul_overflow(total, static_cast<int64_t>(4), &total))
        return fail(LRSCAN_EINVAL, "W*2*B*D*4 overflows int64");
    if (lanes == 0) return LRSCAN_OK;
    if (!maps || !out) return fail(LRSCAN_EINVAL, "NULL maps or out");
    for (const void *p : {static_cast<const void *>(maps), static_cast<const void *>(init),
                          static_cast<const void *>(out)})
        if (reinterpret_cast<uintptr_t>(p) % 4) return fail(LRSCAN_EINVAL, "pointers must be 4-byte aligned");
    DeviceCtx *ctx = nullptr;
    int rc = device_ctx(&ctx);
    if (rc) return rc;
    // forward: maps 0..rank-1 in order; backward: maps W-1..rank+1
    const int r0 = dir == 0 ? 0 : static_cast<int>(W - 1);
    const int step = dir == 0 ? 1 : -1;
    const int n = dir == 0 ? static_cast<int>(rank) : static_cast<int>(W - 1 - rank);
    if (compose_maps_launch(maps, init, out, lanes, r0, step, n, pick_stream(stream)))
        return fail(LRSCAN_ECUDA, "compose launch: %s", cudaGetErrorString(cudaGetLastError()));
    return LRSCAN_OK;
}

int lrscan_cfwd(const void *ar, const void *ai, const void *br, const void *bi, void *out_r, void *out_i,
                float *last_r, float *last_i, int64_t B, int64_t T, int64_t D, int dtype, void *stream,
                const lrscan_opts *opts) {
    const void *in[4] = {ar, ai, br, bi};
    return run_cfwd(in, out_r, out_i, last_r, last_i, B, T, D, dtype, stream, opts);
}

int lrscan_cbwd(const void *ar, const void *ai, const void *out_r, const void *out_i, const void *grad_out_r,
                const void *grad_out_i, void *grad_ar, void *grad_ai, void *grad_br, void *grad_bi, int64_t B,
                int64_t T, int64_t D, int dtype, void *stream, const lrscan_opts *opts) {
    const void *in[6] = {ar, ai, out_r, out_i, grad_out_r, grad_out_i};
    void *const outp[4] = {grad_ar, grad_ai, grad_br, grad_bi};
    return run_cbwd(in, outp, B, T, D, dtype, stream, opts);
}

int lrscan_cfwd_state(const void *ar, const void *ai, const void *br, const void *bi, void *out_r, void *out_i,
                      float *last_r, float *last_i, const lrscan_cstate *state, int64_t B, int64_t T, int64_t D,
                      int dtype, void *stream, const lrscan_opts *opts) {
    const void *in[4] = {ar, ai, br, bi};
    return run_cfwd(in, out_r, out_i, last_r, last_i, B, T, D, dtype, stream, opts, state);
}

int lrscan_cbwd_state(const void *ar, const void *ai, const void *out_r, const void *out_i, const void *grad_out_r,
                      const void *grad_out_i, void *grad_ar, void *grad_ai, void *grad_br, void *grad_bi,
                      const lrscan_cstate *state, int64_t B, int64_t T, int64_t D, int dtype, void *stream,
                      const lrscan_opts *opts) {
    const void *in[6] = {ar, ai, out_r, out_i, grad_out_r, grad_out_i};
    void *const outp[4] = {grad_ar, grad_ai, grad_br, grad_bi};
    return run_cbwd(in, outp, B, T, D, dtype, stream, opts, state);
}

static int plan_complex_entry(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16,
                              const lrscan_opts *opts, lrscan_plan_info *info, bool ext) {
    if (!info || (dir != 0 && dir != 1)) return LRSCAN_EINVAL;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    DeviceCtx *ctx = nullptr;
    if (device_ctx(&ctx) != LRSCAN_OK) ctx = nullptr;
    const bool al = is_aligned16 && (D * esize(dtype)) % 16 == 0;
    Choice ch;
    if ((rc = plan_complex(B > 0 ? B : 1, T > 0 ? T : 1, D > 0 ? D : 1, dtype, dir, al, opts, geometry_of(ctx), &ch,
                           ext)))
        return rc;
    fill_info(ch, info);
    if (ch.path == kPathChunk) {
        info->lanes_per_cta = 128 * ch.vec;
        std::snprintf(info->name, sizeof info->name, "cchunk%d_v%d%s", ch.chunk, ch.vec, ch.vidx == 1 ? "_grouped" : "");
    }
    return LRSCAN_OK;
}

int lrscan_plan_complex(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16,
                        const lrscan_opts *opts, lrscan_plan_info *info) {
    return plan_complex_entry(B, T, D, dtype, dir, is_aligned16, opts, info, false);
}

int lrscan_plan_complex_state(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16,
                              const lrscan_opts *opts, lrscan_plan_info *info) {
    return plan_complex_entry(B, T, D, dtype, dir, is_aligned16, opts, info, true);
}

int lrscan_fwd_gated(const float *eta, const float *nu_log, const void *b, void *out, float *last, int64_t B,
                     int64_t T, int64_t D, int dtype, void *stream, const lrscan_opts *opts) {
    return run_gfwd(eta, nu_log, b, out, last, B, T, D, dtype, stream, opts);
}

int lrscan_bwd_gated(const float *eta, const float *nu_log, const void *out, const void *grad_out, void *grad_b,
                     float *grad_eta, float *grad_nu_log, int64_t B, int64_t T, int64_t D, int dtype, void *stream,
                     const lrscan_opts *opts) {
    return run_gbwd(eta, nu_log, out, grad_out, grad_b, grad_eta, grad_nu_log, B, T, D, dtype, stream, opts);
}

size_t lrscan_gated_workspace_bytes(int64_t B, int64_t T, int64_t D) {
    if (B <= 0 || T <= 0 || D <= 0) return 0;
    return gated_workspace(B, T, D);
}

int lrscan_plan_gated(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16, const lrscan_opts *opts,
                      lrscan_plan_info *info) {
    if (!info || (dir != 0 && dir != 1)) return LRSCAN_EINVAL;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    DeviceCtx *ctx = nullptr;
    if (device_ctx(&ctx) != LRSCAN_OK) ctx = nullptr;
    const bool al = is_aligned16 && (D * esize(dtype)) % 16 == 0;
    Choice ch;
    if ((rc = plan_gated(B > 0 ? B : 1, D > 0 ? D : 1, dtype, dir, al, opts, geometry_of(ctx), &ch))) return rc;
    if (dir == 1) ch.workspace = gated_workspace(B > 0 ? B : 1, T > 0 ? T : 1, D > 0 ? D : 1);
    fill_info(ch, info);
    info->exact = 0;  // generated decays use a fast exponential
    return LRSCAN_OK;
}

int lrscan_set_stream(void *stream) {
    t_stream = static_cast<cudaStream_t>(stream);
    return LRSCAN_OK;
}

size_t lrscan_workspace_bytes(int64_t B, int64_t T, int64_t D, int chunk_len) {
    const int C = chunk_len ? chunk_len : 64;
    if (B <= 0 || T <= 0 || D <= 0 ||
        (C != 16 && C != 32 && C != 64 && C != 128 && C != 256 && C != 512))
        return 0;
    return chunk_workspace(B, T, D, C);
}

static int plan_entry(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16, const lrscan_opts *opts,
                      lrscan_plan_info *info, bool ext) {
    if (!info || (dir != 0 && dir != 1)) return LRSCAN_EINVAL;
    int rc = check_shape(B, T, D, dtype);
    if (rc) return rc;
    DeviceCtx *ctx = nullptr;
    if (device_ctx(&ctx) != LRSCAN_OK) ctx = nullptr;  // no device: plan for one GB300
    const bool al = is_aligned16 && (D * esize(dtype)) % 16 == 0;
    Choice ch;
    if ((rc = plan_call(B > 0 ? B : 1, T > 0 ? T : 1, D > 0 ? D : 1, dtype, dir, al, opts, geometry_of(ctx), &ch,
                        ext)))
        return rc;
    fill_info(ch, info);
    return LRSCAN_OK;
}

int lrscan_plan(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16, const lrscan_opts *opts,
                lrscan_plan_info *info) {
    return plan_entry(B, T, D, dtype, dir, is_aligned16, opts, info, false);
}

int lrscan_plan_state(int64_t B, int64_t T, int64_t D, int dtype, int dir, int is_aligned16,
                      const lrscan_opts *opts, lrscan_plan_info *info) {
    return plan_entry(B, T, D, dtype, dir, is_aligned16, opts, info, true);
}

int lrscan_num_variants(int path, int dtype, int dir) {
    (void)dir;
    if (dtype != LRSCAN_F32 && dtype != LRSCAN_BF16) return LRSCAN_EDTYPE;
    if (path == kPathSeq || path == kPathWindow) {
        int n = 0;
        win_variants(path, dtype, &n);
        return n;
    }
    if (path == kPathStream) {
        int n = 0;
        stream_variants(dtype, &n);
        return n;
    }
    if (path == kPathChunk || path == kPathPlain) return 1;
    return LRSCAN_EINVAL;
}

int lrscan_sync_check(void) {
    DeviceCtx *ctx = nullptr;
    int rc = device_ctx(&ctx);
    if (rc) return rc;
    cudaStream_t st = t_stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return LRSCAN_ECUDA;
    }
    DevStatus s{};
    if (cudaMemcpyAsync(&s, ctx->status, sizeof s, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return LRSCAN_ECUDA;
    }
    if (s.code != 0) {
        cudaMemsetAsync(ctx->status, 0, sizeof s, st);
        cudaStreamSynchronize(st);
        return s.code;
    }
    return LRSCAN_OK;
}

int lrscan_set_wait_timeout_ns(uint64_t ns) {
    // The same limit bounds the waits with which a kernel drains its own bulk
    // copies before it exits: those land within microseconds, and a limit that
    // gave up before they did would let a CTA leave with copies still writing
    // into its shared memory.
    if (ns < 1000000ull) return fail(LRSCAN_EINVAL, "wait limit %llu ns is under 1 ms", static_cast<unsigned long long>(ns));
    g_timeout_ns.store(ns);
    return LRSCAN_OK;
}

int lrscan_selftest_wait_timeout(uint64_t timeout_ns) {
    DeviceCtx *ctx = nullptr;
    int rc = device_ctx(&ctx);
    if (rc) return rc;
    if (timeout_ns == 0 || timeout_ns > 10ull * 1000000000ull) return LRSCAN_EINVAL;
    if (selftest_wait_launch(ctx->status, timeout_ns, t_stream)) return LRSCAN_ECUDA;
    return lrscan_sync_check();
}

const char *lrscan_strerror(int code) {
    switch (code) {
        case LRSCAN_OK: return "success";
        case LRSCAN_EINVAL: return "invalid argument";
        case LRSCAN_EDTYPE: return "unsupported dtype";
        case LRSCAN_ECUDA: return "CUDA runtime error";
        case LRSCAN_ENOMEM: return "workspace allocation failed or too small";
        case LRSCAN_ETIMEOUT: return "a bounded device wait timed out";
        case LRSCAN_ENODEVICE: return "no usable sm_103 device";
        default: return "unknown error";
    }
}

int lrscan_version(void) { return LRSCAN_VERSION; }

const char *lrscan_last_error(void) { return t_detail; }

}  // extern "C"
