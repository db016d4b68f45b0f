/*
 * lrscan oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, obviously correct CPU statement of the differentiable
 * diagonal linear-recurrence scan.  Only the test-suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load this library; the CUDA
 * library never links, includes or calls it, and it shares no code, header or
 * helper with the CUDA sources.
 *
 * What is computed (per batch row b and channel lane d, contiguous [B,T,D]
 * layout with D fastest, as in triton_training_scan.py, _real_forward, where
 * the element offset is (batch*length + t)*width + lane):
 *
 *   forward   h_{-1} = 0,  h_t = a_t * h_{t-1} + b_t   (t = 0..T-1)
 *             out_t = h_t stored in the storage dtype, last = h_{T-1} in fp32
 *             (triton_training_scan.py, _real_forward and real_scan_with_last)
 *
 *   backward  loss L = sum_t grad_out_t * h_t, with h read back from `out`:
 *             g_{T-1} = grad_out_{T-1}
 *             g_t     = grad_out_t + a_{t+1} * g_{t+1}
 *             grad_b_t = g_t
 *             grad_a_t = g_t * out_{t-1}   (out_{-1} = 0)
 *             (triton_training_scan.py, _real_backward)
 *
 * Readings taken where the page is silent (each is listed in the design
 * notes of the repository):
 *   - one rounding per recurrence step: h = fma(a, h, b) and
 *     g = fma(a_{t+1}, g_{t+1}, grad_out_t); grad_a is one rounded product;
 *   - state and accumulation are fp32 whatever the storage dtype; fp32 ->
 *     bf16 is round-to-nearest-even;
 *   - in the bf16 variant the backward reads h_{t-1} from the bf16-stored out.
 *
 * The "chunk" variants restate the two-level affine-map decomposition of the
 * same page (_real_chunk_summary, _real_chunk_prefix, _real_chunk_replay and
 * their _real_reverse_* mirrors) step by step in the page's own order, with
 * the page's reverse carry (the adjoint that leaves a step, a_t*(k+grad_out_t)).
 * They exist only so the tests can check the algebra of that decomposition
 * against the sequential definition.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math: the
 * rounding of every operation above is part of the contract).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define LRO_OK 0
#define LRO_EINVAL (-1)
#define LRO_ENOMEM (-2)

/* ---------------------------------------------------------------------- */
/* bf16 storage: the top 16 bits of an IEEE-754 binary32 value.            */
/* ---------------------------------------------------------------------- */

/* Widening is exact: the bf16 bits become the high half of a binary32. */
float lro_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Narrowing by round-to-nearest, ties-to-even on the 16 discarded bits.
 * NaN stays NaN (quiet bit forced so the truncation cannot make an inf). */
uint16_t lro_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;    /* parity of the kept part */
    u += 0x7fffu + keep_lsb;               /* > half rounds up; == half to even */
    return (uint16_t)(u >> 16);
}

void lro_f32_to_bf16_array(const float *src, uint16_t *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = lro_f32_to_bf16(src[i]);
}

void lro_bf16_to_f32_array(const uint16_t *src, float *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = lro_bf16_to_f32(src[i]);
}

static int bad_shape(int64_t B, int64_t T, int64_t D)
{
    return B < 0 || T < 0 || D < 0;
}

/* ---------------------------------------------------------------------- */
/* Sequential forward                                                      */
/* ---------------------------------------------------------------------- */

int lro_fwd_f32(const float *a, const float *b, float *out, float *last,
                int64_t B, int64_t T, int64_t D)
{
    if (bad_shape(B, T, D)) return LRO_EINVAL;
    float *h = calloc((size_t)(D > 0 ? D : 1), sizeof *h);
    if (!h) return LRO_ENOMEM;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t d = 0; d < D; ++d) h[d] = 0.0f;
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t i = (bb * T + t) * D + d;
                h[d] = fmaf(a[i], h[d], b[i]);
                out[i] = h[d];
            }
        }
        if (last)
            for (int64_t d = 0; d < D; ++d) last[bb * D + d] = h[d];
    }
    free(h);
    return LRO_OK;
}

int lro_fwd_bf16(const uint16_t *a, const uint16_t *b, uint16_t *out,
                 float *last, int64_t B, int64_t T, int64_t D)
{
    if (bad_shape(B, T, D)) return LRO_EINVAL;
    float *h = calloc((size_t)(D > 0 ? D : 1), sizeof *h);
    if (!h) return LRO_ENOMEM;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t d = 0; d < D; ++d) h[d] = 0.0f;
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t i = (bb * T + t) * D + d;
                h[d] = fmaf(lro_bf16_to_f32(a[i]), h[d], lro_bf16_to_f32(b[i]));
                out[i] = lro_f32_to_bf16(h[d]);
            }
        }
        if (last)
            for (int64_t d = 0; d < D; ++d) last[bb * D + d] = h[d];
    }
    free(h);
    return LRO_OK;
}

int lro_fwd_f64(const double *a, const double *b, double *out, double *last,
                int64_t B, int64_t T, int64_t D)
{
    if (bad_shape(B, T, D)) return LRO_EINVAL;
    double *h = calloc((size_t)(D > 0 ? D : 1), sizeof *h);
    if (!h) return LRO_ENOMEM;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t d = 0; d < D; ++d) h[d] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t i = (bb * T + t) * D + d;
                h[d] = fma(a[i], h[d], b[i]);
                out[i] = h[d];
            }
        }
        if (last)
            for (int64_t d = 0; d < D; ++d) last[bb * D + d] = h[d];
    }
    free(h);
    return LRO_OK;
}

/* ---------------------------------------------------------------------- */
/* Sequential backward                                                     */
/* ---------------------------------------------------------------------- */

int lro_bwd_f32(const float *a, const float *out, const float *grad_out,
                float *grad_a, float *grad_b, int64_t B, int64_t T, int64_t D)
{
    if (bad_shape(B, T, D)) return LRO_EINVAL;
    float *g = calloc((size_t)(D > 0 ? D : 1), sizeof *g);
    if (!g) return LRO_ENOMEM;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t t = T - 1; t >= 0; --t) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t i = (bb * T + t) * D + d;
                if (t == T - 1)
                    g[d] = grad_out[i];
                else
                    g[d] = fmaf(a[i + D], g[d], grad_out[i]); /* a_{t+1} */
                float h_prev = (t > 0) ? out[i - D] : 0.0f;   /* out_{t-1} */
                grad_b[i] = g[d];
                grad_a[i] = g[d] * h_prev;
            }
        }
    }
    free(g);
    return LRO_OK;
}

int lro_bwd_bf16(const uint16_t *a, const uint16_t *out,
                 const uint16_t *grad_out, uint16_t *grad_a, uint16_t *grad_b,
                 int64_t B, int64_t T, int64_t D)
{
    if (bad_shape(B, T, D)) return LRO_EINVAL;
    float *g = calloc((size_t)(D > 0 ? D : 1), sizeof *g);
    if (!g) return LRO_ENOMEM;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t t = T - 1; t >= 0; --t) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t i = (bb * T + t) * D + d;
                float go = lro_bf16_to_f32(grad_out[i]);
                if (t == T - 1)
                    g[d] = go;
                else
                    g[d] = fmaf(lro_bf16_to_f32(a[i + D]), g[d], go);
                float h_prev = (t > 0) ? lro_bf16_to_f32(out[i - D]) : 0.0f;
                grad_b[i] = lro_f32_to_bf16(g[d]);
                grad_a[i] = lro_f32_to_bf16(g[d] * h_prev);
            }
        }
    }
    free(g);
    return LRO_OK;
}

int lro_bwd_f64(const double *a, const double *out, const double *grad_out,
                double *grad_a, double *grad_b, int64_t B, int64_t T, int64_t D)
{
    if (bad_shape(B, T, D)) return LRO_EINVAL;
    double *g = calloc((size_t)(D > 0 ? D : 1), sizeof *g);
    if (!g) return LRO_ENOMEM;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t t = T - 1; t >= 0; --t) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t i = (bb * T + t) * D + d;
                if (t == T - 1)
                    g[d] = grad_out[i];
                else
                    g[d] = fma(a[i + D], g[d], grad_out[i]);
                double h_prev = (t > 0) ? out[i - D] : 0.0;
                grad_b[i] = g[d];
                grad_a[i] = g[d] * h_prev;
            }
        }
    }
    free(g);
    return LRO_OK;
}

/* ---------------------------------------------------------------------- */
/* Two-level (chunked) decomposition, in the page's order.                 */
/* A chunk c covers steps [c*C, min((c+1)*C, T)); a short last chunk is    */
/* simply shorter (equivalent to padding it with identity steps a=1, b=0). */
/* ---------------------------------------------------------------------- */

#define CHUNK_BODY_FWD(REAL, FMA)                                              \
    int64_t nc = (T + C - 1) / C;                                              \
    REAL *P = malloc(sizeof(REAL) * (size_t)(nc > 0 ? nc : 1));               \
    REAL *Q = malloc(sizeof(REAL) * (size_t)(nc > 0 ? nc : 1));               \
    REAL *hin = malloc(sizeof(REAL) * (size_t)(nc > 0 ? nc : 1));             \
    if (!P || !Q || !hin) { free(P); free(Q); free(hin); return LRO_ENOMEM; } \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            /* chunk summary: h -> P*h + Q over the chunk */                   \
            for (int64_t c = 0; c < nc; ++c) {                                 \
                REAL prod = 1, state = 0;                                      \
                for (int64_t t = c * C; t < T && t < (c + 1) * C; ++t) {       \
                    int64_t i = (bb * T + t) * D + d;                          \
                    prod = a[i] * prod;                                        \
                    state = FMA(a[i], state, b[i]);                            \
                }                                                              \
                P[c] = prod;                                                   \
                Q[c] = state;                                                  \
            }                                                                  \
            /* serial exclusive prefix over chunks */                          \
            REAL state = 0;                                                    \
            for (int64_t c = 0; c < nc; ++c) {                                 \
                hin[c] = state;                                                \
                state = FMA(P[c], state, Q[c]);                                \
            }                                                                  \
            /* replay every chunk from its entry state */                      \
            for (int64_t c = 0; c < nc; ++c) {                                 \
                REAL h = hin[c];                                               \
                for (int64_t t = c * C; t < T && t < (c + 1) * C; ++t) {       \
                    int64_t i = (bb * T + t) * D + d;                          \
                    h = FMA(a[i], h, b[i]);                                    \
                    out[i] = h;                                                \
                }                                                              \
                if (c == nc - 1 && last) last[bb * D + d] = h;                 \
            }                                                                  \
            if (T == 0 && last) last[bb * D + d] = 0;                          \
        }                                                                      \
    }                                                                          \
    free(P); free(Q); free(hin);                                               \
    return LRO_OK;

#define CHUNK_BODY_BWD(REAL)                                                   \
    int64_t nc = (T + C - 1) / C;                                              \
    REAL *P = malloc(sizeof(REAL) * (size_t)(nc > 0 ? nc : 1));               \
    REAL *Q = malloc(sizeof(REAL) * (size_t)(nc > 0 ? nc : 1));               \
    REAL *fut = malloc(sizeof(REAL) * (size_t)(nc > 0 ? nc : 1));             \
    if (!P || !Q || !fut) { free(P); free(Q); free(fut); return LRO_ENOMEM; } \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            /* reverse summary: carry k leaving the chunk's first step */      \
            for (int64_t c = 0; c < nc; ++c) {                                 \
                REAL prod = 1, k = 0;                                          \
                int64_t hi = (c + 1) * C < T ? (c + 1) * C : T;                \
                for (int64_t t = hi - 1; t >= c * C; --t) {                    \
                    int64_t i = (bb * T + t) * D + d;                          \
                    prod = a[i] * prod;                                        \
                    k = a[i] * k + a[i] * grad_out[i];                         \
                }                                                              \
                P[c] = prod;                                                   \
                Q[c] = k;                                                      \
            }                                                                  \
            /* serial exclusive prefix from the last chunk down */             \
            REAL k = 0;                                                        \
            for (int64_t c = nc - 1; c >= 0; --c) {                            \
                fut[c] = k;                                                    \
                k = P[c] * k + Q[c];                                           \
            }                                                                  \
            /* replay: the sequential reverse body inside every chunk */      \
            for (int64_t c = 0; c < nc; ++c) {                                 \
                REAL adj = fut[c];                                             \
                int64_t hi = (c + 1) * C < T ? (c + 1) * C : T;                \
                for (int64_t t = hi - 1; t >= c * C; --t) {                    \
                    int64_t i = (bb * T + t) * D + d;                          \
                    adj = adj + grad_out[i];                                   \
                    REAL prev = (t > 0) ? out[i - D] : 0;                      \
                    grad_a[i] = adj * prev;                                    \
                    grad_b[i] = adj;                                           \
                    adj = adj * a[i];                                          \
                }                                                              \
            }                                                                  \
        }                                                                      \
    }                                                                          \
    free(P); free(Q); free(fut);                                               \
    return LRO_OK;

int lro_chunk_fwd_f32(const float *a, const float *b, float *out, float *last,
                      int64_t B, int64_t T, int64_t D, int64_t C)
{
    if (bad_shape(B, T, D) || C <= 0) return LRO_EINVAL;
    CHUNK_BODY_FWD(float, fmaf)
}

int lro_chunk_fwd_f64(const double *a, const double *b, double *out,
                      double *last, int64_t B, int64_t T, int64_t D, int64_t C)
{
    if (bad_shape(B, T, D) || C <= 0) return LRO_EINVAL;
    CHUNK_BODY_FWD(double, fma)
}

int lro_chunk_bwd_f32(const float *a, const float *out, const float *grad_out,
                      float *grad_a, float *grad_b, int64_t B, int64_t T,
                      int64_t D, int64_t C)
{
    if (bad_shape(B, T, D) || C <= 0) return LRO_EINVAL;
    CHUNK_BODY_BWD(float)
}

int lro_chunk_bwd_f64(const double *a, const double *out,
                      const double *grad_out, double *grad_a, double *grad_b,
                      int64_t B, int64_t T, int64_t D, int64_t C)
{
    if (bad_shape(B, T, D) || C <= 0) return LRO_EINVAL;
    CHUNK_BODY_BWD(double)
}

/* ---------------------------------------------------------------------- */
/* Carried state and segment resets.                                       */
/*                                                                         */
/* The state-carrying scans of triton_training_scan.py (_samu_tiled_serial */
/* _forward and _samu_tiled_serial_backward: optional initial state h0, a  */
/* per-token segment position whose zeros start a new segment, the         */
/* gradient arriving at the final state, the gradient of the initial       */
/* state) applied to the plain real recurrence; recurrence.py of the KDN    */
/* page carries the same state across calls so that prefill and decode      */
/* continue one sequence exactly.                                           */
/*                                                                         */
/*   forward   h_{-1} = h0 (0 when absent)                                 */
/*             a'_t = 0 where segment_pos[b,t] == 0, else a_t               */
/*             h_t = a'_t * h_{t-1} + b_t;  out_t = h_t;  last = h_{T-1}    */
/*   backward  g_T = grad_last (0 when absent) entering through a'_T = 1    */
/*             g_t = grad_out_t + a'_{t+1} * g_{t+1}    (one rounding)      */
/*             grad_b_t = g_t                                               */
/*             grad_a_t = +0 where step t resets (a_t is not used there),   */
/*                        else g_t * out_{t-1}, with out_{-1} = h0          */
/*             grad_h0  = a'_0 * g_0  (= grad_last when T == 0)             */
/*                                                                         */
/* h0, grad_last and grad_h0 are [B,D] in the state precision (fp32 for    */
/* the fp32 and bf16 storage variants, fp64 for the fp64 one); segment_pos */
/* is int32 [B,T].  Every pointer of the extension may be NULL.            */
/* ---------------------------------------------------------------------- */

static int resets(const int32_t *seg, int64_t bb, int64_t T, int64_t t)
{
    return seg != NULL && t >= 0 && t < T && seg[bb * T + t] == 0;
}

#define STATE_FWD_BODY(STATE, FMA, LOAD, STORE)                                \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE h = h0 ? h0[bb * D + d] : 0;                                 \
            for (int64_t t = 0; t < T; ++t) {                                  \
                int64_t i = (bb * T + t) * D + d;                              \
                STATE x = resets(seg, bb, T, t) ? 0 : LOAD(a[i]);              \
                h = FMA(x, h, LOAD(b[i]));                                     \
                out[i] = STORE(h);                                             \
            }                                                                  \
            if (last) last[bb * D + d] = h;                                    \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

#define STATE_BWD_BODY(STATE, FMA, LOAD, STORE)                                \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE g = grad_last ? grad_last[bb * D + d] : 0;                   \
            for (int64_t t = T - 1; t >= 0; --t) {                             \
                int64_t i = (bb * T + t) * D + d;                              \
                /* a'_{t+1}: 1 past the end (the grad_last entry), 0 at a      \
                 * reset */                                                    \
                STATE x_next = (t == T - 1) ? 1                                \
                               : (resets(seg, bb, T, t + 1) ? 0 : LOAD(a[i + D])); \
                g = FMA(x_next, g, LOAD(grad_out[i]));                         \
                STATE h_prev = (t > 0) ? LOAD(out[i - D])                      \
                               : (h0 ? h0[bb * D + d] : 0);                    \
                grad_b[i] = STORE(g);                                          \
                grad_a[i] = resets(seg, bb, T, t) ? STORE(0) : STORE(g * h_prev); \
            }                                                                  \
            if (grad_h0) {                                                     \
                if (T == 0)                                                    \
                    grad_h0[bb * D + d] = g;                                   \
                else                                                           \
                    grad_h0[bb * D + d] = resets(seg, bb, T, 0)                \
                                          ? 0 : LOAD(a[bb * T * D + d]) * g;   \
            }                                                                  \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

#define LRO_SAME(x) (x)

int lro_fwd_state_f32(const float *a, const float *b, float *out, float *last,
                      const float *h0, const int32_t *seg,
                      int64_t B, int64_t T, int64_t D)
{
    STATE_FWD_BODY(float, fmaf, LRO_SAME, LRO_SAME)
}

int lro_fwd_state_bf16(const uint16_t *a, const uint16_t *b, uint16_t *out,
                       float *last, const float *h0, const int32_t *seg,
                       int64_t B, int64_t T, int64_t D)
{
    STATE_FWD_BODY(float, fmaf, lro_bf16_to_f32, lro_f32_to_bf16)
}

int lro_fwd_state_f64(const double *a, const double *b, double *out,
                      double *last, const double *h0, const int32_t *seg,
                      int64_t B, int64_t T, int64_t D)
{
    STATE_FWD_BODY(double, fma, LRO_SAME, LRO_SAME)
}

int lro_bwd_state_f32(const float *a, const float *out, const float *grad_out,
                      const float *h0, const int32_t *seg,
                      const float *grad_last, float *grad_a, float *grad_b,
                      float *grad_h0, int64_t B, int64_t T, int64_t D)
{
    STATE_BWD_BODY(float, fmaf, LRO_SAME, LRO_SAME)
}

int lro_bwd_state_bf16(const uint16_t *a, const uint16_t *out,
                       const uint16_t *grad_out, const float *h0,
                       const int32_t *seg, const float *grad_last,
                       uint16_t *grad_a, uint16_t *grad_b, float *grad_h0,
                       int64_t B, int64_t T, int64_t D)
{
    STATE_BWD_BODY(float, fmaf, lro_bf16_to_f32, lro_f32_to_bf16)
}

int lro_bwd_state_f64(const double *a, const double *out,
                      const double *grad_out, const double *h0,
                      const int32_t *seg, const double *grad_last,
                      double *grad_a, double *grad_b, double *grad_h0,
                      int64_t B, int64_t T, int64_t D)
{
    STATE_BWD_BODY(double, fma, LRO_SAME, LRO_SAME)
}

/* ---------------------------------------------------------------------- */
/* Complex diagonal scan on separate real / imaginary planes.              */
/*                                                                         */
/* triton_training_scan.py, _complex_forward / _complex_backward and       */
/* complex_scan_with_last: per lane, with complex a_t = ar + i*ai and      */
/* b_t = br + i*bi,                                                        */
/*   forward   h_{-1} = 0,  h_t = a_t * h_{t-1} + b_t;                      */
/*             out_r/out_i = Re/Im h_t in the storage dtype, last_r/last_i  */
/*             = Re/Im h_{T-1} in fp32                                      */
/*   backward  loss L = sum_t Re(conj(grad_out_t) * h_t)                    */
/*             = sum_t (go_r*h_r + go_i*h_i):                               */
/*             g_{T-1} = grad_out_{T-1},                                    */
/*             g_t = grad_out_t + conj(a_{t+1}) * g_{t+1}  (the adjoint     */
/*                   carries the conjugate transition),                     */
/*             grad_b_t = g_t,  grad_a_t = g_t * conj(h_{t-1})  (h_{-1} = 0) */
/*             i.e. grad_ar = gr*pr + gi*pi, grad_ai = gi*pr - gr*pi.       */
/* Rounding reading (the page leaves contraction to the compiler): each     */
/* component is two nested fused multiply-adds,                             */
/*   h_r = fma(ar, h_r, fma(-ai, h_i, br)),  h_i = fma(ai, h_r, fma(ar, h_i, bi)) */
/*   g_r = fma(ar', g_r, fma(ai', g_i, go_r)), g_i = fma(ar', g_i, fma(-ai', g_r, go_i)) */
/*   grad_ar = fma(gr, pr, gi*pi),  grad_ai = fma(gi, pr, -(gr*pi))         */
/* (ar', ai' = a_{t+1}; the product inside is rounded once).               */
/* ---------------------------------------------------------------------- */

#define CPLX_FWD_BODY(STATE, FMA, LOAD, STORE)                                 \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE hr = 0, hi = 0;                                              \
            for (int64_t t = 0; t < T; ++t) {                                  \
                int64_t i = (bb * T + t) * D + d;                              \
                STATE xr = LOAD(ar[i]), xi = LOAD(ai[i]);                      \
                STATE nr = FMA(xr, hr, FMA(-xi, hi, LOAD(br[i])));             \
                STATE ni = FMA(xi, hr, FMA(xr, hi, LOAD(bi[i])));              \
                hr = nr;                                                       \
                hi = ni;                                                       \
                out_r[i] = STORE(hr);                                          \
                out_i[i] = STORE(hi);                                          \
            }                                                                  \
            if (last_r) last_r[bb * D + d] = hr;                               \
            if (last_i) last_i[bb * D + d] = hi;                               \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

#define CPLX_BWD_BODY(STATE, FMA, LOAD, STORE)                                 \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE gr = 0, gi = 0;                                              \
            for (int64_t t = T - 1; t >= 0; --t) {                             \
                int64_t i = (bb * T + t) * D + d;                              \
                STATE yr = LOAD(go_r[i]), yi = LOAD(go_i[i]);                  \
                if (t == T - 1) {                                              \
                    gr = yr;                                                   \
                    gi = yi;                                                   \
                } else {                                                       \
                    STATE xr = LOAD(ar[i + D]), xi = LOAD(ai[i + D]);          \
                    STATE nr = FMA(xr, gr, FMA(xi, gi, yr));                   \
                    STATE ni = FMA(xr, gi, FMA(-xi, gr, yi));                  \
                    gr = nr;                                                   \
                    gi = ni;                                                   \
                }                                                              \
                STATE pr = (t > 0) ? LOAD(out_r[i - D]) : 0;                   \
                STATE pi = (t > 0) ? LOAD(out_i[i - D]) : 0;                   \
                grad_br[i] = STORE(gr);                                        \
                grad_bi[i] = STORE(gi);                                        \
                grad_ar[i] = STORE(FMA(gr, pr, gi * pi));                      \
                grad_ai[i] = STORE(FMA(gi, pr, -(gr * pi)));                   \
            }                                                                  \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

int lro_cfwd_f32(const float *ar, const float *ai, const float *br,
                 const float *bi, float *out_r, float *out_i, float *last_r,
                 float *last_i, int64_t B, int64_t T, int64_t D)
{
    CPLX_FWD_BODY(float, fmaf, LRO_SAME, LRO_SAME)
}

int lro_cfwd_bf16(const uint16_t *ar, const uint16_t *ai, const uint16_t *br,
                  const uint16_t *bi, uint16_t *out_r, uint16_t *out_i,
                  float *last_r, float *last_i, int64_t B, int64_t T, int64_t D)
{
    CPLX_FWD_BODY(float, fmaf, lro_bf16_to_f32, lro_f32_to_bf16)
}

int lro_cfwd_f64(const double *ar, const double *ai, const double *br,
                 const double *bi, double *out_r, double *out_i,
                 double *last_r, double *last_i, int64_t B, int64_t T, int64_t D)
{
    CPLX_FWD_BODY(double, fma, LRO_SAME, LRO_SAME)
}

int lro_cbwd_f32(const float *ar, const float *ai, const float *out_r,
                 const float *out_i, const float *go_r, const float *go_i,
                 float *grad_ar, float *grad_ai, float *grad_br, float *grad_bi,
                 int64_t B, int64_t T, int64_t D)
{
    CPLX_BWD_BODY(float, fmaf, LRO_SAME, LRO_SAME)
}

int lro_cbwd_bf16(const uint16_t *ar, const uint16_t *ai, const uint16_t *out_r,
                  const uint16_t *out_i, const uint16_t *go_r,
                  const uint16_t *go_i, uint16_t *grad_ar, uint16_t *grad_ai,
                  uint16_t *grad_br, uint16_t *grad_bi, int64_t B, int64_t T,
                  int64_t D)
{
    CPLX_BWD_BODY(float, fmaf, lro_bf16_to_f32, lro_f32_to_bf16)
}

int lro_cbwd_f64(const double *ar, const double *ai, const double *out_r,
                 const double *out_i, const double *go_r, const double *go_i,
                 double *grad_ar, double *grad_ai, double *grad_br,
                 double *grad_bi, int64_t B, int64_t T, int64_t D)
{
    CPLX_BWD_BODY(double, fma, LRO_SAME, LRO_SAME)
}

/* ---------------------------------------------------------------------- */
/* Complex scan with carried state and segment resets.                     */
/*                                                                         */
/* triton_training_scan.py, _samu_tiled_serial_forward /                    */
/* _samu_tiled_serial_backward: the page's state-carrying scan is complex  */
/* (an initial state, RESET_FIRST restarts, the gradient arriving at the   */
/* final state and the gradient of the initial state).  With the complex   */
/* steps above and the state rules of the real state-carrying scan:        */
/*   forward   h_{-1} = h0 (0 when absent); a'_t = 0 where segment_pos is 0 */
/*             h_t = a'_t * h_{t-1} + b_t;  last = h_{T-1} (h0 when T = 0)   */
/*   backward  g_T = grad_last (0 when absent) entering through a'_T = 1:   */
/*             g_{T-1} = grad_out_{T-1} + grad_last (one rounding per part) */
/*             g_t = grad_out_t + conj(a'_{t+1}) * g_{t+1}                  */
/*             grad_b_t = g_t; grad_a_t = +0 where step t resets, else      */
/*             g_t * conj(h_{t-1}) with h_{-1} = h0;                        */
/*             grad_h0 = conj(a'_0) * g_0 (+0 at a reset; grad_last when    */
/*             T = 0).                                                      */
/* h0 / grad_last / grad_h0 are re and im [B,D] arrays in the state         */
/* precision; every pointer of the extension may be NULL.                  */
/* ---------------------------------------------------------------------- */

#define CPLX_STATE_FWD_BODY(STATE, FMA, LOAD, STORE)                           \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE hr = h0_r ? h0_r[bb * D + d] : 0;                            \
            STATE hi = h0_i ? h0_i[bb * D + d] : 0;                            \
            for (int64_t t = 0; t < T; ++t) {                                  \
                int64_t i = (bb * T + t) * D + d;                              \
                int r = resets(seg, bb, T, t);                                 \
                STATE xr = r ? 0 : LOAD(ar[i]), xi = r ? 0 : LOAD(ai[i]);      \
                STATE nr = FMA(xr, hr, FMA(-xi, hi, LOAD(br[i])));             \
                STATE ni = FMA(xi, hr, FMA(xr, hi, LOAD(bi[i])));              \
                hr = nr;                                                       \
                hi = ni;                                                       \
                out_r[i] = STORE(hr);                                          \
                out_i[i] = STORE(hi);                                          \
            }                                                                  \
            if (last_r) last_r[bb * D + d] = hr;                               \
            if (last_i) last_i[bb * D + d] = hi;                               \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

#define CPLX_STATE_BWD_BODY(STATE, FMA, LOAD, STORE)                           \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE gr = gl_r ? gl_r[bb * D + d] : 0;                            \
            STATE gi = gl_i ? gl_i[bb * D + d] : 0;                            \
            for (int64_t t = T - 1; t >= 0; --t) {                             \
                int64_t i = (bb * T + t) * D + d;                              \
                /* conj(a'_{t+1}): 1 past the end (the grad_last entry), 0 at  \
                 * a reset */                                                  \
                STATE xr, xi;                                                  \
                if (t == T - 1) {                                              \
                    xr = 1;                                                    \
                    xi = 0;                                                    \
                } else if (resets(seg, bb, T, t + 1)) {                        \
                    xr = 0;                                                    \
                    xi = 0;                                                    \
                } else {                                                       \
                    xr = LOAD(ar[i + D]);                                      \
                    xi = LOAD(ai[i + D]);                                      \
                }                                                              \
                STATE yr = LOAD(go_r[i]), yi = LOAD(go_i[i]);                  \
                STATE nr = FMA(xr, gr, FMA(xi, gi, yr));                       \
                STATE ni = FMA(xr, gi, FMA(-xi, gr, yi));                      \
                gr = nr;                                                       \
                gi = ni;                                                       \
                STATE pr = (t > 0) ? LOAD(out_r[i - D]) : (h0_r ? h0_r[bb * D + d] : 0); \
                STATE pi = (t > 0) ? LOAD(out_i[i - D]) : (h0_i ? h0_i[bb * D + d] : 0); \
                grad_br[i] = STORE(gr);                                        \
                grad_bi[i] = STORE(gi);                                        \
                if (resets(seg, bb, T, t)) {                                   \
                    grad_ar[i] = STORE(0);                                     \
                    grad_ai[i] = STORE(0);                                     \
                } else {                                                       \
                    grad_ar[i] = STORE(FMA(gr, pr, gi * pi));                  \
                    grad_ai[i] = STORE(FMA(gi, pr, -(gr * pi)));               \
                }                                                              \
            }                                                                  \
            if (gh0_r || gh0_i) {                                              \
                STATE hr = gr, hi = gi;                                        \
                if (T > 0 && resets(seg, bb, T, 0)) {                          \
                    hr = 0; /* a'_0 = 0: exactly +0 */                         \
                    hi = 0;                                                    \
                } else if (T > 0) {                                            \
                    /* conj(a'_0) * g_0 */                                     \
                    int64_t i0 = bb * T * D + d;                               \
                    STATE xr = LOAD(ar[i0]), xi = LOAD(ai[i0]);                \
                    hr = FMA(xr, gr, xi * gi);                                 \
                    hi = FMA(xr, gi, -(xi * gr));                              \
                }                                                              \
                if (gh0_r) gh0_r[bb * D + d] = hr;                             \
                if (gh0_i) gh0_i[bb * D + d] = hi;                             \
            }                                                                  \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

#define CFS_ARGS(ST, SS) const ST *ar, const ST *ai, const ST *br, const ST *bi, ST *out_r, ST *out_i,       \
                         SS *last_r, SS *last_i, const SS *h0_r, const SS *h0_i, const int32_t *seg,       \
                         int64_t B, int64_t T, int64_t D
#define CBS_ARGS(ST, SS) const ST *ar, const ST *ai, const ST *out_r, const ST *out_i, const ST *go_r,     \
                         const ST *go_i, const SS *h0_r, const SS *h0_i, const int32_t *seg,               \
                         const SS *gl_r, const SS *gl_i, ST *grad_ar, ST *grad_ai, ST *grad_br,            \
                         ST *grad_bi, SS *gh0_r, SS *gh0_i, int64_t B, int64_t T, int64_t D

int lro_cfwd_state_f32(CFS_ARGS(float, float)) { CPLX_STATE_FWD_BODY(float, fmaf, LRO_SAME, LRO_SAME) }
int lro_cfwd_state_bf16(CFS_ARGS(uint16_t, float)) { CPLX_STATE_FWD_BODY(float, fmaf, lro_bf16_to_f32, lro_f32_to_bf16) }
int lro_cfwd_state_f64(CFS_ARGS(double, double)) { CPLX_STATE_FWD_BODY(double, fma, LRO_SAME, LRO_SAME) }
int lro_cbwd_state_f32(CBS_ARGS(float, float)) { CPLX_STATE_BWD_BODY(float, fmaf, LRO_SAME, LRO_SAME) }
int lro_cbwd_state_bf16(CBS_ARGS(uint16_t, float)) { CPLX_STATE_BWD_BODY(float, fmaf, lro_bf16_to_f32, lro_f32_to_bf16) }
int lro_cbwd_state_f64(CBS_ARGS(double, double)) { CPLX_STATE_BWD_BODY(double, fma, LRO_SAME, LRO_SAME) }

/* ---------------------------------------------------------------------- */
/* Generated (factorized) decay.                                           */
/*                                                                         */
/* triton_training_scan.py, _samu_forward / _samu_precompute_decay: the   */
/* decay of mode d at token t is rebuilt from one value per token and one  */
/* per mode instead of being read from memory,                             */
/*   nu_d = exp(nu_log_d),  E_t = exp(eta_t),  a_{t,d} = exp(-nu_d * E_t)   */
/* (the radius part of the page's transition), and the scan is the real    */
/* one: h_t = a_t * h_{t-1} + b_t.  eta is [B,T], nu_log [D] (both in the  */
/* state precision).  Backward, for L = sum_t grad_out_t * h_t:            */
/*   g as in the plain backward; grad_b = g;                               */
/*   with grad_a_t = g_t * out_{t-1} (out_{-1} = 0) and                     */
/*   q_{t,d} = grad_a_{t,d} * a_{t,d} * (-nu_d * E_t)   (= d L / d log a),  */
/*   grad_eta[b,t] = sum_d q,   grad_nu_log[d] = sum_{b,t} q.              */
/* Every product is rounded in the state precision; the sums accumulate in  */
/* double and are rounded once.                                             */
/* ---------------------------------------------------------------------- */

#define GATED_FWD_BODY(STATE, EXP, FMA, LOAD, STORE)                           \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE nu = EXP(nu_log[d]);                                         \
            STATE h = 0;                                                       \
            for (int64_t t = 0; t < T; ++t) {                                  \
                int64_t i = (bb * T + t) * D + d;                              \
                STATE e = EXP(eta[bb * T + t]);                                \
                STATE la = -(nu * e);                                          \
                h = FMA(EXP(la), h, LOAD(b[i]));                               \
                out[i] = STORE(h);                                             \
            }                                                                  \
            if (last) last[bb * D + d] = h;                                    \
        }                                                                      \
    }                                                                          \
    return LRO_OK;

#define GATED_BWD_BODY(STATE, EXP, FMA, LOAD, STORE)                           \
    if (bad_shape(B, T, D)) return LRO_EINVAL;                                 \
    double *acc_eta = calloc((size_t)(B * T > 0 ? B * T : 1), sizeof *acc_eta); \
    double *acc_nu = calloc((size_t)(D > 0 ? D : 1), sizeof *acc_nu);          \
    if (!acc_eta || !acc_nu) { free(acc_eta); free(acc_nu); return LRO_ENOMEM; } \
    for (int64_t bb = 0; bb < B; ++bb) {                                       \
        for (int64_t d = 0; d < D; ++d) {                                      \
            STATE nu = EXP(nu_log[d]);                                         \
            STATE g = 0, a_next = 0;                                           \
            for (int64_t t = T - 1; t >= 0; --t) {                             \
                int64_t i = (bb * T + t) * D + d;                              \
                STATE e = EXP(eta[bb * T + t]);                                \
                STATE la = -(nu * e);                                          \
                STATE a = EXP(la);                                             \
                g = (t == T - 1) ? LOAD(grad_out[i])                           \
                                 : FMA(a_next, g, LOAD(grad_out[i]));          \
                STATE h_prev = (t > 0) ? LOAD(out[i - D]) : 0;                 \
                STATE grad_a = g * h_prev;                                     \
                STATE q = (grad_a * a) * la;                                   \
                grad_b[i] = STORE(g);                                          \
                acc_eta[bb * T + t] += (double)q;                              \
                acc_nu[d] += (double)q;                                        \
                a_next = a;                                                    \
            }                                                                  \
        }                                                                      \
    }                                                                          \
    for (int64_t k = 0; k < B * T; ++k) grad_eta[k] = (STATE)acc_eta[k];       \
    for (int64_t d = 0; d < D; ++d) grad_nu_log[d] = (STATE)acc_nu[d];         \
    free(acc_eta);                                                             \
    free(acc_nu);                                                              \
    return LRO_OK;

int lro_gated_fwd_f32(const float *eta, const float *nu_log, const float *b,
                      float *out, float *last, int64_t B, int64_t T, int64_t D)
{
    GATED_FWD_BODY(float, expf, fmaf, LRO_SAME, LRO_SAME)
}

int lro_gated_fwd_bf16(const float *eta, const float *nu_log, const uint16_t *b,
                       uint16_t *out, float *last, int64_t B, int64_t T, int64_t D)
{
    GATED_FWD_BODY(float, expf, fmaf, lro_bf16_to_f32, lro_f32_to_bf16)
}

int lro_gated_fwd_f64(const double *eta, const double *nu_log, const double *b,
                      double *out, double *last, int64_t B, int64_t T, int64_t D)
{
    GATED_FWD_BODY(double, exp, fma, LRO_SAME, LRO_SAME)
}

int lro_gated_bwd_f32(const float *eta, const float *nu_log, const float *out,
                      const float *grad_out, float *grad_b, float *grad_eta,
                      float *grad_nu_log, int64_t B, int64_t T, int64_t D)
{
    GATED_BWD_BODY(float, expf, fmaf, LRO_SAME, LRO_SAME)
}

int lro_gated_bwd_bf16(const float *eta, const float *nu_log, const uint16_t *out,
                       const uint16_t *grad_out, uint16_t *grad_b, float *grad_eta,
                       float *grad_nu_log, int64_t B, int64_t T, int64_t D)
{
    GATED_BWD_BODY(float, expf, fmaf, lro_bf16_to_f32, lro_f32_to_bf16)
}

int lro_gated_bwd_f64(const double *eta, const double *nu_log,
                      const double *out, const double *grad_out,
                      double *grad_b, double *grad_eta, double *grad_nu_log,
                      int64_t B, int64_t T, int64_t D)
{
    GATED_BWD_BODY(double, exp, fma, LRO_SAME, LRO_SAME)
}
