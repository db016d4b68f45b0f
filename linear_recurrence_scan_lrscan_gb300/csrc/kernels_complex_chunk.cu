// Launchers of the three-phase chunked complex scan.
#include "complex_chunk_kernels.cuh"

namespace lrscan {

namespace {

CMaps maps_of(float *const (&p)[4]) { return CMaps{p[0], p[1], p[2], p[3]}; }

// Phase 2: the flat warp-per-lane prefix, or the grouped form (group maps,
// their prefix, the per-group rescan) when the launch carries group maps.
template <bool REVERSE>
void cprefix_phase(const CChunkLaunch &L, const ChunkGeom &g, const float *init_r, const float *init_i) {
    const long long lanes = static_cast<long long>(L.B) * L.D;
    const CMaps m = maps_of(L.maps);
    const unsigned pb = static_cast<unsigned>((lanes * 32 + 255) / 256);
    if (L.gmaps[0] == nullptr) {
        cchunk_prefix<REVERSE><<<pb, 256, 0, L.stream>>>(m, g.Nc, g.D, lanes, init_r, init_i);
        return;
    }
    const CMaps gm = maps_of(L.gmaps);
    const int NG = (g.Nc + kGroupChunks - 1) / kGroupChunks;
    const unsigned gb = static_cast<unsigned>((lanes * NG * 32 + 255) / 256);
    cchunk_group_reduce<REVERSE><<<gb, 256, 0, L.stream>>>(m, gm, g.Nc, g.D, kGroupChunks, NG, lanes);
    cchunk_prefix<REVERSE><<<pb, 256, 0, L.stream>>>(gm, NG, g.D, lanes, init_r, init_i);
    cchunk_group_rescan<REVERSE><<<gb, 256, 0, L.stream>>>(m, gm, g.Nc, g.D, kGroupChunks, NG, lanes);
}

template <typename St, int V, bool EXT>
int cfwd_t(const CChunkLaunch &L) {
    const ChunkGeom g = make_chunk_geom(L.T, L.D, L.chunk, V);
    const unsigned nb = chunk_blocks(g, L.B);
    const St *in[4];
    for (int i = 0; i < 4; ++i) in[i] = static_cast<const St *>(L.in[i]);
    cchunk_summary_fwd<St, V, EXT><<<nb, 128, 0, L.stream>>>(in[0], in[1], in[2], in[3], maps_of(L.maps), g, L.chunk, L.sx);
    cprefix_phase<false>(L, g, L.sx.h0_r, L.sx.h0_i);
    cchunk_replay_fwd<St, V, EXT><<<nb, 128, 0, L.stream>>>(in[0], in[1], in[2], in[3], maps_of(L.maps),
                                                    static_cast<St *>(L.out[0]), static_cast<St *>(L.out[1]),
                                                    L.last_r, L.last_i, g, L.chunk, L.sx);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <typename St, int V, bool EXT>
int cbwd_t(const CChunkLaunch &L) {
    const ChunkGeom g = make_chunk_geom(L.T, L.D, L.chunk, V);
    const unsigned nb = chunk_blocks(g, L.B);
    const St *in[6];
    for (int i = 0; i < 6; ++i) in[i] = static_cast<const St *>(L.in[i]);
    cchunk_summary_bwd<St, V, EXT><<<nb, 128, 0, L.stream>>>(in[0], in[1], in[4], in[5], maps_of(L.maps), g, L.chunk, L.sx);
    cprefix_phase<true>(L, g, L.sx.gl_r, L.sx.gl_i);
    cchunk_replay_bwd<St, V, EXT><<<nb, 128, 0, L.stream>>>(in[0], in[1], in[2], in[3], in[4], in[5], maps_of(L.maps),
                                                    static_cast<St *>(L.out[0]), static_cast<St *>(L.out[1]),
                                                    static_cast<St *>(L.out[2]), static_cast<St *>(L.out[3]), g,
                                                    L.chunk, L.sx);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

namespace {

bool has_state(const CStateArgs &sx) {
    return sx.h0_r || sx.h0_i || sx.seg || sx.gl_r || sx.gl_i || sx.gh0_r || sx.gh0_i;
}

template <bool EXT>
int cfwd_any(const CChunkLaunch &L, int dtype) {
    if (L.vec == 4) return dtype == 0 ? cfwd_t<float, 4, EXT>(L) : cfwd_t<bf16_t, 4, EXT>(L);
    return dtype == 0 ? cfwd_t<float, 1, EXT>(L) : cfwd_t<bf16_t, 1, EXT>(L);
}

template <bool EXT>
int cbwd_any(const CChunkLaunch &L, int dtype) {
    if (L.vec == 4) return dtype == 0 ? cbwd_t<float, 4, EXT>(L) : cbwd_t<bf16_t, 4, EXT>(L);
    return dtype == 0 ? cbwd_t<float, 1, EXT>(L) : cbwd_t<bf16_t, 1, EXT>(L);
}

}  // namespace

int cchunk_fwd_launch(const CChunkLaunch &L, int dtype) {
    return has_state(L.sx) ? cfwd_any<true>(L, dtype) : cfwd_any<false>(L, dtype);
}

int cchunk_bwd_launch(const CChunkLaunch &L, int dtype) {
    return has_state(L.sx) ? cbwd_any<true>(L, dtype) : cbwd_any<false>(L, dtype);
}

}  // namespace lrscan
