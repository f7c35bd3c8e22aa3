// Host-side launch of the fused kernels: picks the tiling from T and the load width
// from alignment, then launches on the caller's stream.
#pragma once

#include "kernels.cuh"

namespace rlca {

// Threads per CTA and steps per thread of the fused kernels.
constexpr int kThreads = 128;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;

struct LaunchShape {
    Tiling tiling;
    unsigned grid;
    int rows_per_tile;
    int chunks_per_row;
    int segs;
};

// Look-back tiles of an [N, T] problem (0 when T fits one tile: no look-back needed).
inline int64_t lookback_tiles(int64_t N, int64_t T)
{
    return T > kTile ? N * ((T + kTile - 1) / kTile) : 0;
}

inline size_t workspace_bytes(int64_t N, int64_t T)
{
    const int64_t tiles = lookback_tiles(N, T);
    return tiles ? (size_t)(kWsHeaderBytes + tiles * kTileStateBytes) : 0;
}

// Bounded wait of the look-back: consecutive empty polls of a later tile (each poll
// sleeps up to 256 ns, so about a second) before the launch reports RLCA_ERR_TIMEOUT.
constexpr int kDefaultSpinLimit = 1 << 22;

inline LaunchShape plan_launch(int64_t N, int T, bool lookback)
{
    LaunchShape s{};
    if (T <= kTile) {
        const int t_pad = (T + kItems - 1) / kItems * kItems;
        s.tiling = Tiling::kRows;
        s.chunks_per_row = t_pad / kItems;
        s.rows_per_tile = kTile / t_pad;
        s.segs = 1;
        s.grid = (unsigned)((N + s.rows_per_tile - 1) / s.rows_per_tile);
    } else {
        s.chunks_per_row = kTile / kItems;
        s.rows_per_tile = 1;
        s.segs = (T + kTile - 1) / kTile;
        s.tiling = lookback ? Tiling::kLookback : Tiling::kRowLoop;
        s.grid = (unsigned)(lookback ? N * s.segs : N);
    }
    return s;
}

template <Est E, bool VEC, bool TRUNC>
cudaError_t launch_variant(Params p, const LaunchShape &s, cudaStream_t stream)
{
    p.rows_per_tile = s.rows_per_tile;
    p.chunks_per_row = s.chunks_per_row;
    p.segs = s.segs;
    if (s.tiling == Tiling::kRows)
        credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kRows>
            <<<s.grid, kThreads, 0, stream>>>(p);
    else if (s.tiling == Tiling::kRowLoop)
        credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kRowLoop>
            <<<s.grid, kThreads, 0, stream>>>(p);
    else
        credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kLookback>
            <<<s.grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// Launch one estimator. With p.ws set (and T longer than a tile) the tiles of a row run
// in parallel with decoupled look-back; otherwise a CTA walks each long row.
template <Est E>
cudaError_t launch_estimator(const Params &p, bool vec, cudaStream_t stream)
{
    const LaunchShape s = plan_launch(p.N, p.T, p.ws != nullptr);
    const bool trunc = p.trunc != nullptr;
    if (vec)
        return trunc ? launch_variant<E, true, true>(p, s, stream)
                     : launch_variant<E, true, false>(p, s, stream);
    return trunc ? launch_variant<E, false, true>(p, s, stream)
                 : launch_variant<E, false, false>(p, s, stream);
}

// One definition per estimator, each in its own translation unit.
cudaError_t launch_return(const Params &p, bool vec, cudaStream_t stream);
cudaError_t launch_td_lambda(const Params &p, bool vec, cudaStream_t stream);
cudaError_t launch_gae(const Params &p, bool vec, cudaStream_t stream);
cudaError_t launch_vtrace(const Params &p, bool vec, cudaStream_t stream);
cudaError_t launch_retrace(const Params &p, bool vec, cudaStream_t stream);

}  // namespace rlca
