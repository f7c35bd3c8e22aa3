// Host-side launch of the fused kernels: picks the tiling from T and the load width
// from alignment, then launches on the caller's stream.
#pragma once

#include "kernels.cuh"

namespace rlca {

// Threads per CTA and steps per thread of the fused kernels.
constexpr int kThreads = 256;
constexpr int kItems = 4;
constexpr int kTile = kThreads * kItems;

struct LaunchShape {
    Tiling tiling;
    unsigned grid;
    int rows_per_tile;
    int chunks_per_row;
    int segs;
};

inline LaunchShape plan_launch(int64_t N, int T)
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
        s.tiling = Tiling::kRowLoop;
        s.chunks_per_row = kTile / kItems;
        s.rows_per_tile = 1;
        s.segs = (T + kTile - 1) / kTile;
        s.grid = (unsigned)N;
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
    else
        credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kRowLoop>
            <<<s.grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <Est E>
cudaError_t launch_estimator(const Params &p, bool vec, cudaStream_t stream)
{
    const LaunchShape s = plan_launch(p.N, p.T);
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
