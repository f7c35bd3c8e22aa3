// Kernels of one estimator (instantiated in a translation unit of its own so the
// library builds in parallel).
#include "launch.cuh"

namespace rlca {
cudaError_t launch_vtrace(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator<Est::kVtrace>(p, vec, stream);
}

cudaError_t launch_vtrace_bf16(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator_bf16<Est::kVtrace>(p, vec, stream);
}

// Fused GAE + V-trace: CTA tiles (whole rows, one row per CTA, or the row loop). The
// whole-row tiles need 76-87 registers (5-6 CTAs per SM); capped at 6 per SM (no spills)
// the one-row tile ran 4% faster at [4096, 1024] (17.9 vs 18.7 us).
constexpr int kPairMinBlocks = 6;

template <int VEC, bool TRUNC>
cudaError_t launch_gae_vtrace_variant(Params pg, Params pv, cudaStream_t stream)
{
    unsigned grid;
    constexpr int CH = 32 * kItems;
    if (pv.T <= CH) {  // warp-owned rows, capped at 6 CTAs per SM like the tiles
        const int t_pad = (pv.T + kItems - 1) / kItems * kItems;
        pv.chunks_per_row = t_pad / kItems;
        pv.rows_per_tile = CH / t_pad;
        pv.segs = 1;
        const int64_t jobs = (pv.N + pv.rows_per_tile - 1) / pv.rows_per_tile;
        grid = (unsigned)((jobs + kWarpsPerCta - 1) / kWarpsPerCta);
        return launch_pdl(credit_gae_vtrace_warp_kernel<kItems, VEC, TRUNC, kWarpsPerCta,
                                                        kPairMinBlocks>,
                          grid, 32 * kWarpsPerCta, 0, stream, pg, pv);
    }
    if (pv.T <= kTile) {
        const int t_pad = (pv.T + kItems - 1) / kItems * kItems;
        pv.chunks_per_row = t_pad / kItems;
        pv.rows_per_tile = kTile / t_pad;
        pv.segs = 1;
        grid = (unsigned)((pv.N + pv.rows_per_tile - 1) / pv.rows_per_tile);
        if (pv.rows_per_tile == 1)
            return launch_pdl(credit_gae_vtrace_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRow,
                                                       kPairMinBlocks>,
                              grid, kThreads, 0, stream, pg, pv);
        return launch_pdl(credit_gae_vtrace_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRows,
                                                   kPairMinBlocks>,
                          grid, kThreads, 0, stream, pg, pv);
    }
    pv.chunks_per_row = kTile / kItems;
    pv.rows_per_tile = 1;
    pv.segs = (pv.T + kTile - 1) / kTile;
    return launch_pdl(credit_gae_vtrace_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRowLoop>,
                      (unsigned)pv.N, kThreads, 0, stream, pg, pv);
}

cudaError_t launch_gae_vtrace(const Params &pg_in, const Params &pv, int vec,
                              cudaStream_t stream)
{
    Params pg = pg_in;
    set_beta_pow<Est::kGae>(pg);
    return with_vec_trunc(vec, pv.trunc != nullptr, [&](auto v, auto r) {
        return launch_gae_vtrace_variant<decltype(v)::value, decltype(r)::value>(pg, pv,
                                                                                 stream);
    });
}
}  // namespace rlca
