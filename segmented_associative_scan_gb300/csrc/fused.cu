// The fused calls, fp32 inputs: TD(lambda) for several lambdas from one read of the
// inputs, and GAE with V-trace from one read (Method section 2: the load is what costs).
#include "launch.cuh"

namespace rlca {

// Fused TD(lambda) on pipelined warp rows: CTAs per SM the register allocator must fit.
// Measured on GB300 at [4096, 1024], lambda in {0, 0.9, 1}: 15.58 us capped at 7 per SM,
// 17.16 uncapped (72 registers either way), 15.93 with 256-bit access, 18.76 with two
// chunks in flight (95 registers), against 17.30 for one row per CTA.
constexpr int kMultiPipeMinBlocks = 7;

// Fused TD(lambda) for several lambdas: warp-owned rows up to one warp chunk, pipelined
// warp rows for rows of 513-1024 steps in device memory with 16-byte aligned rows,
// whole-row CTA tiles otherwise, and the row loop beyond 1024 steps.
template <int VEC, bool TRUNC>
cudaError_t launch_td_multi_variant(Params p, cudaStream_t stream)
{
    constexpr int CH = 32 * kItems;
    if (p.T <= CH) {  // warp-owned rows: whole rows per warp, no CTA barrier
        const int t_pad = (p.T + kItems - 1) / kItems * kItems;
        p.chunks_per_row = t_pad / kItems;
        p.rows_per_tile = CH / t_pad;
        p.segs = 1;
        set_lane_split(p);
        const int64_t jobs = (p.N + p.rows_per_tile - 1) / p.rows_per_tile;
        const unsigned grid = (unsigned)((jobs + kWarpRowsPerCta - 1) / kWarpRowsPerCta);
        return launch_pdl(credit_td_multi_warp_kernel<kItems, VEC, TRUNC, kWarpRowsPerCta>,
                          grid, 32 * kWarpRowsPerCta, 0, stream, p);
    }
    if constexpr ((VEC & kVec16) != 0) {
        if (2 * p.T > kTile && p.T <= kTile && !p.host) {
            set_pipe_prefetch<Est::kTdLambda, float, true>(p);
            p.segs = (p.T + CH - 1) / CH;
            p.chunks_per_row = CH / kItems;
            p.rows_per_tile = 1;
            const unsigned grid = (unsigned)((p.N + kWarpsPerCta - 1) / kWarpsPerCta);
            return launch_pdl(credit_td_multi_pipe_kernel<kItems, kVec16, TRUNC, 1, kWarpsPerCta,
                                                          kMultiPipeMinBlocks>,
                              grid, 32 * kWarpsPerCta, 0, stream, p);
        }
    }
    if (p.T <= kTile) {
        const int t_pad = (p.T + kItems - 1) / kItems * kItems;
        p.chunks_per_row = t_pad / kItems;
        p.rows_per_tile = kTile / t_pad;
        p.segs = 1;
        const unsigned grid = (unsigned)((p.N + p.rows_per_tile - 1) / p.rows_per_tile);
        if (p.rows_per_tile == 1)
            return launch_pdl(credit_td_multi_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRow>,
                              grid, kThreads, 0, stream, p);
        return launch_pdl(credit_td_multi_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRows>,
                          grid, kThreads, 0, stream, p);
    }
    p.chunks_per_row = kTile / kItems;
    p.rows_per_tile = 1;
    p.segs = (p.T + kTile - 1) / kTile;
    return launch_pdl(credit_td_multi_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRowLoop>,
                      (unsigned)p.N, kThreads, 0, stream, p);
}

cudaError_t launch_td_multi(const Params &p_in, int vec, cudaStream_t stream)
{
    Params p = p_in;
    for (int k = 0; k < p.multi.count; ++k) {
        const float beta = p.multi.gamma_lambda[k];
        float pw = beta;
        for (int i = 1; i < kItems; ++i) pw = beta * pw;
        p.multi.beta_pow[k] = pw;
    }
    const bool trunc = p.trunc != nullptr;
    return with_vec_trunc(vec, trunc, [&](auto v, auto r) {
        return launch_td_multi_variant<decltype(v)::value, decltype(r)::value>(p, stream);
    });
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
        set_lane_split(pv);
        const int64_t jobs = (pv.N + pv.rows_per_tile - 1) / pv.rows_per_tile;
        grid = (unsigned)((jobs + kWarpRowsPerCta - 1) / kWarpRowsPerCta);
        return launch_pdl(credit_gae_vtrace_warp_kernel<kItems, VEC, TRUNC, kWarpRowsPerCta,
                                                        kPairMinBlocks * 4 / kWarpRowsPerCta>,
                          grid, 32 * kWarpRowsPerCta, 0, stream, pg, pv);
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
