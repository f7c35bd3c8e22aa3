// Kernels of one estimator (instantiated in a translation unit of its own so the
// library builds in parallel).
#include "launch.cuh"

namespace rlca {
cudaError_t launch_td_lambda(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator<Est::kTdLambda>(p, vec, stream);
}

cudaError_t launch_td_lambda_bf16(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator_bf16<Est::kTdLambda>(p, vec, stream);
}
// Fused TD(lambda) for several lambdas: whole-row CTA tiles, or the row loop.
template <int VEC, bool TRUNC>
cudaError_t launch_td_multi_variant(Params p, cudaStream_t stream)
{
    constexpr int CH = 32 * kItems;
    if (p.T <= CH) {  // warp-owned rows: whole rows per warp, no CTA barrier
        const int t_pad = (p.T + kItems - 1) / kItems * kItems;
        p.chunks_per_row = t_pad / kItems;
        p.rows_per_tile = CH / t_pad;
        p.segs = 1;
        const int64_t jobs = (p.N + p.rows_per_tile - 1) / p.rows_per_tile;
        const unsigned grid = (unsigned)((jobs + kWarpsPerCta - 1) / kWarpsPerCta);
        return launch_pdl(credit_td_multi_warp_kernel<kItems, VEC, TRUNC, kWarpsPerCta>, grid,
                          32 * kWarpsPerCta, 0, stream, p);
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

}  // namespace rlca
