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
        const int64_t jobs = (p.N + p.rows_per_tile - 1) / p.rows_per_tile;
        const unsigned grid = (unsigned)((jobs + kWarpsPerCta - 1) / kWarpsPerCta);
        return launch_pdl(credit_td_multi_warp_kernel<kItems, VEC, TRUNC, kWarpsPerCta>, grid,
                          32 * kWarpsPerCta, 0, stream, p);
    }
    if constexpr ((VEC & kVec16) != 0) {
        if (2 * p.T > kTile && p.T <= kTile && !p.host) {
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

}  // namespace rlca
