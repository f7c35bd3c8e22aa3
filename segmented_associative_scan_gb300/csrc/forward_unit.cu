// Forward scans (eligibility traces, episodic prefix sums), walked from the first step
// to the last, in one input format: compiled once per format with RLCA_UNIT_FMT (the Fmt
// value) set by the build.
#include "forward.cuh"
#include "launch.cuh"

#if !defined(RLCA_UNIT_FMT)
#error "forward_unit.cu is compiled with -DRLCA_UNIT_FMT=<0..2>"
#endif

namespace rlca {

// Pipelined forward warp rows: chunks in flight in registers (1 or 2), L2 prefetch
// before the wait (steps) and ahead of the walk (chunks), and the rows they take
// (pipe_from < T <= 1024, device memory, 16-byte aligned rows). Measured on GB300 at
// [4096, 1024], eligibility trace / prefix sum, us per launch: CTA tiles with the
// prefetch 8.19 / 8.40; one chunk in flight, 256 steps before the wait 8.44 / 8.45;
// two chunks, 256 steps 7.59 / 7.65 (bf16 7.73 / 7.73, fp16 7.66 / 7.67); two chunks,
// 1024 steps 7.66 / 7.55 (bf16 7.47 / 7.57, fp16 7.87 / 7.89); three chunks (fp32 1024
// steps, bf16 1024, fp16 256): fp32 8.08 / 8.07, bf16 7.06 / 7.07 against 7.29 / 7.29
// with two, fp16 7.36 / 7.36 against 7.61 / 7.62 (fp32 58-64 registers, one wave still).
// fp16 now prefetches 1024 steps as bf16 does: 7.39 -> 7.15 us at [4096, 1024] (7.02 vs
// 6.91 at [4096, 600]).
// fp32 rows take three chunks too, under a 7-CTA cap (68 registers), where the grid
// fills most of one wave of warps at that cap (4.5 to 7 CTAs per SM). Eligibility
// trace, us per launch, two chunks uncapped -> three capped: [N, 1024] for N = 2200
// 5.54 -> 5.54, 2432 5.80 -> 5.80, 2440 5.81 -> 6.57, 2600 5.96 -> 6.71, 2800 7.09 ->
// 6.79, 3000 7.19 -> 6.85, 3200 7.24 -> 6.94, 3600 7.28 -> 7.16, 4000 7.47 -> 7.28,
// 4096 7.57 -> 7.32, 4256 7.66 -> 7.46, 8192 13.62 -> 14.34 (two waves); [4096, 600]
// 7.07 -> 6.30. Each form steps up where its CTAs per SM pass 4 (three chunks) or about
// 4.4 (two).
struct ForwardPipe {
    int depth, first, ahead, pipe_from;
};

template <typename TIn>
constexpr ForwardPipe forward_pipe()
{
    if (std::is_same<TIn, uint16_t>::value) return {3, 1024, 0, 256};  // bf16
    if (std::is_same<TIn, __half>::value) return {3, 1024, 0, 256};
    return {2, 256, 0, 256};
}

// Rows of at most one warp chunk (256 steps): warp-owned rows. Longer rows up to one CTA
// tile in device memory with 16-byte aligned rows: a warp per row with its next chunk's
// loads in flight. Otherwise CTA tiles of 1024 steps (whole rows, or a row walked tile by
// tile), which load a whole tile at once.
template <int VEC, bool TRUNC, typename TIn = float>
cudaError_t launch_forward_variant(Params p, cudaStream_t stream)
{
    constexpr int CH = 32 * kItems;
    if constexpr ((VEC & kVec16) != 0) {
        constexpr ForwardPipe fp = forward_pipe<TIn>();
        if (p.T > fp.pipe_from && p.T <= kTile && !p.host) {
            p.segs = (p.T + CH - 1) / CH;
            p.chunks_per_row = CH / kItems;
            p.rows_per_tile = 1;
            p.pf_first = fp.first;
            p.pf_ahead = fp.ahead;
            const unsigned grid = (unsigned)((p.N + kWarpsPerCta - 1) / kWarpsPerCta);
            if constexpr (sizeof(TIn) == 4) {
                constexpr int kCap = 7;  // CTAs of 4 warps per SM: 72 registers
                const int64_t sms = sm_count();
                if (2 * (int64_t)grid >= 9 * sms && (int64_t)grid <= kCap * sms)
                    return launch_pdl(credit_forward_pipe_kernel<kItems, kVec16, TRUNC, 3,
                                                                 kWarpsPerCta, TIn, kCap>,
                                      grid, 32 * kWarpsPerCta, 0, stream, p);
            }
            return launch_pdl(
                credit_forward_pipe_kernel<kItems, kVec16, TRUNC, fp.depth, kWarpsPerCta, TIn>,
                grid, 32 * kWarpsPerCta, 0, stream, p);
        }
    }
    if (p.T <= CH) {
        const int t_pad = (p.T + kItems - 1) / kItems * kItems;
        p.segs = 1;
        p.chunks_per_row = t_pad / kItems;
        p.rows_per_tile = CH / t_pad;
        set_lane_split(p);
        const int64_t jobs = (p.N + p.rows_per_tile - 1) / p.rows_per_tile;
        const unsigned grid = (unsigned)((jobs + kWarpRowsPerCta - 1) / kWarpRowsPerCta);
        return launch_pdl(credit_forward_kernel<kItems, VEC, TRUNC, kWarpRowsPerCta, TIn>,
                          grid, 32 * kWarpRowsPerCta, 0, stream, p);
    }
    if (p.T <= kTile) {
        const int t_pad = (p.T + kItems - 1) / kItems * kItems;
        p.segs = 1;
        p.chunks_per_row = t_pad / kItems;
        p.rows_per_tile = kTile / t_pad;
        const unsigned grid = (unsigned)((p.N + p.rows_per_tile - 1) / p.rows_per_tile);
        if (p.rows_per_tile == 1)
            return launch_pdl(
                credit_forward_tile_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRow, TIn>,
                grid, kThreads, 0, stream, p);
        return launch_pdl(
            credit_forward_tile_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRows, TIn>, grid,
            kThreads, 0, stream, p);
    }
    p.segs = (p.T + kTile - 1) / kTile;
    p.chunks_per_row = kTile / kItems;
    p.rows_per_tile = 1;
    return launch_pdl(
        credit_forward_tile_kernel<kThreads, kItems, VEC, TRUNC, Tiling::kRowLoop, TIn>,
        (unsigned)p.N, kThreads, 0, stream, p);
}

template <Fmt F>
cudaError_t launch_forward_unit(const Params &p_in, int vec, cudaStream_t stream)
{
    using TIn = typename FmtType<F>::type;
    Params p = p_in;
    // decay^kItems in the kernel's multiply order, for the per-lane composite.
    p.beta_pow = p.gamma;
    for (int i = 1; i < kItems; ++i) p.beta_pow = p.gamma * p.beta_pow;
    const bool trunc = p.trunc != nullptr;
    // 128-bit access where a CTA tile holds one row (measured faster there, 8.46 vs
    // 8.53 us at [4096, 1024]); 256-bit elsewhere when the rows allow it.
    if (one_row_per_cta(p.T) && !p.host) vec = vec < 1 ? vec : 1;
    return with_vec_trunc(vec, trunc, [&](auto v, auto r) {
        return launch_forward_variant<decltype(v)::value, decltype(r)::value, TIn>(p, stream);
    });
}

template cudaError_t launch_forward_unit<static_cast<Fmt>(RLCA_UNIT_FMT)>(const Params &, int,
                                                                       cudaStream_t);

}  // namespace rlca
