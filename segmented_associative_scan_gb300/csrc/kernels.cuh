// Fused credit-assignment kernels: load -> build (alpha, beta, reset) -> segmented
// reverse scan -> epilogue, one HBM read of the inputs and one write of the outputs
// (Method section 2 of "rl-triton: High-Performance Triton GPU Kernels for
// Reinforcement Learning Credit Assignment").
//
// A CTA of NT threads scans a tile of NT * ITEMS steps; thread i owns ITEMS consecutive
// steps. Inside the tile: each thread composes its ITEMS pairs serially, a warp suffix
// scan (5 shuffle rounds) combines the threads of a warp, and the NT/32 warp totals are
// combined through shared memory. Each thread then replays its own items from its
// carry-in, so every A_t comes out of registers and is written once.
//
// Two tilings of the [N, T] rollout:
//   kRows     (T <= NT*ITEMS): a tile holds rows_per_tile whole rows, each padded to a
//             multiple of ITEMS. Every row ends in a reset at t = T-1, so tiles are
//             independent and no carry crosses a tile.
//   kRowLoop  (T > NT*ITEMS): one CTA per row walks the row's segs tiles from the last
//             to the first, carrying A at the first step of the later tile in registers.
//             Only one tile is on chip at a time, so long sequences never exhaust
//             registers or shared memory (the register-pressure limit the pages report
//             for Retrace at T > 2048 does not arise).
#pragma once

#include "estimators.cuh"

namespace rlca {

enum class Tiling : int { kRows = 0, kRowLoop = 1 };

template <int NT>
struct ScanSmem {
    float a[2][NT / 32];
    float b[2][NT / 32];
    int f[2][NT / 32];
};

// One tile: scan the steps this thread owns, given the tile's carry-in (A at the step
// after the tile), write the outputs and return A at the tile's first step.
template <Est E, int NT, int ITEMS, bool VEC, bool TRUNC>
__device__ __forceinline__ float scan_tile(const Params &p, int64_t row, int t0, bool active,
                                           float carry_in, ScanSmem<NT> &sm, int buf)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    Chunk<ITEMS> c;
    load_chunk<E, ITEMS, VEC, TRUNC>(p, row, t0, active, lane, c);
    Affine e[ITEMS];
    build<E, ITEMS>(p, c, e);

    // Thread aggregate: e_0 (+) e_1 (+) ... (+) e_{ITEMS-1}.
    Affine agg = e[ITEMS - 1];
#pragma unroll
    for (int j = ITEMS - 2; j >= 0; --j) agg = affine_compose(e[j], agg);

    // Warp suffix scan; the exclusive value of a lane is the inclusive one of lane+1.
    const Affine incl = warp_suffix_scan(agg, lane);
    Affine excl = shfl_down(incl, 1);
    if (lane == 31) excl = affine_identity();
    if (lane == 0) {
        sm.a[buf][warp] = incl.a;
        sm.b[buf][warp] = incl.b;
        sm.f[buf][warp] = incl.f;
    }
    __syncthreads();

    // A at the step after this warp: later warps applied to the tile carry-in.
    float x = carry_in;
#pragma unroll
    for (int w = NW - 1; w >= 0; --w)
        if (w > warp) x = affine_apply(Affine{sm.a[buf][w], sm.b[buf][w], sm.f[buf][w]}, x);
    const float a_after = affine_apply(excl, x);

    // A at the tile's first step: continue through this warp and the earlier ones.
    float tile_first = x;
#pragma unroll
    for (int w = NW - 1; w >= 0; --w)
        if (w <= warp)
            tile_first =
                affine_apply(Affine{sm.a[buf][w], sm.b[buf][w], sm.f[buf][w]}, tile_first);

    float A[ITEMS];
    A[ITEMS - 1] = affine_apply(e[ITEMS - 1], a_after);
#pragma unroll
    for (int j = ITEMS - 2; j >= 0; --j) A[j] = affine_apply(e[j], A[j + 1]);
    epilogue<E, ITEMS, VEC>(p, c, A, a_after, row, t0);
    return tile_first;
}

template <Est E, int NT, int ITEMS, bool VEC, bool TRUNC, Tiling TL>
__global__ void __launch_bounds__(NT) credit_scan_kernel(const Params p)
{
    __shared__ ScanSmem<NT> sm;
    if (TL == Tiling::kRows) {
        const int local_row = threadIdx.x / p.chunks_per_row;
        const int chunk = threadIdx.x - local_row * p.chunks_per_row;
        const int64_t row = (int64_t)blockIdx.x * p.rows_per_tile + local_row;
        const bool active = local_row < p.rows_per_tile && row < p.N;
        scan_tile<E, NT, ITEMS, VEC, TRUNC>(p, row, chunk * ITEMS, active, 0.f, sm, 0);
    } else {
        constexpr int TILE = NT * ITEMS;
        const int64_t row = blockIdx.x;
        float carry = 0.f;
        for (int s = p.segs - 1; s >= 0; --s)
            carry = scan_tile<E, NT, ITEMS, VEC, TRUNC>(p, row, s * TILE + threadIdx.x * ITEMS,
                                                        true, carry, sm, s & 1);
    }
}

}  // namespace rlca
