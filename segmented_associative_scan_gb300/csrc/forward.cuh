// Forward-time scans: eligibility traces and episodic prefix sums.
//
// Method section 1 of "rl-triton: High-Performance Triton GPU Kernels for Reinforcement
// Learning Credit Assignment" lists eligibility traces (the forward-time mirror of the
// recurrence) and episodic prefix sums among the estimators. Both are
//   A_t = x_t + decay * A_{t-1}   inside an episode,   A_t = x_t   right after one ends,
// with A_{-1} = init[n] carried into the window (the forward counterpart of the window-end
// bootstrap of Method section 3); prefix sums have decay = 1. The same operator composes
// them, applied in the other time order: a warp prefix scan (shfl_up) instead of a
// suffix scan, chunks walked from the first to the last.
//
// Two layouts, as for the reverse scans: warp-owned rows for rows of at most one warp
// chunk (several short rows per warp, each row's first step resetting and folding in
// init; no CTA barrier, no shared memory), and CTA tiles of 1024 steps for longer rows
// (whole rows per tile, or a row walked tile by tile with the carry in registers).
// decay >= 0 (checked on the host), so the reset marker of the scan is exact.
#pragma once

#include "kernels.cuh"

namespace rlca {

// One loaded chunk of a warp: x (ITEMS steps per lane, zero past the row's end), `ended`
// (bit j: step t0+j terminated or truncated) and `valid` (bit j: step t0+j exists). A at
// the step before the chunk is `carry_in`; `prev_ended` says whether the step before
// lane 0's first step ended an episode; `init` is init[row] for the thread holding the
// row's first step (load_init, read with the chunk's data). Returns A at the chunk's last
// step; *last_ended gets whether that step ended an episode. Every lane of the warp calls
// this. EARLY_INIT false: `init` is ignored and init[row] is read here, after the chunk.
template <int ITEMS, int VEC, typename TIn = float, bool EARLY_INIT = true>
__device__ __forceinline__ float forward_chunk_scan(const Params &p, int64_t row, int t0,
                                                    bool active, float (&x)[ITEMS],
                                                    unsigned ended, unsigned valid,
                                                    float carry_in, bool prev_ended,
                                                    float init, bool *last_ended)
{
    const int lane = threadIdx.x & 31;
    const int64_t off = active ? row * p.ld : 0;

    // Item j starts afresh when step t0+j-1 ended an episode; the row's first step resets
    // too and takes the carried-in value as its own term.
    const unsigned prev_lane = __shfl_up_sync(kFullMask, ended >> (ITEMS - 1), 1) & 1u;
    const unsigned before = lane == 0 ? (prev_ended ? 1u : 0u) : prev_lane;
    unsigned reset = ((ended << 1) | before) | ~valid;
    if (t0 == 0 && active) {
        reset |= 1u;
        if (p.boot) x[0] = fmaf(p.gamma, EARLY_INIT ? init : __ldg(p.boot + row), x[0]);
    }
    reset &= all_items<ITEMS>();

    // Composite of the lane's items in time order, e_{ITEMS-1} o ... o e_0.
    const float decay = p.gamma;
    float a = x[0];
#pragma unroll
    for (int j = 1; j < ITEMS; ++j) a = ((reset >> j) & 1u) ? x[j] : fmaf(decay, a, x[j]);
    const Affine agg{a, reset ? kResetB : p.beta_pow};

    // Inclusive prefix scan over lanes: lane i gets agg_i o ... o agg_0.
    Affine incl = agg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Affine y{__shfl_up_sync(kFullMask, incl.a, d), __shfl_up_sync(kFullMask, incl.b, d)};
        if (lane >= d) incl = affine_compose(incl, y);
    }
    Affine excl{__shfl_up_sync(kFullMask, incl.a, 1), __shfl_up_sync(kFullMask, incl.b, 1)};
    if (lane == 0) excl = affine_identity();
    const Affine whole = shfl_idx(incl, 31);

    float A[ITEMS];
    float prev = affine_apply(excl, carry_in);
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        prev = ((reset >> j) & 1u) ? x[j] : fmaf(decay, prev, x[j]);
        A[j] = prev;
    }
    if (valid) store_items<ITEMS, VEC>(p.out0 + off, t0, valid, A);
    *last_ended = (__shfl_sync(kFullMask, ended, 31) >> (ITEMS - 1)) & 1u;
    return affine_apply(whole, carry_in);
}

// init[row], the value carried into the window, for the thread holding the row's first
// step (else 0). Its address needs no loaded data, so it is read together with the
// chunk's data rather than after the chunk's flags arrive.
__device__ __forceinline__ float load_init(const Params &p, int64_t row, int t0, bool active)
{
    return (active && t0 == 0 && p.boot) ? __ldg(p.boot + row) : 0.f;
}

// The same, loading the chunk first (ragged and inactive chunks allowed).
template <int ITEMS, int VEC, bool TRUNC, typename TIn = float>
__device__ __forceinline__ float forward_chunk(const Params &p, int64_t row, int t0, bool active,
                                               float carry_in, bool prev_ended,
                                               bool *last_ended)
{
    const int T = p.T;
    const int Te = active ? T : 0;
    const int64_t off = active ? row * p.ld : 0;
    const float init = load_init(p, row, t0, active);
    float x[ITEMS];
    load_items<ITEMS, VEC, TIn>(in_row<TIn>(p.reward, off), t0, Te, x);
    const unsigned ended = TRUNC ? load_flag_bits_or<ITEMS, VEC>(p.term + off, p.trunc + off, t0, Te)
                                 : load_flag_bits<ITEMS, VEC>(p.term + off, t0, Te);
    const unsigned valid = valid_items<ITEMS>(t0, Te);
#pragma unroll
    for (int j = 0; j < ITEMS; ++j)
        if (!((valid >> j) & 1u)) x[j] = 0.f;
    return forward_chunk_scan<ITEMS, VEC, TIn>(p, row, t0, active, x, ended, valid, carry_in,
                                               prev_ended, init, last_ended);
}

template <int ITEMS, int VEC, bool TRUNC, int WARPS = 4, typename TIn = float>
__global__ void __launch_bounds__(32 * WARPS) credit_forward_kernel(const Params p)
{
    constexpr int CH = 32 * ITEMS;
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    const LaneSlot ls = lane_slot(p, lane);  // index math before the wait: no memory read
    const int64_t row = job * p.rows_per_tile + ls.local_row;
    const bool active = ls.local_row < p.rows_per_tile && row < p.N;
    // x and the flags are what the discounted return streams in, too.
    if (p.segs == 1) {
        prefetch_warp_rows<Est::kReturn, TRUNC, TIn>(p, job, p.T);
    } else if (lane == 0) {
        prefetch_row<Est::kReturn, TRUNC, TIn>(p, job, 0, p.T < 1024 ? p.T : 1024);
    }
    grid_dependency_sync();
    bool last_ended = false;
    if (p.segs == 1) {
        forward_chunk<ITEMS, VEC, TRUNC, TIn>(p, row, ls.chunk * ITEMS, active, 0.f, false,
                                              &last_ended);
    } else {
        if (job >= p.N) return;  // the whole warp leaves together
        float carry = 0.f;
        for (int s = 0; s < p.segs; ++s)
            carry = forward_chunk<ITEMS, VEC, TRUNC, TIn>(p, job, s * CH + lane * ITEMS, true,
                                                          carry, last_ended, &last_ended);
    }
}

// ------------------------------------------------------- pipelined warp rows, forward

// One row per warp, walked in chunks of 32 * ITEMS steps from the first to the last
// with the next chunks' loads in flight: before a chunk is scanned, the raw words of the
// DEPTH chunks after it have been requested into registers, so the warp's HBM reads
// overlap its own scans and stores (the forward mirror of warp_pipe_row). L2 prefetch:
// the first pf_first steps before the grid dependency wait, and at chunk s the chunk
// s + pf_ahead (0: none). Full chunks go through the pipeline; a ragged last chunk is
// loaded plainly at the end. Needs 16-byte aligned rows (VEC >= 1).
template <int ITEMS, int VEC, bool TRUNC, int DEPTH, int WARPS = 4, typename TIn = float,
          int MINB = 0>
__global__ void __launch_bounds__(32 * WARPS, MINB) credit_forward_pipe_kernel(const Params p)
{
    static_assert(DEPTH >= 1 && DEPTH <= 3, "one to three chunks in flight");
    static_assert(VEC & kVec16, "raw chunks are read with vector loads");
    constexpr Est E = Est::kReturn;  // streams x (as reward) and the flags, nothing else
    constexpr int CH = 32 * ITEMS;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (lane == 0) prefetch_row<E, TRUNC, TIn>(p, row, 0, p.T < p.pf_first ? p.T : p.pf_first);
    grid_dependency_sync();
    if (row >= p.N) return;  // the whole warp leaves together
    const int64_t off = row * p.ld;
    const int full = p.T / CH;
    float carry = 0.f;
    bool ended_before = false;
    // w[d] holds chunk s + d (registers: every index below is a compile-time constant).
    RawChunk<E, ITEMS, TIn> w[DEPTH];
#pragma unroll
    for (int d = 0; d < DEPTH; ++d)
        if (d < full) load_raw<E, ITEMS, VEC, TRUNC>(p, off, d * CH + lane * ITEMS, lane, w[d]);
    // init[row] is read after chunk 0 arrives: reading it with chunk 0's raw words (and
    // peeling chunk 0's step off the loop) measured 1.6% slower for fp32 at [4096, 1024]
    // and within the spread between GPUs for 16-bit inputs.
    auto step = [&](int k) {
        const int t0 = k * CH + lane * ITEMS;
        if (lane == 0 && p.pf_ahead > 0 && (k + p.pf_ahead) * CH < p.T) {
            const int lo = (k + p.pf_ahead) * CH;
            prefetch_row<E, TRUNC, TIn>(p, row, lo, lo + CH < p.T ? lo + CH : p.T);
        }
        float x[ITEMS];
        widen_words<TIn>(w[0].r, x);
        unsigned ended = 0;
#pragma unroll
        for (int k = 0; k < ITEMS / 4; ++k)
            ended |= nonzero_bytes(TRUNC ? (w[0].term[k] | w[0].trunc[k]) : w[0].term[k])
                     << (4 * k);
#pragma unroll
        for (int d = 0; d + 1 < DEPTH; ++d) w[d] = w[d + 1];
        if (k + DEPTH < full)
            load_raw<E, ITEMS, VEC, TRUNC>(p, off, (k + DEPTH) * CH + lane * ITEMS, lane,
                                           w[DEPTH - 1]);
        carry = forward_chunk_scan<ITEMS, VEC, TIn, false>(p, row, t0, true, x, ended,
                                                           all_items<ITEMS>(), carry,
                                                           ended_before, 0.f, &ended_before);
    };
    for (int s = 0; s < full; ++s) step(s);
    if (full * CH < p.T)
        forward_chunk<ITEMS, VEC, TRUNC, TIn>(p, row, full * CH + lane * ITEMS, true, carry,
                                              ended_before, &ended_before);
}

// ------------------------------------------------------------------ CTA tiles

// One tile of NT * ITEMS steps scanned forward by a CTA: lane composites, warp prefix
// scans, the NT/32 warp totals combined through shared memory. `carry_in` is A at the
// step before the tile and `prev_ended` whether that step ended an episode; returns A at
// the tile's last step and sets *last_ended.
//
// A warp's first step starts afresh when the step before it ended an episode. That flag
// belongs to the previous warp, so the warp scans as if it did not, and the flag is
// applied after the exchange instead: the warp's carry-in becomes 0 (its first step then
// equals x exactly) and its total is marked as a reset for the warps after it.
// EARLY_INIT: init[row] is read with the tile's data (load_init), else after it.
template <int NT, int ITEMS, int VEC, bool TRUNC, typename TIn = float, bool EARLY_INIT = true>
__device__ __forceinline__ float forward_tile(const Params &p, int64_t row, int t0, bool active,
                                              float carry_in, bool prev_ended, bool *last_ended,
                                              ScanSmem<NT> &sm, int buf)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int T = p.T;
    const int Te = active ? T : 0;
    const int64_t off = active ? row * p.ld : 0;

    const float init = EARLY_INIT ? load_init(p, row, t0, active) : 0.f;
    float x[ITEMS];
    load_items<ITEMS, VEC, TIn>(in_row<TIn>(p.reward, off), t0, Te, x);
    const unsigned ended = TRUNC ? load_flag_bits_or<ITEMS, VEC>(p.term + off, p.trunc + off, t0, Te)
                                 : load_flag_bits<ITEMS, VEC>(p.term + off, t0, Te);
    const unsigned valid = valid_items<ITEMS>(t0, Te);

    const unsigned prev_lane = __shfl_up_sync(kFullMask, ended >> (ITEMS - 1), 1) & 1u;
    unsigned reset = ((ended << 1) | (lane == 0 ? 0u : prev_lane)) | ~valid;
    if (t0 == 0 && active) {
        reset |= 1u;
        if (p.boot) x[0] = fmaf(p.gamma, EARLY_INIT ? init : __ldg(p.boot + row), x[0]);
    }
    reset &= all_items<ITEMS>();
#pragma unroll
    for (int j = 0; j < ITEMS; ++j)
        if (!((valid >> j) & 1u)) x[j] = 0.f;

    const float decay = p.gamma;
    float a = x[0];
#pragma unroll
    for (int j = 1; j < ITEMS; ++j) a = ((reset >> j) & 1u) ? x[j] : fmaf(decay, a, x[j]);
    Affine incl{a, reset ? kResetB : p.beta_pow};
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Affine y{__shfl_up_sync(kFullMask, incl.a, d), __shfl_up_sync(kFullMask, incl.b, d)};
        if (lane >= d) incl = affine_compose(incl, y);
    }
    Affine excl{__shfl_up_sync(kFullMask, incl.a, 1), __shfl_up_sync(kFullMask, incl.b, 1)};
    if (lane == 0) excl = affine_identity();
    if (lane == 31) {
        sm.a[buf][warp] = incl.a;
        sm.b[buf][warp] = incl.b;
        sm.e[buf][warp] = (ended >> (ITEMS - 1)) & 1u;
    }
    __syncthreads();

    // Prefix over the warp totals (lane w ends with total_w o ... o total_0); a warp whose
    // first step follows an episode end contributes a reset.
    Affine tw = affine_identity();
    if (lane < NW) {
        const bool fresh = lane == 0 ? prev_ended : sm.e[buf][lane - 1] != 0;
        tw = Affine{sm.a[buf][lane], fresh ? kResetB : sm.b[buf][lane]};
    }
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
        const Affine y{__shfl_up_sync(kFullMask, tw.a, d), __shfl_up_sync(kFullMask, tw.b, d)};
        if (lane >= d && lane < NW) tw = affine_compose(tw, y);
    }
    Affine earlier = shfl_idx(tw, (warp + 31) & 31);
    if (warp == 0) earlier = affine_identity();
    const Affine whole = shfl_idx(tw, NW - 1);
    const bool warp_fresh = warp == 0 ? prev_ended : sm.e[buf][warp - 1] != 0;
    *last_ended = sm.e[buf][NW - 1] != 0;

    float A[ITEMS];
    float prev = affine_apply(excl, warp_fresh ? 0.f : affine_apply(earlier, carry_in));
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        prev = ((reset >> j) & 1u) ? x[j] : fmaf(decay, prev, x[j]);
        A[j] = prev;
    }
    if (valid) store_items<ITEMS, VEC>(p.out0 + off, t0, valid, A);
    return affine_apply(whole, carry_in);
}

// CTA-tiled forward scan: T <= NT * ITEMS packs whole rows into a tile; longer rows are
// walked tile by tile from the first, with the carry in registers.
template <int NT, int ITEMS, int VEC, bool TRUNC, Tiling TL, typename TIn = float>
__global__ void __launch_bounds__(NT) credit_forward_tile_kernel(const Params p)
{
    __shared__ ScanSmem<NT> sm;
    constexpr int TILE = NT * ITEMS;
    // x and the flags (the discounted return's arrays); the row loop starts at tile 0.
    if (TL == Tiling::kRows) {
        if ((int)threadIdx.x < p.rows_per_tile)
            prefetch_row<Est::kReturn, TRUNC, TIn>(
                p, (int64_t)blockIdx.x * p.rows_per_tile + threadIdx.x, 0, p.T);
    } else if (threadIdx.x == 0) {
        prefetch_row<Est::kReturn, TRUNC, TIn>(p, blockIdx.x, 0, p.T < TILE ? p.T : TILE);
    }
    grid_dependency_sync();
    if (TL == Tiling::kRows) {
        const int local_row = threadIdx.x / p.chunks_per_row;
        const int chunk = threadIdx.x - local_row * p.chunks_per_row;
        const int64_t row = (int64_t)blockIdx.x * p.rows_per_tile + local_row;
        const bool active = local_row < p.rows_per_tile && row < p.N;
        bool last_ended = false;
        forward_tile<NT, ITEMS, VEC, TRUNC, TIn>(p, row, chunk * ITEMS, active, 0.f, false,
                                                 &last_ended, sm, 0);
    } else if (TL == Tiling::kRow) {
        bool last_ended = false;
        forward_tile<NT, ITEMS, VEC, TRUNC, TIn>(p, blockIdx.x, threadIdx.x * ITEMS, true, 0.f,
                                                 false, &last_ended, sm, 0);
    } else {
        const int64_t row = blockIdx.x;
        float carry = 0.f;
        bool ended = false;
        for (int s = 0; s < p.segs; ++s) {
            if (threadIdx.x == 0 && s + 1 < p.segs)
                prefetch_row<Est::kReturn, TRUNC, TIn>(
                    p, row, (s + 1) * TILE, (s + 2) * TILE < p.T ? (s + 2) * TILE : p.T);
            // init[row] read late, as the reverse row loop reads its bootstrap.
            carry = forward_tile<NT, ITEMS, VEC, TRUNC, TIn, false>(
                p, row, s * TILE + threadIdx.x * ITEMS, true, carry, ended, &ended, sm, s & 1);
        }
    }
}

}  // namespace rlca
