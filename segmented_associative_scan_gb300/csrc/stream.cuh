// Shared-memory stages filled by TMA bulk copies: the layout of one stage, the copy of
// one job's inputs into it, and the loading of a thread's steps back out of it. Used by
// the warp-streaming kernel (warp_stream.cuh).
//
// A job is `len` consecutive elements of every per-step array. The copies need every
// base pointer 16-byte aligned, ld % 16 == 0 and T % 16 == 0 (checked by the launcher),
// so each copy starts on a 16-byte boundary and moves a multiple of 16 bytes, and every
// thread's 8 steps are either all inside or all outside the row.
#pragma once

#include "kernels.cuh"
#include "tma.cuh"

namespace rlca {

// Bounded waits on the pipeline's own copies (each try_wait suspends a while).
constexpr int kStreamWaitLimit = 1 << 22;

// Shared-memory layout of one stage holding CH steps of every input the estimator reads.
template <Est E, int CH>
struct ChunkLayout {
    using Tr = EstTraits<E>;
    static constexpr int kR = 0;
    static constexpr int kV = kR + 4 * CH;
    static constexpr int kX = kV + (Tr::kValue ? 4 * CH : 0);
    static constexpr int kY = kX + (Tr::kAux ? 4 * CH : 0);
    static constexpr int kTerm = kY + (Tr::kRho ? 4 * CH : 0);
    static constexpr int kTrunc = kTerm + CH;
    static constexpr int kBytes = kTrunc + CH;
};
// One job: `len` consecutive elements starting at element `src` of every per-step array.
struct StreamJob {
    int64_t row;   // row of the first element
    int64_t src;   // element offset of the first element (row * ld + t_start)
    int t_start;   // column of the first element
    int len;       // elements in the job (a multiple of 16)
};

template <Est E, bool TRUNC, class L>
__device__ __forceinline__ void stream_issue(const Params &p, const StreamJob &j,
                                             unsigned char *stage, uint64_t *bar,
                                             uint64_t policy)
{
    using Tr = EstTraits<E>;
    const uint32_t fb = 4u * (uint32_t)j.len;  // bytes per fp32 array
    const uint32_t bb = (uint32_t)j.len;       // bytes per flag array
    const uint32_t n_f32 = 1 + Tr::kValue + Tr::kAux + Tr::kRho;
    mbar_arrive_expect_tx(bar, n_f32 * fb + (TRUNC ? 2u : 1u) * bb);
    bulk_g2s(stage + L::kR, p.reward + j.src, fb, bar, policy);
    if (Tr::kValue) bulk_g2s(stage + L::kV, p.value + j.src, fb, bar, policy);
    if (Tr::kAux) bulk_g2s(stage + L::kX, p.aux + j.src, fb, bar, policy);
    if (Tr::kRho) bulk_g2s(stage + L::kY, p.rho + j.src, fb, bar, policy);
    bulk_g2s(stage + L::kTerm, p.term + j.src, bb, bar, policy);
    if (TRUNC) bulk_g2s(stage + L::kTrunc, p.trunc + j.src, bb, bar, policy);
}

template <int ITEMS>
__device__ __forceinline__ void load_stage_items(const float *s, float (&x)[ITEMS])
{
#pragma unroll
    for (int k = 0; k < ITEMS / 4; ++k) {
        const float4 q = reinterpret_cast<const float4 *>(s)[k];
        x[4 * k + 0] = q.x;
        x[4 * k + 1] = q.y;
        x[4 * k + 2] = q.z;
        x[4 * k + 3] = q.w;
    }
}

template <int ITEMS>
__device__ __forceinline__ unsigned stage_flag_bits(const unsigned char *s)
{
    unsigned bits = 0;
#pragma unroll
    for (int k = 0; k < ITEMS / 4; ++k)
        bits |= nonzero_bytes(reinterpret_cast<const uint32_t *>(s)[k]) << (4 * k);
    return bits;
}

// The successor of the thread's last step: in the stage when it is part of the job,
// else (a row segment's last thread) read directly from global memory.
__device__ __forceinline__ float stage_next(const float *stage_arr, const float *global_arr,
                                            const StreamJob &j, int li, int t0, int items)
{
    if (li + items < j.len) return stage_arr[li + items];
    return __ldg(global_arr + j.src + li + items);
}

// This thread's ITEMS steps of the job from the stage (chunks are all-or-nothing).
template <Est E, int ITEMS, bool TRUNC, class L>
__device__ __forceinline__ void load_chunk_stage(const Params &p, const unsigned char *stage,
                                                 const StreamJob &j, int li, int64_t row,
                                                 int t0, bool active, Chunk<ITEMS> &c)
{
    using Tr = EstTraits<E>;
    const float *sr = reinterpret_cast<const float *>(stage + L::kR);
    const float *sv = reinterpret_cast<const float *>(stage + L::kV);
    const float *sx = reinterpret_cast<const float *>(stage + L::kX);
    const float *sy = reinterpret_cast<const float *>(stage + L::kY);
    if (active) {
        load_stage_items<ITEMS>(sr + li, c.r);
        if (Tr::kValue) load_stage_items<ITEMS>(sv + li, c.v);
        if (Tr::kAux) load_stage_items<ITEMS>(sx + li, c.x);
        if (Tr::kRho) load_stage_items<ITEMS>(sy + li, c.y);
        c.term = stage_flag_bits<ITEMS>(stage + L::kTerm + li);
        c.trunc = TRUNC ? stage_flag_bits<ITEMS>(stage + L::kTrunc + li) : 0u;
        c.valid = all_items<ITEMS>();
    } else {
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) c.r[i] = c.v[i] = c.x[i] = c.y[i] = 0.f;
        c.term = c.trunc = 0u;
        c.valid = 0u;
    }
    const int last = p.T - 1 - t0;
    const unsigned window_end = (last >= 0 && last < ITEMS) ? (1u << last) : 0u;
    c.stop = (c.term | c.trunc | window_end | ~c.valid) & all_items<ITEMS>();
    const bool need = active && (t0 + ITEMS < p.T);
    c.v_next = c.x_next = c.y_next = 0.f;
    if (need) {
        if (Tr::kNextValue) c.v_next = stage_next(sv, p.value, j, li, t0, ITEMS);
        if (Tr::kNextAux) c.x_next = stage_next(sx, p.aux, j, li, t0, ITEMS);
        if (Tr::kNextRho) c.y_next = stage_next(sy, p.rho, j, li, t0, ITEMS);
    }
}

}  // namespace rlca
