// Warp-owned rows with a per-warp TMA pipeline (the warp-streaming tiling).
//
// Every warp of a persistent grid owns a contiguous, balanced range of rows and needs no
// other warp: no CTA barrier and no shared scan state. It walks each of its rows in
// chunks of WCH = 32 * ITEMS steps from the last to the first, carrying A between them
// in a register (rows are longer than one chunk: shorter rows take warp-owned rows).
// Lane 0 keeps STAGES chunks in flight with cp.async.bulk copies into the warp's own ring
// of shared-memory stages (one mbarrier per stage); the whole warp scans the current
// chunk from shared memory meanwhile: lane aggregates, a 5-round shuffle suffix scan,
// the carry applied, outputs stored from registers once.
// Requirements (checked by the launcher) as for the streaming tiling: 16-byte aligned
// bases, ld % 16 == 0, T % 16 == 0.
#pragma once

#include "stream.cuh"

namespace rlca {

constexpr int kWarpChunk = 256;  // 32 lanes x 8 steps

template <Est E>
using WarpStage = ChunkLayout<E, kWarpChunk>;

// Bytes of one warp's ring for an estimator: the ring depth shrinks as the chunk grows
// so that every resident warp's ring fits next to its neighbours'.
template <Est E>
__host__ __device__ constexpr int warp_stages()
{
    return WarpStage<E>::kBytes <= 1536 ? 4 : (WarpStage<E>::kBytes <= 2560 ? 3 : 2);
}

// Job cursor: (unit, chunk) walking units in order and each row's chunks last to first.
struct WarpCursor {
    int64_t unit;
    int chunk;
};

__device__ __forceinline__ StreamJob warp_job(const Params &p, WarpCursor c)
{
    StreamJob j;
    j.row = c.unit;
    j.t_start = c.chunk * kWarpChunk;
    j.src = j.row * p.ld + j.t_start;
    j.len = min(kWarpChunk, p.T - j.t_start);
    return j;
}

__device__ __forceinline__ void warp_advance(const Params &p, WarpCursor &c)
{
    if (--c.chunk < 0) {
        c.chunk = p.segs - 1;
        ++c.unit;
    }
}

template <Est E, bool TRUNC, int WARPS>
__global__ void __launch_bounds__(32 * WARPS) credit_warp_stream_kernel(const Params p)
{
    grid_dependency_sync();
    constexpr int ITEMS = kWarpChunk / 32;
    constexpr int STAGES = warp_stages<E>();
    using L = WarpStage<E>;
    extern __shared__ __align__(128) unsigned char rings[];
    __shared__ __align__(8) uint64_t bars[WARPS][STAGES];

    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    unsigned char *ring = rings + w * (STAGES * L::kBytes);
    uint64_t *full = bars[w];

    const int64_t units = p.N;
    const int64_t G = (int64_t)gridDim.x * WARPS;
    const int64_t g = (int64_t)blockIdx.x * WARPS + w;
    const int64_t u0 = units * g / G;
    const int64_t u1 = units * (g + 1) / G;
    const int64_t nchunks = (u1 - u0) * p.segs;
    if (nchunks == 0) return;  // the whole warp leaves; nothing here waits on other warps

    uint64_t policy = 0;
    WarpCursor prod{u0, p.segs - 1};
    if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
        policy = evict_first_policy();
        for (int64_t k = 0; k < nchunks && k < STAGES; ++k) {
            stream_issue<E, TRUNC, L>(p, warp_job(p, prod), ring + k * L::kBytes, &full[k],
                                      policy);
            warp_advance(p, prod);
        }
    }
    __syncwarp();

    WarpCursor cons{u0, p.segs - 1};
    float carry = 0.f;
    for (int64_t k = 0; k < nchunks; ++k) {
        // Every lane finished reading the previous chunk's stage: refill it.
        __syncwarp();
        if (lane == 0 && k > 0 && k - 1 + STAGES < nchunks) {
            const int s = (int)((k - 1) % STAGES);
            stream_issue<E, TRUNC, L>(p, warp_job(p, prod), ring + s * L::kBytes, &full[s],
                                      policy);
            warp_advance(p, prod);
        }
        const int s = (int)(k % STAGES);
        const bool arrived =
            mbar_wait(&full[s], (uint32_t)((k / STAGES) & 1), kStreamWaitLimit);
        const StreamJob j = warp_job(p, cons);
        const int li = lane * ITEMS;
        const bool active = li < j.len;
        const int64_t row = j.row;
        const int t0 = j.t_start + li;
        Chunk<ITEMS> c;
        load_chunk_stage<E, ITEMS, TRUNC, L>(p, ring + s * L::kBytes, j, li, row, t0, active, c);
        if (!arrived) {  // the copy never completed: mark this chunk's outputs invalid
#pragma unroll
            for (int i = 0; i < ITEMS; ++i) c.r[i] = __int_as_float(0x7fc00000);
        }
        const float carry_in = cons.chunk == p.segs - 1 ? 0.f : carry;

        Affine e[ITEMS];
        build<E, ITEMS>(p, row, t0, c, e);
        const Affine agg = thread_aggregate<E, ITEMS>(p, c, e);
        const Affine incl = warp_suffix_scan(agg, lane);
        Affine excl = shfl_down(incl, 1);
        if (lane == 31) excl = affine_identity();
        const Affine whole = shfl_idx(incl, 0);
        const float a_after = affine_apply(excl, carry_in);
        float A[ITEMS];
        replay<E, ITEMS>(p, c, e, a_after, A);
        epilogue<E, ITEMS, kVec16>(p, c, A, a_after, row, t0);
        carry = affine_apply(whole, carry_in);
        warp_advance(p, cons);
    }
}

}  // namespace rlca
