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
// Four tilings of the [N, T] rollout:
//   kRows      (T <= NT*ITEMS): a tile holds rows_per_tile whole rows, each padded to a
//              multiple of ITEMS. Every row ends in a reset at t = T-1, so tiles are
//              independent and no carry crosses a tile.
//   kRow       (NT*ITEMS/2 < T <= NT*ITEMS): kRows with exactly one row per tile; the
//              row and a thread's first step follow from the indices alone.
//   kRowLoop   (T > NT*ITEMS): one CTA per row walks the row's segs tiles from the last
//              to the first, carrying A at the first step of the later tile in registers.
//              Only one tile is on chip at a time, so long sequences never exhaust
//              registers or shared memory (the register-pressure limit the pages report
//              for Retrace at T > 2048 does not arise).
//   kLookback  (T > NT*ITEMS, caller workspace): one CTA per tile, all tiles of all rows
//              in flight at once. A tile's carry-in comes from the later tiles of its row
//              by decoupled look-back (Merrill & Garland 2016, run towards larger t):
//              each tile publishes its aggregate, then its inclusive value (A at its
//              first step) once known; a tile folds later aggregates until it meets an
//              inclusive value. A tile whose aggregate contains a reset knows its
//              inclusive value at once, so look-back never passes an episode boundary.
//
// Also here: the fused kernels (TD(lambda) for several lambdas, GAE with V-trace: one
// load of a tile, one scan per estimator), the warp-owned-rows kernel (a warp scans
// whole short rows, or walks a row in warp-sized chunks, with no CTA barrier), its
// pipelined form (a warp per row that keeps the next chunks' loads in flight) and the
// walked rows (a grid of one wave whose warps walk blocks of short rows, the next
// block's loads in flight). Where a thread holds a row's last step, the per-env
// bootstrap is read beside its data on most paths (load_boot), late where that measured
// faster (pipe_boot_mode, the row loops).
#pragma once

#include <type_traits>

#include "estimators.cuh"

namespace rlca {

enum class Tiling : int { kRows = 0, kRowLoop = 1, kLookback = 2, kRow = 4 };

template <int NT>
struct ScanSmem {
    float a[2][NT / 32];
    float b[2][NT / 32];
    unsigned e[2][NT / 32];  // forward scans: whether each warp's last step ended an episode
    float carry;
    unsigned tile;
    unsigned epoch;
};

// ------------------------------------------------------------------ look-back state

// Workspace: a 256-byte header, then one 32-byte state per tile (row-major over
// [N, segs]). A state word packs a float value (high 32 bits) with a tag (low 32 bits):
// tag = epoch * 4 + kind, kind 1 = aggregate alpha, 2 = aggregate beta, 3 = inclusive.
// The epoch advances once per launch, so states left by earlier launches never match
// and the workspace needs zeroing only once, before its first use.
struct LookbackHeader {
    unsigned epoch;         // launches completed on this workspace (mod 2^30)
    unsigned tile_counter;  // next virtual tile id of the running launch
    unsigned done_counter;  // CTAs of the running launch that have finished
    int error;              // 0, or RLCA_ERR_TIMEOUT (-7) after a wait gave up
};
constexpr int kWsHeaderBytes = 256;
constexpr int kTileStateBytes = 32;
constexpr unsigned kEpochMask = 0x3fffffffu;
constexpr int kErrTimeout = -7;

__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long pack(float v, unsigned tag)
{
    return ((unsigned long long)__float_as_uint(v) << 32) | tag;
}

__device__ __forceinline__ float unpack_value(unsigned long long w)
{
    return __uint_as_float((unsigned)(w >> 32));
}

__device__ __forceinline__ unsigned long long *tile_state(void *ws, int64_t tile)
{
    return reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kWsHeaderBytes +
                                                  tile * kTileStateBytes);
}

// Run by one thread: publish this tile's aggregate, find its carry-in from the later
// tiles of the row, publish its inclusive value, return the carry-in.
__device__ __forceinline__ float lookback_carry(const Params &p, int64_t row, int seg, unsigned epoch,
                                const Affine &tot)
{
    const unsigned tag_a = epoch * 4u + 1u, tag_b = epoch * 4u + 2u, tag_p = epoch * 4u + 3u;
    unsigned long long *me = tile_state(p.ws, row * p.segs + seg);
    const bool publish = p.stall == 0;
    if (seg == p.segs - 1) {  // the row's last tile ends in a reset at t = T-1
        if (publish) st_relaxed(me + 2, pack(affine_apply(tot, 0.f), tag_p));
        return 0.f;
    }
    const bool tot_reset = is_reset(tot.b);
    if (publish) {
        if (tot_reset) {
            st_relaxed(me + 2, pack(tot.a, tag_p));
        } else {
            st_relaxed(me + 0, pack(tot.a, tag_a));
            st_relaxed(me + 1, pack(tot.b, tag_b));
        }
    }
    Affine acc = affine_identity();
    float carry = 0.f;
    int j = seg + 1;
    int idle = 0;
    while (true) {
        unsigned long long *st = tile_state(p.ws, row * p.segs + j);
        const unsigned long long wp = ld_relaxed(st + 2);
        if ((unsigned)wp == tag_p) {
            carry = affine_apply(acc, unpack_value(wp));
            break;
        }
        const unsigned long long wa = ld_relaxed(st + 0);
        const unsigned long long wb = ld_relaxed(st + 1);
        if ((unsigned)wa == tag_a && (unsigned)wb == tag_b) {
            acc = affine_compose(acc, Affine{unpack_value(wa), unpack_value(wb)});
            ++j;  // the row's last tile always publishes an inclusive value: j < segs
            idle = 0;
            continue;
        }
        if (++idle > p.spin_limit) {  // bounded wait: report, never hang
            atomicExch(&static_cast<LookbackHeader *>(p.ws)->error, kErrTimeout);
            carry = __int_as_float(0x7fc00000);  // NaN marks this tile's outputs
            break;
        }
        __nanosleep(idle < 64 ? 32 : 256);
    }
    if (publish && !tot_reset) st_relaxed(me + 2, pack(affine_apply(tot, carry), tag_p));
    return carry;
}

// ------------------------------------------------------------------------- one tile

// Scan the loaded steps this thread owns, write the outputs and return A at the tile's
// first step. The tile's carry-in (A at the step after the tile) is `carry_in`, or,
// with LB, the result of the look-back (`epoch` and `seg` identify the tile's state).
template <Est E, int NT, int ITEMS, int VEC, bool LB, typename TIn = float>
__device__ __forceinline__ float scan_chunk(const Params &p, Chunk<ITEMS> &c, int64_t row,
                                            int t0, float carry_in, ScanSmem<NT> &sm, int buf,
                                            int seg = 0, unsigned epoch = 0)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    Affine e[ITEMS];
    build<E, ITEMS, TIn>(p, row, t0, c, e);

    // Thread aggregate: e_0 (+) e_1 (+) ... (+) e_{ITEMS-1}.
    const Affine agg = thread_aggregate<E, ITEMS>(p, c, e);

    // Warp suffix scan; the exclusive value of a lane is the inclusive one of lane+1.
    const Affine incl = warp_suffix_scan(agg, lane);
    Affine excl = shfl_down(incl, 1);
    if (lane == 31) excl = affine_identity();
    if (lane == 0) {
        sm.a[buf][warp] = incl.a;
        sm.b[buf][warp] = incl.b;
    }
    __syncthreads();

    if (LB) {
        if (threadIdx.x == 0) {
            Affine tot = Affine{sm.a[buf][0], sm.b[buf][0]};
#pragma unroll
            for (int w = 1; w < NW; ++w)
                tot = affine_compose(tot, Affine{sm.a[buf][w], sm.b[buf][w]});
            sm.carry = lookback_carry(p, row, seg, epoch, tot);
        }
        __syncthreads();
        carry_in = sm.carry;
    }

    // Combine the NW warp totals with a suffix scan over lanes 0..NW-1 of every warp:
    // lane w ends with S_w = total_w (+) ... (+) total_{NW-1}.
    Affine tw = affine_identity();
    if (lane < NW) tw = Affine{sm.a[buf][lane], sm.b[buf][lane]};
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
        const Affine y = shfl_down(tw, d);
        if (lane + d < NW) tw = affine_compose(tw, y);
    }
    // A at the step after this warp is S_{warp+1} applied to the tile carry-in; A at the
    // tile's first step is S_0 applied to it.
    Affine later = shfl_idx(tw, (warp + 1) & 31);
    if (warp == NW - 1) later = affine_identity();
    const Affine whole = shfl_idx(tw, 0);
    const float x = affine_apply(later, carry_in);
    const float a_after = affine_apply(excl, x);
    const float tile_first = affine_apply(whole, carry_in);

    float A[ITEMS];
    replay<E, ITEMS>(p, c, e, a_after, A);
    epilogue<E, ITEMS, VEC>(p, c, A, a_after, row, t0);
    return tile_first;
}

// Load this thread's steps from global memory, then scan_chunk. EARLY_BOOT: as in
// load_chunk.
template <Est E, int NT, int ITEMS, int VEC, bool TRUNC, bool LB, typename TIn = float,
          bool EARLY_BOOT = true>
__device__ __forceinline__ float scan_tile(const Params &p, int64_t row, int t0, bool active,
                                           float carry_in, ScanSmem<NT> &sm, int buf,
                                           int seg = 0, unsigned epoch = 0)
{
    Chunk<ITEMS> c;
    load_chunk<E, ITEMS, VEC, TRUNC, TIn, EARLY_BOOT>(p, row, t0, active, threadIdx.x & 31, c);
    return scan_chunk<E, NT, ITEMS, VEC, LB, TIn>(p, c, row, t0, carry_in, sm, buf, seg, epoch);
}

// Programmatic dependent launch: wait until the previous kernel in the stream has
// completed and its writes are visible (a no-op when the launch has no such
// dependency), then let the next kernel be scheduled while this one runs; that kernel
// in turn waits for this one to complete before it touches memory.
__device__ __forceinline__ void grid_dependency_sync()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Where a lane of a warp that owns whole rows works: its row within the warp's rows and
// its chunk within that row (a shift when the lanes per row are a power of two).
struct LaneSlot {
    int local_row, chunk;
};

__device__ __forceinline__ LaneSlot lane_slot(const Params &p, int lane)
{
    const int r = p.row_shift1 ? lane >> (p.row_shift1 - 1) : lane / p.chunks_per_row;
    return LaneSlot{r, lane - r * p.chunks_per_row};
}

// What a CTA of a tile kernel reads first, prefetched into L2 before its grid dependency
// wait: its whole rows (kRows, kRow) or the first tile it scans (kRowLoop: the row's
// last tile). One thread per row. Look-back tiles learn their tile only after the wait.
template <Est E, bool TRUNC, typename TIn, Tiling TL, int TILE>
__device__ __forceinline__ void prefetch_cta_rows(const Params &p)
{
    if (TL == Tiling::kRows) {
        if ((int)threadIdx.x < p.rows_per_tile)
            prefetch_row<E, TRUNC, TIn>(p, (int64_t)blockIdx.x * p.rows_per_tile + threadIdx.x,
                                        0, p.T);
    } else if (TL == Tiling::kRow) {
        if (threadIdx.x == 0) prefetch_row<E, TRUNC, TIn>(p, blockIdx.x, 0, p.T);
    } else if (TL == Tiling::kRowLoop) {
        if (threadIdx.x == 0)
            prefetch_row<E, TRUNC, TIn>(p, blockIdx.x, (p.segs - 1) * TILE, p.T);
    }
}

// The same for a warp that owns rows_per_tile whole rows (segs == 1; lane i takes row
// row0 + i) or walks one row (the last `steps` steps, which it scans first).
template <Est E, bool TRUNC, typename TIn>
__device__ __forceinline__ void prefetch_warp_rows(const Params &p, int64_t job, int steps)
{
    const int lane = threadIdx.x & 31;
    if (p.segs == 1) {
        if (lane < p.rows_per_tile)
            prefetch_row<E, TRUNC, TIn>(p, job * p.rows_per_tile + lane, 0, p.T);
    } else if (lane == 0) {
        prefetch_row<E, TRUNC, TIn>(p, job, p.T > steps ? p.T - steps : 0, p.T);
    }
}

template <Est E, int NT, int ITEMS, int VEC, bool TRUNC, Tiling TL, int MINB = 1,
          typename TIn = float>
__global__ void __launch_bounds__(NT, MINB) credit_scan_kernel(const Params p)
{
    __shared__ ScanSmem<NT> sm;
    prefetch_cta_rows<E, TRUNC, TIn, TL, NT * ITEMS>(p);
    grid_dependency_sync();
    constexpr int TILE = NT * ITEMS;
    if (TL == Tiling::kRows) {
        const int local_row = threadIdx.x / p.chunks_per_row;
        const int chunk = threadIdx.x - local_row * p.chunks_per_row;
        const int64_t row = (int64_t)blockIdx.x * p.rows_per_tile + local_row;
        const bool active = local_row < p.rows_per_tile && row < p.N;
        scan_tile<E, NT, ITEMS, VEC, TRUNC, false, TIn>(p, row, chunk * ITEMS, active, 0.f, sm,
                                                        0);
    } else if (TL == Tiling::kRow) {
        // One whole row per CTA (TILE / 2 < T <= TILE): the row and the thread's first
        // column follow from the indices alone (measured 4-5% faster than kRows there).
        scan_tile<E, NT, ITEMS, VEC, TRUNC, false, TIn>(p, blockIdx.x, threadIdx.x * ITEMS, true,
                                                        0.f, sm, 0);
    } else if (TL == Tiling::kRowLoop) {
        // The bootstrap is read late here: reading it with the last tile's data was
        // measured slower (Retrace [2048, 4096] 26.8 vs 25.8 us).
        const int64_t row = blockIdx.x;
        float carry = 0.f;
        for (int s = p.segs - 1; s >= 0; --s) {
            if (threadIdx.x == 0 && s > 0)  // the next tile's reads overlap this tile
                prefetch_row<E, TRUNC, TIn>(p, row, (s - 1) * TILE, s * TILE);
            carry = scan_tile<E, NT, ITEMS, VEC, TRUNC, false, TIn, false>(
                p, row, s * TILE + threadIdx.x * ITEMS, true, carry, sm, s & 1);
        }
    } else {
        LookbackHeader *h = static_cast<LookbackHeader *>(p.ws);
        if (threadIdx.x == 0) {
            // Virtual tile ids in start order; a row's later tiles get smaller ids, so
            // every tile waits only on tiles whose CTAs started before it.
            sm.tile = atomicAdd(&h->tile_counter, 1u);
            sm.epoch = *reinterpret_cast<volatile unsigned *>(&h->epoch);
        }
        __syncthreads();
        const unsigned vid = sm.tile;
        const unsigned epoch = sm.epoch;
        const int64_t row = vid / (unsigned)p.segs;
        const int seg = p.segs - 1 - (int)(vid - row * p.segs);
        scan_tile<E, NT, ITEMS, VEC, TRUNC, true, TIn>(p, row, seg * TILE + threadIdx.x * ITEMS,
                                                       true, 0.f, sm, 0, seg, epoch);
        // The last CTA to finish rearms the workspace for the next launch.
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned done = atomicAdd(&h->done_counter, 1u);
            if (done == gridDim.x - 1) {
                h->tile_counter = 0;
                h->done_counter = 0;
                h->epoch = (epoch + 1u) & kEpochMask;
                __threadfence();
            }
        }
    }
}

// ------------------------------------------------------ fused TD(lambda) (several)

// TD(lambda) for p.multi.count lambdas from one load of a tile: the chunk is read once,
// then built, scanned and stored once per lambda (each scan alternates the shared
// buffers, so consecutive scans never race on them).
template <int NT, int ITEMS, int VEC, bool TRUNC, Tiling TL>
__global__ void __launch_bounds__(NT) credit_td_multi_kernel(const Params p)
{
    __shared__ ScanSmem<NT> sm;
    prefetch_cta_rows<Est::kTdLambda, TRUNC, float, TL, NT * ITEMS>(p);
    grid_dependency_sync();
    constexpr int TILE = NT * ITEMS;
    int call = 0;
    auto tile = [&](int64_t row, int t0, bool active, float (&carry)[kMaxLambdas]) {
        Chunk<ITEMS> c;
        load_chunk<Est::kTdLambda, ITEMS, VEC, TRUNC>(p, row, t0, active, threadIdx.x & 31, c);
#pragma unroll
        for (int k = 0; k < kMaxLambdas; ++k) {
            if (k < p.multi.count) {
                Params q = p;
                q.gamma_lambda = p.multi.gamma_lambda[k];
                q.gamma_one_m_lambda = p.multi.gamma_one_m_lambda[k];
                q.beta_pow = p.multi.beta_pow[k];
                q.out0 = p.multi.out[k];
                carry[k] = scan_chunk<Est::kTdLambda, NT, ITEMS, VEC, false>(q, c, row, t0,
                                                                          carry[k], sm,
                                                                          call & 1);
                ++call;
            }
        }
    };
    float carry[kMaxLambdas] = {0.f, 0.f, 0.f, 0.f};
    if (TL == Tiling::kRows) {
        const int local_row = threadIdx.x / p.chunks_per_row;
        const int chunk = threadIdx.x - local_row * p.chunks_per_row;
        const int64_t row = (int64_t)blockIdx.x * p.rows_per_tile + local_row;
        tile(row, chunk * ITEMS, local_row < p.rows_per_tile && row < p.N, carry);
    } else if (TL == Tiling::kRow) {
        tile(blockIdx.x, threadIdx.x * ITEMS, true, carry);
    } else {
        const int64_t row = blockIdx.x;
        for (int s = p.segs - 1; s >= 0; --s) {
            if (threadIdx.x == 0 && s > 0)
                prefetch_row<Est::kTdLambda, TRUNC>(p, row, (s - 1) * TILE, s * TILE);
            tile(row, s * TILE + threadIdx.x * ITEMS, true, carry);
        }
    }
}

// Fused TD(lambda) on warp-owned rows (T <= 32 * ITEMS): each warp loads its whole rows
// once and scans them once per lambda with shuffles only (no CTA barrier). Rows end in a
// reset at the window end, so each lambda's scan starts from a carry of 0.
template <int ITEMS, int VEC, bool TRUNC, int WARPS = 4>
__global__ void __launch_bounds__(32 * WARPS) credit_td_multi_warp_kernel(const Params p)
{
    constexpr Est E = Est::kTdLambda;
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    const LaneSlot ls = lane_slot(p, lane);  // index math before the wait: no memory read
    const int64_t row = job * p.rows_per_tile + ls.local_row;
    const bool active = ls.local_row < p.rows_per_tile && row < p.N;
    const int t0 = ls.chunk * ITEMS;
    prefetch_warp_rows<E, TRUNC, float>(p, job, p.T);
    grid_dependency_sync();
    Chunk<ITEMS> c;
    load_chunk<E, ITEMS, VEC, TRUNC>(p, row, t0, active, lane, c);
#pragma unroll
    for (int k = 0; k < kMaxLambdas; ++k) {
        if (k < p.multi.count) {
            Params q = p;
            q.gamma_lambda = p.multi.gamma_lambda[k];
            q.gamma_one_m_lambda = p.multi.gamma_one_m_lambda[k];
            q.beta_pow = p.multi.beta_pow[k];
            q.out0 = p.multi.out[k];
            Affine e[ITEMS];
            build<E, ITEMS>(q, row, t0, c, e);
            const Affine incl = warp_suffix_scan(thread_aggregate<E, ITEMS>(q, c, e), lane);
            Affine excl = shfl_down(incl, 1);
            if (lane == 31) excl = affine_identity();
            const float a_after = affine_apply(excl, 0.f);
            float A[ITEMS];
            replay<E, ITEMS>(q, c, e, a_after, A);
            epilogue<E, ITEMS, VEC>(q, c, A, a_after, row, t0);
        }
    }
}

// ------------------------------------------------------ fused GAE + V-trace

// GAE and V-trace from one load of a tile: the V-trace chunk (reward, value, log ratios,
// flags) holds every input GAE reads, so the tile is loaded once and scanned twice. GAE
// goes first: V-trace's build turns the log ratios into ratios in place. `pg` holds the
// GAE parameters and outputs, `pv` the V-trace ones; the two scans alternate the shared
// buffers.
template <int NT, int ITEMS, int VEC, bool TRUNC, Tiling TL, int MINB = 1>
__global__ void __launch_bounds__(NT, MINB) credit_gae_vtrace_kernel(const Params pg,
                                                                      const Params pv)
{
    __shared__ ScanSmem<NT> sm;
    prefetch_cta_rows<Est::kVtrace, TRUNC, float, TL, NT * ITEMS>(pv);
    grid_dependency_sync();
    constexpr int TILE = NT * ITEMS;
    auto tile = [&](int64_t row, int t0, bool active, float (&carry)[2], int buf) {
        Chunk<ITEMS> c;
        load_chunk<Est::kVtrace, ITEMS, VEC, TRUNC>(pv, row, t0, active, threadIdx.x & 31, c);
        carry[0] = scan_chunk<Est::kGae, NT, ITEMS, VEC, false>(pg, c, row, t0, carry[0], sm,
                                                                  buf);
        carry[1] = scan_chunk<Est::kVtrace, NT, ITEMS, VEC, false>(pv, c, row, t0, carry[1],
                                                                     sm, buf ^ 1);
    };
    float carry[2] = {0.f, 0.f};
    if (TL == Tiling::kRows) {
        const int local_row = threadIdx.x / pv.chunks_per_row;
        const int chunk = threadIdx.x - local_row * pv.chunks_per_row;
        const int64_t row = (int64_t)blockIdx.x * pv.rows_per_tile + local_row;
        tile(row, chunk * ITEMS, local_row < pv.rows_per_tile && row < pv.N, carry, 0);
    } else if (TL == Tiling::kRow) {
        tile(blockIdx.x, threadIdx.x * ITEMS, true, carry, 0);
    } else {
        const int64_t row = blockIdx.x;
        for (int s = pv.segs - 1; s >= 0; --s) {
            if (threadIdx.x == 0 && s > 0)
                prefetch_row<Est::kVtrace, TRUNC>(pv, row, (s - 1) * TILE, s * TILE);
            tile(row, s * TILE + threadIdx.x * ITEMS, true, carry, 0);
        }
    }
}

// Fused GAE + V-trace on warp-owned rows (T <= 32 * ITEMS): each warp loads its whole
// rows once (the V-trace chunk) and scans them for GAE, then for V-trace, with shuffles
// only. MINB: CTAs per SM the register allocator must fit (0 = no request).
template <int ITEMS, int VEC, bool TRUNC, int WARPS = 4, int MINB = 0>
__global__ void __launch_bounds__(32 * WARPS, MINB) credit_gae_vtrace_warp_kernel(
    const Params pg, const Params pv)
{
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    const LaneSlot ls = lane_slot(pv, lane);
    const int64_t row = job * pv.rows_per_tile + ls.local_row;
    const bool active = ls.local_row < pv.rows_per_tile && row < pv.N;
    const int t0 = ls.chunk * ITEMS;
    prefetch_warp_rows<Est::kVtrace, TRUNC, float>(pv, job, pv.T);
    grid_dependency_sync();
    Chunk<ITEMS> c;
    load_chunk<Est::kVtrace, ITEMS, VEC, TRUNC>(pv, row, t0, active, lane, c);
    {
        Affine e[ITEMS];
        build<Est::kGae, ITEMS>(pg, row, t0, c, e);
        const Affine incl = warp_suffix_scan(thread_aggregate<Est::kGae, ITEMS>(pg, c, e), lane);
        Affine excl = shfl_down(incl, 1);
        if (lane == 31) excl = affine_identity();
        const float a_after = affine_apply(excl, 0.f);
        float A[ITEMS];
        replay<Est::kGae, ITEMS>(pg, c, e, a_after, A);
        epilogue<Est::kGae, ITEMS, VEC>(pg, c, A, a_after, row, t0);
    }
    {
        Affine e[ITEMS];
        build<Est::kVtrace, ITEMS>(pv, row, t0, c, e);
        const Affine incl =
            warp_suffix_scan(thread_aggregate<Est::kVtrace, ITEMS>(pv, c, e), lane);
        Affine excl = shfl_down(incl, 1);
        if (lane == 31) excl = affine_identity();
        const float a_after = affine_apply(excl, 0.f);
        float A[ITEMS];
        replay<Est::kVtrace, ITEMS>(pv, c, e, a_after, A);
        epilogue<Est::kVtrace, ITEMS, VEC>(pv, c, A, a_after, row, t0);
    }
}

// ------------------------------------------------------------------ warp-owned rows

// One warp scans a chunk of 32 * ITEMS steps with no help from other warps: lane
// aggregates, a warp suffix scan, and the chunk's carry-in (A at the step after the
// chunk) applied directly. Returns A at the chunk's first step.
template <Est E, int ITEMS, int VEC, typename TIn = float>
__device__ __forceinline__ float warp_chunk_scan(const Params &p, int64_t row, int t0,
                                                 Chunk<ITEMS> &c, float carry_in)
{
    const int lane = threadIdx.x & 31;
    Affine e[ITEMS];
    build<E, ITEMS, TIn>(p, row, t0, c, e);
    const Affine agg = thread_aggregate<E, ITEMS>(p, c, e);
    const Affine incl = warp_suffix_scan(agg, lane);
    Affine excl = shfl_down(incl, 1);
    if (lane == 31) excl = affine_identity();
    const Affine whole = shfl_idx(incl, 0);
    const float a_after = affine_apply(excl, carry_in);
    float A[ITEMS];
    replay<E, ITEMS>(p, c, e, a_after, A);
    epilogue<E, ITEMS, VEC>(p, c, A, a_after, row, t0);
    return affine_apply(whole, carry_in);
}

// The same, loading the chunk first (ragged and inactive chunks allowed).
template <Est E, int ITEMS, int VEC, bool TRUNC, typename TIn = float>
__device__ __forceinline__ float warp_chunk(const Params &p, int64_t row, int t0, bool active,
                                            float carry_in)
{
    Chunk<ITEMS> c;
    load_chunk<E, ITEMS, VEC, TRUNC, TIn>(p, row, t0, active, threadIdx.x & 31, c);
    return warp_chunk_scan<E, ITEMS, VEC, TIn>(p, row, t0, c, carry_in);
}

// Every warp of the grid owns one job, with no barrier and no shared memory:
//   T <= 32 * ITEMS: rows_per_tile whole rows (padded to a multiple of ITEMS) per warp;
//   longer T: one row per warp, walked in chunks of 32 * ITEMS steps from the last to the
//   first with the carry in a register.
// All warps of a typical launch are resident at once, so each keeps its next chunk's
// loads in flight without any cross-warp wait.
// MINB: CTAs per SM the register allocator must fit (0 = no request; an explicit 1
// changes the allocation, so 0 is the default).
template <Est E, int ITEMS, int VEC, bool TRUNC, int WARPS = 4, typename TIn = float,
          int MINB = 0>
__global__ void __launch_bounds__(32 * WARPS, MINB) credit_warp_kernel(const Params p)
{
    constexpr int CH = 32 * ITEMS;
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    // Whole rows per warp: the index math reads no memory, so it can run before the wait
    // and leave the critical path (measured at [4096, 128]: return 2.22 -> 2.15 us,
    // TD(lambda) 2.61 -> 2.50). A register-capped kernel does it after the wait (V-trace
    // at [8192, 256]: 8.22 us after, 8.33 before).
    LaneSlot ls;
    int64_t row = 0;
    bool active = false;
    auto slot = [&] {
        ls = lane_slot(p, lane);
        row = job * p.rows_per_tile + ls.local_row;
        active = ls.local_row < p.rows_per_tile && row < p.N;
    };
    if constexpr (MINB == 0) slot();
    prefetch_warp_rows<E, TRUNC, TIn>(p, job, 1024);
    grid_dependency_sync();
    if (p.segs == 1) {
        if constexpr (MINB != 0) slot();
        warp_chunk<E, ITEMS, VEC, TRUNC, TIn>(p, row, ls.chunk * ITEMS, active, 0.f);
    } else {
        if (job >= p.N) return;  // the whole warp leaves together
        float carry = 0.f;
        for (int s = p.segs - 1; s >= 0; --s)
            carry = warp_chunk<E, ITEMS, VEC, TRUNC, TIn>(p, job, s * CH + lane * ITEMS, true,
                                                          carry);
    }
}

// Walks one row per warp in chunks of 32 * ITEMS steps from the last to the first with
// the next chunks' loads in flight: before a chunk is scanned, the warp has already
// asked for the raw words of the DEPTH chunks before it (registers as a software
// pipeline), so its HBM reads overlap its own scans and stores instead of alternating
// with them. A ragged last chunk goes first through the plain load, before the
// pipeline starts; every chunk after that is full. scan(t0, c) scans one loaded chunk
// (thread's first step t0). Needs 16-byte aligned rows (VEC >= 1). BOOT: how the
// bootstrap of the row's end is read (pipe_boot_mode).
template <Est E, int ITEMS, int VEC, bool TRUNC, int DEPTH, typename TIn, int BOOT,
          typename Scan>
__device__ __forceinline__ void warp_pipe_row(const Params &p, int64_t row, Scan &&scan)
{
    static_assert(DEPTH >= 1 && DEPTH <= 3, "one to three chunks in flight");
    static_assert(VEC & kVec16, "raw chunks are read with vector loads");
    constexpr int CH = 32 * ITEMS;
    const int lane = threadIdx.x & 31;
    const int64_t off = row * p.ld;
    int s = p.segs - 1;
    if (p.T != p.segs * CH) {
        Chunk<ITEMS> c;
        load_chunk<E, ITEMS, VEC, TRUNC, TIn>(p, row, s * CH + lane * ITEMS, true, lane, c);
        scan(s * CH + lane * ITEMS, c);
        --s;
    }
    if (s < 0) return;
    // The row's last step is in chunk s unless a ragged chunk took it above.
    const float boot = BOOT > 0 ? load_boot<ITEMS>(p, row, s * CH + lane * ITEMS, true) : 0.f;
    // w[d] holds chunk s - d (registers: every index below is a compile-time constant).
    RawChunk<E, ITEMS, TIn> w[DEPTH];
#pragma unroll
    for (int d = 0; d < DEPTH; ++d)
        if (s - d >= 0)
            load_raw<E, ITEMS, VEC, TRUNC>(p, off, (s - d) * CH + lane * ITEMS, lane, w[d]);
    auto step = [&](int k, float boot_v) {
        const int t0 = k * CH + lane * ITEMS;
        if (lane == 0 && p.pf_ahead > 0 && k >= p.pf_ahead)  // beyond the registers' reach
            prefetch_row<E, TRUNC, TIn>(p, row, (k - p.pf_ahead) * CH,
                                        (k - p.pf_ahead + 1) * CH);
        Chunk<ITEMS> c;
        unpack_raw<E, ITEMS, TRUNC>(w[0], p.T, t0, lane, boot_v, c);
        c.boot_late = BOOT == 0;
#pragma unroll
        for (int d = 0; d + 1 < DEPTH; ++d) w[d] = w[d + 1];
        if (k - DEPTH >= 0)
            load_raw<E, ITEMS, VEC, TRUNC>(p, off, (k - DEPTH) * CH + lane * ITEMS, lane,
                                           w[DEPTH - 1]);
        scan(t0, c);
    };
    if (BOOT == 2) {  // the first chunk scanned holds the row's end; the rest need no value
        step(s, boot);
        --s;
    }
    for (; s >= 0; --s) step(s, BOOT == 1 ? boot : 0.f);
}

// How the pipelined rows read the per-env bootstrap (the successor value of the row's
// last step, in the first chunk they scan): 0, once that chunk's flags are in (a second
// memory latency on the warp's path, no register held); 1, together with the chunk's
// raw words (load_boot; the value is held through the walk); 2, the same with the first
// chunk's step peeled off the loop, so the value is dead after it (a second copy of the
// scan code). Measured on GB300 at [4096, 1024], us per launch for modes 0 / 1 / 2:
// fp32 TD(lambda) 9.33 / 9.05 / 9.02, GAE 12.29 / 12.31 / 12.31; bf16 TD(lambda)
// 7.99 / 7.79 / 7.01, GAE 11.00 / 10.90 / 10.45, V-trace 11.89 / 11.54 / 11.70, Retrace
// 9.17 / 8.96 / 9.43; fp16 TD(lambda) 7.40 / 7.60 / 7.50, GAE 10.89 / 10.74 / 10.43,
// V-trace 11.89 / 12.36 / 12.27, Retrace 9.91 / 9.02 / 9.20; fused TD(lambda) 14.40 /
// 14.53 / 14.55. The differences follow the register allocation of each kernel more
// than the latency itself. The fp32 return's pipelined rows (rows of 513-960 steps)
// take mode 2 as TD(lambda) does.
template <Est E, typename TIn>
__host__ __device__ constexpr int pipe_boot_mode()
{
    if (sizeof(TIn) == 4) return (E == Est::kTdLambda || E == Est::kReturn) ? 2 : 0;
    if (E == Est::kVtrace || E == Est::kRetrace)
        return (E == Est::kVtrace && !std::is_same<TIn, uint16_t>::value) ? 0 : 1;
    if (E == Est::kTdLambda && !std::is_same<TIn, uint16_t>::value) return 0;
    return 2;
}

// Pipelined warp-owned rows (warp_pipe_row): one row per warp, T > 32 * ITEMS. MINB:
// CTAs per SM the register allocator must fit (0 = no request).
template <Est E, int ITEMS, int VEC, bool TRUNC, int DEPTH, int WARPS = 4,
          typename TIn = float, int MINB = 0>
__global__ void __launch_bounds__(32 * WARPS, MINB) credit_warp_pipe_kernel(const Params p)
{
    const int64_t row = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if ((threadIdx.x & 31) == 0)  // the row's last pf_first steps, scanned first
        prefetch_row<E, TRUNC, TIn>(p, row, p.T > p.pf_first ? p.T - p.pf_first : 0, p.T);
    grid_dependency_sync();
    if (row >= p.N) return;  // the whole warp leaves together
    float carry = 0.f;
    constexpr int BOOT = pipe_boot_mode<E, TIn>();
    warp_pipe_row<E, ITEMS, VEC, TRUNC, DEPTH, TIn, BOOT>(p, row, [&](int t0, Chunk<ITEMS> &c) {
        carry = warp_chunk_scan<E, ITEMS, VEC, TIn>(p, row, t0, c, carry);
    });
}

// Rows that tile one warp chunk exactly (rows_per_tile rows of T steps, T * rows_per_tile
// == 32 * ITEMS, contiguous when there are several), more of these jobs than one wave of
// warps holds: a grid of one wave in which each warp walks jobs j, j + stride, ... and
// asks for the next job's raw words before it scans the current one, so its loads
// overlap its own scans instead of waiting for a warp of a second wave to start.
// 16-byte aligned rows; N a multiple of rows_per_tile.
template <Est E, int ITEMS, int VEC, bool TRUNC, int WARPS, typename TIn = float,
          int MINB = 0>
__global__ void __launch_bounds__(32 * WARPS, MINB) credit_warp_rows_pipe_kernel(const Params p)
{
    static_assert(VEC & kVec16, "raw chunks are read with vector loads");
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * WARPS;
    const int64_t jobs = p.N / p.rows_per_tile;
    int64_t job = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    const LaneSlot ls = lane_slot(p, lane);
    const int t0 = ls.chunk * ITEMS;  // within the lane's row
    const int tb = lane * ITEMS;      // within the job's block of rows
    if (lane < p.rows_per_tile)
        prefetch_row<E, TRUNC, TIn>(p, job * p.rows_per_tile + lane, 0, p.T);
    grid_dependency_sync();
    if (job >= jobs) return;  // the whole warp leaves together
    // The bootstrap of each job's rows is read with its raw words, except for GAE, which
    // reads it once the flags are in (walked rows at [8192, 256], us per launch, late vs
    // early: return 4.22 vs 3.86, TD(lambda) 4.82 vs 4.56, GAE 7.06 vs 7.18).
    constexpr bool EARLY = E != Est::kGae;
    RawChunk<E, ITEMS, TIn> w;
    load_raw<E, ITEMS, VEC, TRUNC>(p, job * p.rows_per_tile * p.ld, tb, lane, w);
    float boot = EARLY ? load_boot<ITEMS>(p, job * p.rows_per_tile + ls.local_row, t0, true)
                       : 0.f;
    while (true) {
        Chunk<ITEMS> c;
        unpack_raw<E, ITEMS, TRUNC>(w, p.T, t0, lane, boot, c);
        c.boot_late = !EARLY;
        const int64_t next = job + stride;
        if (next < jobs) {
            load_raw<E, ITEMS, VEC, TRUNC>(p, next * p.rows_per_tile * p.ld, tb, lane, w);
            if (EARLY)
                boot = load_boot<ITEMS>(p, next * p.rows_per_tile + ls.local_row, t0, true);
        }
        warp_chunk_scan<E, ITEMS, VEC, TIn>(p, job * p.rows_per_tile + ls.local_row, t0, c,
                                            0.f);
        if (next >= jobs) break;
        job = next;
    }
}

// Fused TD(lambda) on pipelined warp-owned rows: each loaded chunk is scanned once per
// lambda, each lambda with its own carry.
template <int ITEMS, int VEC, bool TRUNC, int DEPTH, int WARPS = 4, int MINB = 0>
__global__ void __launch_bounds__(32 * WARPS, MINB) credit_td_multi_pipe_kernel(const Params p)
{
    constexpr Est E = Est::kTdLambda;
    const int64_t row = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if ((threadIdx.x & 31) == 0)
        prefetch_row<E, TRUNC, float>(p, row, p.T > p.pf_first ? p.T - p.pf_first : 0, p.T);
    grid_dependency_sync();
    if (row >= p.N) return;
    float carry[kMaxLambdas] = {0.f, 0.f, 0.f, 0.f};
    warp_pipe_row<E, ITEMS, VEC, TRUNC, DEPTH, float, 0>(p, row, [&](int t0, Chunk<ITEMS> &c) {
#pragma unroll
        for (int k = 0; k < kMaxLambdas; ++k) {
            if (k < p.multi.count) {
                Params q = p;
                q.gamma_lambda = p.multi.gamma_lambda[k];
                q.gamma_one_m_lambda = p.multi.gamma_one_m_lambda[k];
                q.beta_pow = p.multi.beta_pow[k];
                q.out0 = p.multi.out[k];
                carry[k] = warp_chunk_scan<E, ITEMS, VEC>(q, row, t0, c, carry[k]);
            }
        }
    });
}

}  // namespace rlca
