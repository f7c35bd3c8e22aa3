// Host-side launch of the fused kernels: picks the kernel from the shape, the layout and
// whether the caller gave a look-back workspace, then launches on the caller's stream.
//
// Every kernel begins with griddepcontrol.wait, so it is launched with programmatic
// stream serialization (PDL): when the previous kernel in the stream allows it, this
// launch is scheduled while that kernel drains, and still touches no memory before it
// has completed. With a predecessor that does not opt in, the launch behaves as usual.
#pragma once

#include <atomic>
#include <type_traits>

#include "kernels.cuh"

namespace rlca {

// CTA tiles: 128 threads x 8 steps.
constexpr int kThreads = 128;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;
// Warp-owned rows: independent warps per CTA, 32 lanes x 8 steps per chunk; 4 for the
// pipelined rows, kWarpRowsPerCta for the rows a warp owns whole (short rows). Measured
// on GB300, 2 / 4 / 8 warps per CTA, us per launch: TD(lambda) [4096, 128] 2.375 / 2.50 /
// 2.63, fused TD(lambda) 3.31 / 3.36 / 3.50, return 2.154 / 2.156 / 2.252, V-trace
// [8192, 256] 8.13 / 8.15 / 9.23.
constexpr int kWarpsPerCta = 4;
constexpr int kWarpRowsPerCta = 2;

// Look-back tiles of an [N, T] problem (0 when T fits one tile: no look-back needed).
inline int64_t lookback_tiles(int64_t N, int64_t T)
{
    return T > kTile ? N * ((T + kTile - 1) / kTile) : 0;
}

inline size_t workspace_bytes(int64_t N, int64_t T)
{
    const int64_t tiles = lookback_tiles(N, T);
    return tiles ? (size_t)(kWsHeaderBytes + tiles * kTileStateBytes) : 0;
}

// Bounded wait of the look-back: consecutive empty polls of a later tile (each poll
// sleeps up to 256 ns, so about a second) before the launch reports RLCA_ERR_TIMEOUT.
constexpr int kDefaultSpinLimit = 1 << 22;

// Launch with programmatic stream serialization (PDL); `args` are the kernel's Params.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, const Args &...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Warp-owned whole rows: lanes per row as a shift when a power of two (lane_slot).
inline void set_lane_split(Params &p)
{
    const int c = p.chunks_per_row;
    int k = 0;
    while ((1 << k) < c) ++k;
    p.row_shift1 = (c > 0 && (1 << k) == c) ? k + 1 : 0;
}

// ------------------------------------------------------------------ kernel choice

enum class Path : int { kCtaRows, kCtaRowLoop, kLookback, kWarpRows, kWarpPipe };

constexpr int kMaxDevices = 64;

// SMs of the current device (cached per device; 152 on GB300).
inline int sm_count()
{
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Look-back pays when the rows alone cannot fill the GPU: one CTA per row walking its
// tiles serially leaves SMs idle below about two rows per SM (measured: at [152, 65536]
// look-back is 1.9x faster, at [512, 16384] 1.1x slower, at [2048, 4096] 1.3x slower).
inline bool lookback_pays(int64_t N) { return N < 2 * (int64_t)sm_count(); }

// fp32 inputs (16-bit: launch_estimator_narrow below). Measured on GB300 (CUDA-event timing,
// inputs rotated past L2): rows of at most one warp chunk (256 steps) go to warp-owned
// rows, which need no CTA barrier; up to one CTA tile (1024 steps) the CTA tile kernel,
// which loads a whole row at once, wins for every estimator but GAE with truncation (or
// rows of at most 512 steps): there the dependent load of the truncation values stalls a
// whole CTA, and a warp per row that keeps its next chunk's loads in flight
// (credit_warp_pipe_kernel) is fastest: at [4096, 1024] 12.90 us against 13.90 for a
// per-warp TMA ring of bulk copies (itself 8% faster than the CTA tile there); 7.29 vs
// 8.25 at [4096, 512], 5.38 vs 6.04 at [1024, 1024]. Without truncation the CTA tile
// stays. Longer rows loop over CTA tiles (or use
// look-back with a workspace). Data in pinned host memory take the CTA tiles for GAE
// too (a GAE step at [4096, 1024] over NVLink-C2C: 275 us, at 335 GB/s).
// `aligned`: rows fit for 128-bit access.
template <Est E>
inline Path choose_path(int64_t N, int T, bool aligned, bool lookback, bool trunc, bool host)
{
    if (T > kTile) return lookback && lookback_pays(N) ? Path::kLookback : Path::kCtaRowLoop;
    if (T <= 32 * kItems) return Path::kWarpRows;
    if (E == Est::kGae && (trunc || 2 * T <= kTile) && !host)
        return aligned ? Path::kWarpPipe : Path::kWarpRows;
    return Path::kCtaRows;
}

// ------------------------------------------------------------------ CTA tile paths

// CTAs per SM the CTA tiles ask the register allocator to fit. The tiles were tuned with
// an explicit 1: leaving the request out gives fewer registers but made Retrace's row
// loop 2.3% slower (28.23 vs 27.58 us at [2048, 4096]) and changed nothing else
// measurably. V-trace's tiles need
// 74-96 registers (5-6 CTAs per SM); capped they ran faster: one row per CTA at 7 per
// SM 15.95 vs 16.75 us at [4096, 1024]; packed rows at 7 per SM 16.17 vs 16.87 us at
// [8192, 512]; the row loop at 6 per SM 28.33 vs 31.39 us at [2048, 4096]. Caps gained
// nothing (or lost) for the other estimators.
template <Est E, typename TIn, Tiling TL>
constexpr int cta_min_blocks()
{
    if (E != Est::kVtrace || !std::is_same<TIn, float>::value) return 1;
    return TL == Tiling::kRowLoop ? 6 : (TL == Tiling::kLookback ? 1 : 7);
}

template <Est E, int VEC, bool TRUNC, typename TIn = float>
cudaError_t launch_cta(Params p, Path path, cudaStream_t stream)
{
    if (path == Path::kCtaRows) {
        const int t_pad = (p.T + kItems - 1) / kItems * kItems;
        p.chunks_per_row = t_pad / kItems;
        p.rows_per_tile = kTile / t_pad;
        p.segs = 1;
        const unsigned grid = (unsigned)((p.N + p.rows_per_tile - 1) / p.rows_per_tile);
        if (p.rows_per_tile == 1)
            return launch_pdl(credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kRow,
                                                 cta_min_blocks<E, TIn, Tiling::kRow>(), TIn>,
                              grid, kThreads, 0, stream, p);
        return launch_pdl(credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kRows,
                                             cta_min_blocks<E, TIn, Tiling::kRows>(), TIn>,
                          grid, kThreads, 0, stream, p);
    }
    p.chunks_per_row = kTile / kItems;
    p.rows_per_tile = 1;
    p.segs = (p.T + kTile - 1) / kTile;
    if (path == Path::kLookback)
        return launch_pdl(
            credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kLookback,
                               cta_min_blocks<E, TIn, Tiling::kLookback>(), TIn>,
            (unsigned)(p.N * p.segs), kThreads, 0, stream, p);
    return launch_pdl(credit_scan_kernel<E, kThreads, kItems, VEC, TRUNC, Tiling::kRowLoop,
                                         cta_min_blocks<E, TIn, Tiling::kRowLoop>(), TIn>,
                      (unsigned)p.N, kThreads, 0, stream, p);
}

// ------------------------------------------------------------------ warp paths

// CTAs per SM the warp-owned-rows kernel asks the register allocator to fit (0 = no
// request). V-trace's needs 80 registers (6 CTAs of 4 warps per SM); capped at 28 warps
// per SM (72 registers, 28 bytes of spill) it ran faster on [8192, 256]: 9.16 us
// against 9.72.
template <Est E, typename TIn, int ITEMS>
constexpr int warp_min_blocks()
{
    return (E == Est::kVtrace && std::is_same<TIn, float>::value && ITEMS == kItems)
               ? 28 / kWarpRowsPerCta
               : 0;
}

template <Est E, int VEC, bool TRUNC, typename TIn = float, int ITEMS = kItems>
cudaError_t launch_warp_rows(Params p, cudaStream_t stream)
{
    constexpr int CH = 32 * ITEMS;
    if (ITEMS != kItems) {  // the constant beta to the power of the steps per lane
        const float beta = E == Est::kReturn ? p.gamma : p.gamma_lambda;
        p.beta_pow = beta;
        for (int i = 1; i < ITEMS; ++i) p.beta_pow = beta * p.beta_pow;
    }
    int64_t jobs;
    if (p.T <= CH) {
        const int t_pad = (p.T + ITEMS - 1) / ITEMS * ITEMS;
        p.segs = 1;
        p.chunks_per_row = t_pad / ITEMS;
        p.rows_per_tile = CH / t_pad;
        set_lane_split(p);
        jobs = (p.N + p.rows_per_tile - 1) / p.rows_per_tile;
    } else {
        p.segs = (p.T + CH - 1) / CH;
        p.chunks_per_row = CH / ITEMS;
        p.rows_per_tile = 1;
        jobs = p.N;
    }
    const unsigned grid = (unsigned)((jobs + kWarpRowsPerCta - 1) / kWarpRowsPerCta);
    return launch_pdl(credit_warp_kernel<E, ITEMS, VEC, TRUNC, kWarpRowsPerCta, TIn,
                                         warp_min_blocks<E, TIn, ITEMS>()>,
                      grid, 32 * kWarpRowsPerCta, 0, stream, p);
}

// L2 prefetch of the pipelined warp rows: steps prefetched before the grid dependency
// wait (from the row's end, where the walk starts) and how many chunks ahead of the scan
// a chunk is prefetched inside the walk (0: none), beyond the chunks whose loads the
// registers already hold. Measured on GB300 at [4096, 1024], us per launch, for (before
// the wait, ahead) = (0, 0) / (256, 0) / (256, 2) / (1024, 0) / (0, 2) / (512, 3):
//   GAE fp32 12.86 / 12.30 / 12.76 / 14.29 / 13.23 / 12.94;
//   GAE bf16 10.84 / 10.85 / 12.29 / 12.98 / 12.04 / 11.98;
//   fused TD(lambda), 3 lambdas, 15.63 / 14.82 / 15.08 / 16.49 / 15.72 / 14.39;
//   return bf16 7.79 / 7.50 / 8.28 / 7.10 / 8.49 / 7.35;
//   TD(lambda) bf16 8.58 / 7.76 / 9.04 / 8.15 / 8.98 / 7.96;
//   V-trace bf16 14.78 / 14.43 / 13.88 / 14.00 / 14.29 / 13.62 (two waves of warps then,
//     at 87-90 registers; below 72, see pipe_min_blocks);
//   Retrace bf16 10.26 / 9.30 / 10.30 / 11.15 / 11.40 / 9.21.
// Prefetching whole rows before the wait floods L2 when the whole grid is resident at
// once (one wave: every warp's row requested at the same moment). fp16 inputs move the
// same bytes as bf16 and take its settings.
struct PipePrefetch {
    int first, ahead;
};

template <Est E, typename TIn, bool MULTI = false>
constexpr PipePrefetch pipe_prefetch()
{
    if (MULTI) return {512, 3};
    if (std::is_same<TIn, float>::value) return E == Est::kTdLambda ? PipePrefetch{512, 2}
                                                                    : PipePrefetch{256, 0};
    if (E == Est::kGae || E == Est::kTdLambda) return {256, 0};
    if (E == Est::kReturn) return {1024, 0};
    // V-trace and Retrace; with the 7-CTA cap bf16 V-trace prefers (256, 0): 11.90 vs
    // 12.24 us, while fp16 V-trace (11.84 vs 12.19) and Retrace keep (512, 3).
    if (E == Est::kVtrace && std::is_same<TIn, uint16_t>::value) return {256, 0};
    return {512, 3};
}

// fp32 TD(lambda), alone or fused, keeps its setting only on rows of whole chunks; a
// row that starts with a ragged chunk takes (256, 0). Measured on GB300 at [4096, T], us
// per launch, (256, 0) / (512, 0) / (512, 2) / (512, 3) / (768, 0): TD(lambda) T = 520
// 7.01 / 6.98 / 6.97 / 6.99 / 6.97; 700 8.31 / 9.09 / 9.09 / 9.10 / 9.15; 900 10.20 /
// 10.70 / 10.65 / 10.71 / 11.37; 1024 9.38 / 9.94 / 8.89 / 9.03 / 10.54; fused TD(lambda)
// (256, 0) / (512, 2) / (512, 3): T = 700 12.16 / 12.76 / 12.79, 1024 14.76 / 15.42 /
// 14.34. GAE takes (256, 0) at every one of these lengths (at 700: 11.63 against
// 12.38-12.67 for the others); the 16-bit settings above were confirmed at T = 1024.
template <Est E, typename TIn, bool MULTI = false>
void set_pipe_prefetch(Params &p)
{
    constexpr PipePrefetch pf = pipe_prefetch<E, TIn, MULTI>();
    p.pf_first = pf.first;
    p.pf_ahead = pf.ahead;
    if (E == Est::kTdLambda && std::is_same<TIn, float>::value && p.T % (32 * kItems) != 0) {
        p.pf_first = 256;
        p.pf_ahead = 0;
    }
}

// One row per warp, kItems steps per lane, DEPTH chunks' loads in flight ahead of the
// scan (credit_warp_pipe_kernel). Rows longer than one warp chunk, 16-byte aligned.
// CTAs per SM the register allocator must fit for the pipelined warp rows (0 = no
// request). One warp per row must be resident at once: 4096 rows need 27 warps per SM on
// GB300, 7 CTAs of 4 warps, at most 72 registers. Uncapped, 16-bit V-trace needs 87-90
// registers and fp16 Retrace 78-88 (5-6 CTAs per SM: two waves of warps), so the 16-bit
// rows ask for 7 CTAs per SM (the others fit in 72 registers anyway). fp32 GAE and
// TD(lambda) fit too; a cap was slower for the fused TD(lambda) (its own, in fused.cu).
template <typename TIn>
constexpr int pipe_min_blocks()
{
    return sizeof(TIn) == 2 ? 7 : 0;
}

template <Est E, int VEC, bool TRUNC, int DEPTH, typename TIn = float,
          int MINB = pipe_min_blocks<TIn>()>
cudaError_t launch_warp_pipe(Params p, cudaStream_t stream)
{
    constexpr int CH = 32 * kItems;
    set_pipe_prefetch<E, TIn>(p);
    p.segs = (p.T + CH - 1) / CH;
    p.chunks_per_row = CH / kItems;
    p.rows_per_tile = 1;
    const unsigned grid = (unsigned)((p.N + kWarpsPerCta - 1) / kWarpsPerCta);
    return launch_pdl(
        credit_warp_pipe_kernel<E, kItems, VEC, TRUNC, DEPTH, kWarpsPerCta, TIn, MINB>, grid,
        32 * kWarpsPerCta, 0, stream, p);
}

// ------------------------------------------------------------------ dispatch

// Access widths. Rows that allow 256-bit access (32-byte aligned, access level 2) use
// 256-bit loads and stores (kWideVec) unless measured slower. Data in pinned host memory
// always take the wide access when aligned: over NVLink-C2C it moved a GAE step at 335
// GB/s against 195 GB/s with 128-bit access. Measured on GB300 in device memory, 128-bit
// vs 256-bit loads and stores, in us per launch:
//   warp-owned rows [4096, 128]: return 2.23 vs 2.14, TD(lambda) 2.36 vs 2.26, V-trace
//     3.86 vs 3.48, Retrace 3.37 vs 2.52, GAE 2.97 vs 2.51, fused TD 4.21 vs 3.93;
//   row loop [2048, 4096]: return 15.79 vs 15.43, TD 19.90 vs 19.10, V-trace 32.46 vs
//     31.38, Retrace 30.77 vs 27.63, GAE 24.86 vs 23.51, fused TD 33.82 vs 32.45;
//   one row per CTA [4096, 1024]: return 7.71 vs 7.52, GAE 12.52 vs 12.05, V-trace 16.88
//     vs 16.70, fused TD 17.33 vs 17.11, but TD 10.07 vs 10.16 and the forward scan 8.46
//     vs 8.53, which keep 128-bit access there (Retrace was 15.22 vs 15.36 before the
//     L2 prefetch, 14.42 vs 14.16 with it: 256-bit now);
//   pipelined warp rows, GAE [4096, 1024]: 12.90 with 128-bit access, 13.24 with
//     256-bit, 13.27 with 256-bit loads and 128-bit stores: 128-bit there (with the L2
//     prefetch 12.30 vs 12.78 with 256-bit stores).
// Wide loads alone or wide stores alone were slower than either.
constexpr int kWideVec = kVec16 | kWideLoads | kWideStores;

// Calls f(integral_constant<int, V>, integral_constant<bool, R>) with the access width for
// the run-time level `vec` (0 scalar, 1 128-bit, 2 kWideVec) and the truncation flag.
template <class F>
cudaError_t with_vec_trunc(int vec, bool trunc, F &&f)
{
    using V0 = std::integral_constant<int, 0>;
    using V1 = std::integral_constant<int, kVec16>;
    using V2 = std::integral_constant<int, kWideVec>;
    using R1 = std::true_type;
    using R0 = std::false_type;
    if (vec >= 2) return trunc ? f(V2{}, R1{}) : f(V2{}, R0{});
    if (vec == 1) return trunc ? f(V1{}, R1{}) : f(V1{}, R0{});
    return trunc ? f(V0{}, R1{}) : f(V0{}, R0{});
}

// True when a CTA tile holds exactly one row (TILE / 2 < T <= TILE).
inline bool one_row_per_cta(int T) { return 2 * T > kTile && T <= kTile; }

// Steps per lane of the fp32 warp-owned rows (rows of at most 32 lanes x these steps).
template <Est E>
constexpr int warp_rows_items()
{
    return kItems;
}

// Rows that tile one warp chunk (256 steps: one row, or 2 or 4 contiguous rows of 128 or
// 64 steps), more such jobs than one wave of warps holds: one wave of warps walking the
// jobs with the next job's loads in flight (credit_warp_rows_pipe_kernel), sized from the
// kernel's occupancy. Measured on GB300, us per launch, walked vs warp-owned rows in
// waves: [8192, 256] return 4.22 vs 4.92, TD(lambda) 4.86 vs 5.75, GAE 7.10 vs 8.61;
// [16384, 128] return 4.33 vs 4.99, TD(lambda) 4.86 vs 5.76, GAE 7.02 vs 8.40; [32768, 64]
// return 4.48 vs 5.06. V-trace 11.84 vs 8.14 (its raw chunk does not fit
// the 72 registers of its cap) and Retrace 7.92 vs 7.82 keep the waves. Jobs that fit
// one wave gain nothing: half the warps walking two jobs each took return [4096, 128]
// from 2.19 to 2.91 us.
template <Est E>
constexpr bool walk_rows_when_many()
{
    return E == Est::kReturn || E == Est::kTdLambda || E == Est::kGae;
}

template <Est E, int VEC, bool TRUNC, typename TIn = float>
cudaError_t launch_warp_rows_pipe(Params p, cudaStream_t stream, bool *launched)
{
    constexpr int W = kWarpRowsPerCta;
    constexpr int MINB = warp_min_blocks<E, TIn, kItems>();
    auto kernel = credit_warp_rows_pipe_kernel<E, kItems, VEC, TRUNC, W, TIn, MINB>;
    static std::atomic<int> per_sm_cache{0};
    int per_sm = per_sm_cache.load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * W, 0) !=
                cudaSuccess || per_sm <= 0) {
            (void)cudaGetLastError();
            *launched = false;
            return cudaSuccess;
        }
        per_sm_cache.store(per_sm, std::memory_order_relaxed);
    }
    const int64_t wave = (int64_t)per_sm * sm_count();  // CTAs resident at once
    const int rpt = 32 * kItems / p.T;                  // rows per job
    const int64_t ctas = (p.N / rpt + W - 1) / W;
    if (ctas <= wave) {  // one wave already: nothing to walk
        *launched = false;
        return cudaSuccess;
    }
    p.segs = 1;
    p.chunks_per_row = p.T / kItems;
    p.rows_per_tile = rpt;
    set_lane_split(p);
    *launched = true;
    return launch_pdl(kernel, (unsigned)wave, 32 * W, 0, stream, p);
}

template <Est E, int VEC, bool TRUNC>
cudaError_t launch_path(const Params &p, Path path, cudaStream_t stream)
{
    if constexpr (walk_rows_when_many<E>() && (VEC & kVec16) != 0) {
        // Jobs of whole contiguous rows: T divides the warp chunk, rows packed when
        // several share a job (ld == T), N a multiple of the rows per job.
        const bool tiles = p.T == 32 * kItems ||
                           ((p.T == 16 * kItems || p.T == 8 * kItems) && p.ld == p.T &&
                            p.N % (32 * kItems / p.T) == 0);
        if (path == Path::kWarpRows && tiles && !p.host) {
            bool launched = false;
            const cudaError_t err = launch_warp_rows_pipe<E, VEC, TRUNC>(p, stream, &launched);
            if (launched || err != cudaSuccess) return err;
        }
    }
    if (path == Path::kWarpRows) {
        constexpr int I = warp_rows_items<E>();
        if (I != kItems && p.T <= 32 * I)
            return launch_warp_rows<E, VEC, TRUNC, float, I>(p, stream);
        return launch_warp_rows<E, VEC, TRUNC>(p, stream);
    }
    return launch_cta<E, VEC, TRUNC>(p, path, stream);
}

// beta^kItems in the order the kernels multiply (b = beta * b), for the constant-beta
// estimators' per-thread composite.
template <Est E>
void set_beta_pow(Params &p)
{
    const float beta = E == Est::kReturn ? p.gamma : p.gamma_lambda;
    p.beta_pow = beta;
    for (int i = 1; i < kItems; ++i) p.beta_pow = beta * p.beta_pow;
}

// 16-bit per-step inputs (TIn: uint16_t bf16 bit patterns or __half; fp32 arithmetic).
// The two formats move the same bytes and take the same kernels. Measured on GB300 at
// [4096, 1024], us per launch, the tiles below against a warp per row with its next
// chunks' loads in flight (credit_warp_pipe_kernel): GAE 14.15 vs 10.84, TD(lambda)
// 10.64 vs 8.38, V-trace 20.95 vs 14.32, Retrace 15.33 vs 10.24, return 7.86 vs 7.69;
// GAE at [16384, 512] 28.33 vs 20.32. So rows longer than two warp chunks (GAE: one)
// up to one CTA tile take the pipelined warp rows, with two chunks in flight (one for
// V-trace and Retrace, whose larger raw chunks then keep one wave of warps resident:
// 14.32 vs 14.59 and 10.24 vs 12.55) and 64-bit flag loads where rows are 32-byte
// aligned (256-bit stores: GAE 12.77 vs 10.84). Otherwise warp-owned rows up to one
// warp chunk, CTA tiles (whole rows or the row loop) beyond; GAE rows longer than a warp
// chunk go to warp-owned rows with 16 steps per lane there.
template <Est E, typename TIn>
cudaError_t launch_estimator_narrow(const Params &p_in, int vec, cudaStream_t stream)
{
    static_assert(sizeof(TIn) == 2, "16-bit inputs");
    Params p = p_in;
    set_beta_pow<E>(p);
    const bool trunc = p.trunc != nullptr;
    // The 16-bit discounted return keeps CTA rows up to one tile: with the L2 prefetch
    // and 256-bit output stores they beat its pipelined warp rows at [4096, 1024] (bf16
    // 6.48 vs 7.08 us, fp16 6.45 vs 6.89); the other estimators lost there (TD(lambda)
    // 9.52 vs 7.86, GAE 14.0 vs 10.9, V-trace 15.2 vs 13.9, Retrace 12.6 vs 9.2, bf16).
    const int pipe_from = E == Est::kGae ? 32 * kItems : (E == Est::kReturn ? kTile : 64 * kItems);
    if (!p.host && vec >= 1 && p.T > pipe_from && p.T <= kTile) {
        constexpr int D = (E == Est::kVtrace || E == Est::kRetrace) ? 1 : 2;
        constexpr int kFlags64 = kVec16 | kWideLoads;
        if (vec >= 2)
            return trunc ? launch_warp_pipe<E, kFlags64, true, D, TIn>(p, stream)
                         : launch_warp_pipe<E, kFlags64, false, D, TIn>(p, stream);
        return trunc ? launch_warp_pipe<E, kVec16, true, D, TIn>(p, stream)
                     : launch_warp_pipe<E, kVec16, false, D, TIn>(p, stream);
    }
    // 16-bit data loads stay 128-bit; wide flag loads and output stores were measured
    // slower for bf16 GAE at [4096, 1024] (14.63 vs 14.25 us), so 128-bit throughout in
    // device memory, except the return's CTA rows (6.48 vs 6.74 us, bf16).
    if (!p.host && !(E == Est::kReturn && p.T > 32 * kItems)) vec = vec < 1 ? vec : 1;
    if constexpr (E == Est::kGae) {
        if (p.T > 32 * kItems) {  // 16 steps per lane
            return with_vec_trunc(vec, trunc, [&](auto v, auto r) {
                return launch_warp_rows<E, decltype(v)::value, decltype(r)::value, TIn,
                                        16>(p, stream);
            });
        }
    }
    const Path path = p.T <= 32 * kItems ? Path::kWarpRows
                                         : (p.T > kTile ? Path::kCtaRowLoop : Path::kCtaRows);
    return with_vec_trunc(vec, trunc, [&](auto v, auto r) {
        constexpr int V = decltype(v)::value;
        constexpr bool R = decltype(r)::value;
        if (path == Path::kWarpRows) return launch_warp_rows<E, V, R, TIn>(p, stream);
        return launch_cta<E, V, R, TIn>(p, path, stream);
    });
}

// fp32 estimators other than GAE on rows of 513-1024 steps (one row per CTA tile): the
// pipelined warp rows with this many chunks in flight instead of the CTA tile (0: the
// CTA tile). Measured on GB300 at [4096, 1024] with the L2 prefetch, us per launch, CTA
// tile / one chunk in flight (256 steps before the wait) / two chunks / one chunk
// (512 steps before the wait, 3 chunks ahead): return 6.84 / 7.82 / 7.78 / 7.43;
// TD(lambda) 10.14 / 9.52 / 11.93 / 9.34; V-trace 14.88 / 16.80 / 16.80 / 16.87;
// Retrace 14.48 / 15.53 / 15.56 / 16.69.
template <Est E>
constexpr int fp32_row_pipe_depth()
{
    return E == Est::kTdLambda ? 1 : 0;
}

// Launch one estimator; `vec` = access level (0 scalar, 1 16-byte aligned rows with
// 128-bit access, 2 32-byte aligned rows fit for 256-bit access).
template <Est E>
cudaError_t launch_estimator(const Params &p_in, int vec, cudaStream_t stream)
{
    Params p = p_in;
    set_beta_pow<E>(p);
    const bool trunc = p.trunc != nullptr;
    const Path path = choose_path<E>(p.N, p.T, vec >= 1, p.ws != nullptr, trunc, p.host);
    if constexpr (E == Est::kGae) {
        if (path == Path::kWarpPipe)
            return trunc ? launch_warp_pipe<E, kVec16, true, 1>(p, stream)
                         : launch_warp_pipe<E, kVec16, false, 1>(p, stream);
    } else if constexpr (fp32_row_pipe_depth<E>() > 0) {
        if (path == Path::kCtaRows && one_row_per_cta(p.T) && vec >= 1 && !p.host) {
            constexpr int D = fp32_row_pipe_depth<E>();
            return trunc ? launch_warp_pipe<E, kVec16, true, D>(p, stream)
                         : launch_warp_pipe<E, kVec16, false, D>(p, stream);
        }
    } else if constexpr (E == Est::kReturn) {
        // Rows of 513-960 steps that one wave of 7 CTAs of 4 warps per SM holds: the
        // pipelined warp rows with two chunks in flight under that cap beat the CTA row,
        // whose threads past the row's end idle. Measured on GB300, us per launch, CTA
        // row vs pipelined rows at [4096, T]: T = 520 5.89 vs 5.24, 600 6.06 vs 5.40, 700
        // 6.92 vs 6.13, 768 5.80 vs 5.17, 900 7.95 vs 7.53, 1000 7.79 vs 8.01, 1024 6.66
        // vs 7.11; [2048, 600] 4.69 vs 4.36, [2048, 1024] 3.76 vs 5.14.
        constexpr int kCap = 7;
        if (path == Path::kCtaRows && one_row_per_cta(p.T) && p.T <= 960 && vec >= 1 &&
            !p.host && (p.N + kWarpsPerCta - 1) / kWarpsPerCta <= (int64_t)kCap * sm_count())
            return trunc ? launch_warp_pipe<E, kVec16, true, 2, float, kCap>(p, stream)
                         : launch_warp_pipe<E, kVec16, false, 2, float, kCap>(p, stream);
    }
    // TD(lambda) keeps 128-bit access on a CTA row (measured 10.07 vs 10.16 us at
    // [4096, 1024]); it takes the CTA row only without 16-byte aligned rows now.
    // Retrace moved to 256-bit with the L2 prefetch: 14.16 vs 14.42 us, and every output
    // sector written whole (1.19x the output bytes reached L2 with 128-bit stores).
    if (E == Est::kTdLambda && path == Path::kCtaRows && one_row_per_cta(p.T) && !p.host)
        vec = vec < 1 ? vec : 1;
    return with_vec_trunc(vec, trunc, [&](auto v, auto r) {
        return launch_path<E, decltype(v)::value, decltype(r)::value>(p, path, stream);
    });
}

// Input formats of the per-step data (rewards, values, ratios, truncation values, x).
enum class Fmt : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

template <Fmt F>
struct FmtType;
template <>
struct FmtType<Fmt::kF32> {
    using type = float;
};
template <>
struct FmtType<Fmt::kBF16> {
    using type = uint16_t;  // bf16 bit patterns
};
template <>
struct FmtType<Fmt::kF16> {
    using type = __half;
};

// One estimator in one input format. Each (E, F) pair is instantiated in a translation
// unit of its own (reverse_unit.cu, compiled once per pair) so the library builds in
// parallel; the callers see only this declaration.
template <Est E, Fmt F>
cudaError_t launch_unit(const Params &p, int vec, cudaStream_t stream);

template <Est E>
cudaError_t launch_in_format(Fmt f, const Params &p, int vec, cudaStream_t stream)
{
    if (f == Fmt::kBF16) return launch_unit<E, Fmt::kBF16>(p, vec, stream);
    if (f == Fmt::kF16) return launch_unit<E, Fmt::kF16>(p, vec, stream);
    return launch_unit<E, Fmt::kF32>(p, vec, stream);
}

// Forward scans in one input format (forward_unit.cu, compiled once per format):
// p.reward = x, p.boot = carried-in values, p.gamma = decay, p.out0 = output.
template <Fmt F>
cudaError_t launch_forward_unit(const Params &p, int vec, cudaStream_t stream);

inline cudaError_t launch_forward_in_format(Fmt f, const Params &p, int vec,
                                            cudaStream_t stream)
{
    if (f == Fmt::kBF16) return launch_forward_unit<Fmt::kBF16>(p, vec, stream);
    if (f == Fmt::kF16) return launch_forward_unit<Fmt::kF16>(p, vec, stream);
    return launch_forward_unit<Fmt::kF32>(p, vec, stream);
}

// Fused calls (fused.cu; fp32 inputs). TD(lambda) for p.multi.count lambdas (outputs in
// p.multi.out); GAE (parameters and outputs in pg) and V-trace (pv) from one load.
cudaError_t launch_td_multi(const Params &p, int vec, cudaStream_t stream);
cudaError_t launch_gae_vtrace(const Params &pg, const Params &pv, int vec, cudaStream_t stream);

// GAE with the checks of rlca_gae_ex on a workspace the library owns (ws_bytes at ws);
// `prepare` runs after every check has passed, right before the launch, and only when
// the call takes the look-back path (it clears what must start at zero). Returns an
// RLCA status code.
int gae_on_library_workspace(const float *reward, const float *value, const uint8_t *terminated,
                             const uint8_t *truncated, const float *trunc_value,
                             const float *bootstrap, float gamma, float lambda, int64_t N,
                             int64_t T, int64_t ld, float *advantages, float *returns,
                             void *ws, size_t ws_bytes,
                             cudaError_t (*prepare)(void *ws, cudaStream_t stream), void *stream);

}  // namespace rlca
