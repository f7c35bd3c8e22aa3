// Per-estimator operand builders and epilogues (Method section 2 of "rl-triton:
// High-Performance Triton GPU Kernels for Reinforcement Learning Credit Assignment":
// the recurrence coefficients are formed in registers straight from the raw rollout
// inputs and are never written to memory).
//
// Each thread owns ITEMS consecutive steps t0 .. t0+ITEMS-1 of one env row. For every
// step it forms (alpha_t, beta_t) of A_t = alpha_t + beta_t * A_{t+1}, with beta < 0
// marking a reset (scan_core.cuh):
//
//   estimator   alpha_t                                       beta_t          output
//   return      r_t (+ gamma * sv_t if the episode stops)     gamma           G = A
//   TD(lambda)  r_t + gamma(1-lambda) V_{t+1}  | r_t+gamma sv  gamma lambda    G = A
//   GAE         r_t + gamma V(s_{t+1}) - V_t                  gamma lambda    adv = A,
//                                                                             ret = A + V
//   V-trace     rho_hat_t (r_t + gamma V(s_{t+1}) - V_t)     gamma c_t       vs = V + A
//   Retrace     r_t + gamma EQ(s_{t+1}) - Q_t                 gamma c_{t+1}   Q^ret = A + Q
//
// where sv_t (successor value, Method section 3) is 0 for a terminated step, the
// supplied truncation value for a truncated one and the per-env bootstrap at t = T-1;
// V(s_{t+1}) / EQ(s_{t+1}) is V_{t+1} / E_pi Q_{t+1} inside an episode and sv_t at its
// last step, where the step resets. Every step is first built as if its episode went
// on; the few steps where an episode stops are then patched.
#pragma once

#include "scan_core.cuh"

namespace rlca {

enum class Est : int { kReturn = 0, kTdLambda = 1, kGae = 2, kVtrace = 3, kRetrace = 4 };

// Fused TD(lambda) for several lambdas from one read of the inputs (at most 4).
constexpr int kMaxLambdas = 4;
struct MultiLambda {
    int count;
    float gamma_lambda[kMaxLambdas];
    float gamma_one_m_lambda[kMaxLambdas];
    float beta_pow[kMaxLambdas];
    float *out[kMaxLambdas];
};

// Kernel arguments, passed by value.
struct Params {
    const float *reward;
    const float *value;  // V (TD, GAE, V-trace) or Q(s_t, a_t) (Retrace)
    const float *aux;    // log importance ratios (V-trace) or E_pi Q(s_t, .) (Retrace)
    const float *rho;    // importance ratios (Retrace)
    const uint8_t *term;
    const uint8_t *trunc;
    const float *trunc_value;
    const float *boot;
    float *out0;
    float *out1;  // nullable
    int64_t N;
    int64_t ld;
    int T;
    float gamma;
    float lambda;
    float gamma_lambda;        // gamma * lambda, rounded to fp32
    float gamma_one_m_lambda;  // gamma * (1 - lambda), rounded to fp32
    float beta_pow;            // the constant beta to the power of the steps per thread
    float rho_bar;
    float c_bar;
    float pg_rho_bar;
    // Geometry of the launch (see kernels.cuh).
    int rows_per_tile;
    int chunks_per_row;
    int row_shift1;  // log2(chunks_per_row) + 1 when that is a power of two, else 0
    int segs;
    // Decoupled look-back across the tiles of a row (kernels.cuh, Tiling::kLookback).
    void *ws;         // caller-owned workspace: header + one 32-byte state per tile
    int spin_limit;   // consecutive empty polls of a later tile before giving up
    int stall;        // testing only: nonzero = tiles never publish their state
    int forward;      // host-side only: a forward scan (truncation needs no values)
    int host;         // some data live in pinned host memory (picks the kernel)
    int prefetch;     // every buffer is plain device memory: L2 prefetches allowed
    int pf_first;     // pipelined warp rows: steps prefetched into L2 before the wait
    int pf_ahead;     // pipelined warp rows: chunk s - pf_ahead prefetched at chunk s (0: off)
    MultiLambda multi;  // fused TD(lambda) only
};

template <Est E>
struct EstTraits {
    static constexpr bool kValue = E != Est::kReturn;
    static constexpr bool kAux = E == Est::kVtrace || E == Est::kRetrace;
    static constexpr bool kRho = E == Est::kRetrace;
    static constexpr bool kNextValue =
        E == Est::kTdLambda || E == Est::kGae || E == Est::kVtrace;
    static constexpr bool kNextAux = E == Est::kRetrace;
    static constexpr bool kNextRho = E == Est::kRetrace;
    static constexpr bool kTwoOutputs = E == Est::kGae || E == Est::kVtrace;
    // beta_t is the same at every step that does not reset (gamma or gamma*lambda).
    static constexpr bool kConstBeta =
        E == Est::kReturn || E == Est::kTdLambda || E == Est::kGae;
};

// Raw inputs of one thread's ITEMS steps, plus the successor (step t0+ITEMS) of the
// arrays whose next step an estimator reads.
template <int ITEMS>
struct Chunk {
    float r[ITEMS];
    float v[ITEMS];
    float x[ITEMS];
    float y[ITEMS];
    float sv[ITEMS];  // successor value where the episode stops (V-trace keeps it)
    float v_next, x_next, y_next;
    float boot_v;    // the per-env bootstrap if the thread holds the row's last step, else 0
    bool boot_late;  // boot_v unset: build() reads the bootstrap once the flags are in
    unsigned stop;   // bit j: the recursion stops at step j (boundary or padding)
    unsigned term;   // bit j: step j terminated
    unsigned trunc;  // bit j: step j truncated
    unsigned valid;  // bit j: step t0+j exists in this row
};

// Row `off` of a per-step input array holding TIn elements (the Params pointers are
// typed fp32; bf16 inputs are stored behind them as uint16_t bit patterns).
template <typename TIn>
__device__ __forceinline__ const TIn *in_row(const float *base, int64_t off)
{
    return reinterpret_cast<const TIn *>(base) + off;
}

// Columns [t_lo, t_hi) of one row of every per-step array estimator E streams in (data
// and flags; the sparse truncation values are left out) prefetched into L2. A kernel
// issues this before its grid dependency wait, so the reads of its first rows overlap
// the tail of the previous kernel in the stream. Only when every buffer is plain device
// memory (not pinned host or managed memory).
template <Est E, bool TRUNC, typename TIn = float>
__device__ __forceinline__ void prefetch_row(const Params &p, int64_t row, int t_lo, int t_hi)
{
    using Tr = EstTraits<E>;
    if (!p.prefetch || row >= p.N || t_hi <= t_lo) return;
    const int64_t off = row * p.ld + t_lo;
    const int64_t n = t_hi - t_lo;
    prefetch_l2(in_row<TIn>(p.reward, off), n * (int64_t)sizeof(TIn));
    if (Tr::kValue) prefetch_l2(in_row<TIn>(p.value, off), n * (int64_t)sizeof(TIn));
    if (Tr::kAux) prefetch_l2(in_row<TIn>(p.aux, off), n * (int64_t)sizeof(TIn));
    if (Tr::kRho) prefetch_l2(in_row<TIn>(p.rho, off), n * (int64_t)sizeof(TIn));
    prefetch_l2(p.term + off, n);
    if (TRUNC) prefetch_l2(p.trunc + off, n);
}

// Successor of item ITEMS-1: the next lane's first item, or (lane 31) a direct load.
// Every lane of the warp must call this (it shuffles).
template <typename TIn = float>
__device__ __forceinline__ float next_item(float first_item, const TIn *__restrict__ row,
                                           int t_next, bool need, int lane)
{
    float s = __shfl_down_sync(kFullMask, first_item, 1);
    if (lane == 31) s = need ? InType<TIn>::cached(row + t_next) : 0.f;
    return need ? s : 0.f;
}

// The per-env bootstrap (successor value at the window end, Method section 3) for a
// thread whose items t0 .. t0+ITEMS-1 hold the row's last step, else 0. Its address needs
// no loaded data, so it is read together with the chunk's data instead of after the
// chunk's flags arrive (that would put a second memory latency on the thread's path).
template <int ITEMS>
__device__ __forceinline__ float load_boot(const Params &p, int64_t row, int t0, bool active)
{
    const int last = p.T - 1 - t0;
    return (active && p.boot && last >= 0 && last < ITEMS) ? __ldg(p.boot + row) : 0.f;
}

// EARLY_BOOT: the bootstrap is read with the data (load_boot); else build() reads it
// where it is used, once the chunk's flags are in (a second memory latency on the
// thread's path, but no register held from the load to the use).
template <Est E, int ITEMS, int VEC, bool TRUNC, typename TIn = float, bool EARLY_BOOT = true>
__device__ __forceinline__ void load_chunk(const Params &p, int64_t row, int t0, bool active,
                                           int lane, Chunk<ITEMS> &c)
{
    using Tr = EstTraits<E>;
    const int T = p.T;
    const int Te = active ? T : 0;  // an inactive thread sees an empty row
    const int64_t off = active ? row * p.ld : 0;

    c.boot_v = EARLY_BOOT ? load_boot<ITEMS>(p, row, t0, active) : 0.f;
    c.boot_late = !EARLY_BOOT;
    load_items<ITEMS, VEC, TIn>(in_row<TIn>(p.reward, off), t0, Te, c.r);
    if (Tr::kValue) load_items<ITEMS, VEC, TIn>(in_row<TIn>(p.value, off), t0, Te, c.v);
    if (Tr::kAux) load_items<ITEMS, VEC, TIn>(in_row<TIn>(p.aux, off), t0, Te, c.x);
    if (Tr::kRho) load_items<ITEMS, VEC, TIn>(in_row<TIn>(p.rho, off), t0, Te, c.y);
    c.term = load_flag_bits<ITEMS, VEC>(p.term + off, t0, Te);
    c.trunc = TRUNC ? load_flag_bits<ITEMS, VEC>(p.trunc + off, t0, Te) : 0u;
    c.valid = valid_items<ITEMS>(t0, Te);
    const int last = T - 1 - t0;
    const unsigned window_end = (last >= 0 && last < ITEMS) ? (1u << last) : 0u;
    c.stop = (c.term | c.trunc | window_end | ~c.valid) & all_items<ITEMS>();

    const bool need = active && (t0 + ITEMS < T);
    if (Tr::kNextValue)
        c.v_next = next_item<TIn>(c.v[0], in_row<TIn>(p.value, off), t0 + ITEMS, need, lane);
    if (Tr::kNextAux)
        c.x_next = next_item<TIn>(c.x[0], in_row<TIn>(p.aux, off), t0 + ITEMS, need, lane);
    if (Tr::kNextRho)
        c.y_next = next_item<TIn>(c.y[0], in_row<TIn>(p.rho, off), t0 + ITEMS, need, lane);
}

// The raw 32-bit words of one thread's ITEMS steps of every array an estimator reads,
// held in registers between their load and their use, so a warp can ask for the next
// chunk's words before it scans the current one. Full, aligned chunks only (each array's
// words fill whole 128-bit loads).
template <Est E, int ITEMS, typename TIn>
struct RawChunk {
    using Tr = EstTraits<E>;
    static constexpr int kWords = ITEMS * (int)sizeof(TIn) / 4;
    static_assert(kWords % 4 == 0, "a thread's items fill whole 128-bit loads");
    uint32_t r[kWords];
    uint32_t v[Tr::kValue ? kWords : 1];
    uint32_t x[Tr::kAux ? kWords : 1];
    uint32_t y[Tr::kRho ? kWords : 1];
    uint32_t term[ITEMS / 4];
    uint32_t trunc[ITEMS / 4];
    float v_next, x_next, y_next;  // thread 31 of a warp: the next chunk's first step
};

// kWords words of one row from column t0 (VEC bit 1: 256-bit loads, else 128-bit).
template <int kWords, int VEC, typename TIn>
__device__ __forceinline__ void load_words(const TIn *__restrict__ row, int t0,
                                           uint32_t (&w)[kWords])
{
    const uint32_t *src = reinterpret_cast<const uint32_t *>(row + t0);
    if constexpr ((VEC & kWideLoads) && kWords % 8 == 0) {
#pragma unroll
        for (int k = 0; k < kWords / 8; ++k) {
            float f[8];
            ld_stream8(reinterpret_cast<const float *>(src) + 8 * k, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) w[8 * k + i] = __float_as_uint(f[i]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < kWords / 4; ++k) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(src) + k);
            w[4 * k] = q.x;
            w[4 * k + 1] = q.y;
            w[4 * k + 2] = q.z;
            w[4 * k + 3] = q.w;
        }
    }
}

// The flag bytes of ITEMS steps as ITEMS / 4 words (VEC bit 1: 64-bit loads).
template <int ITEMS, int VEC>
__device__ __forceinline__ void load_flag_words(const uint8_t *__restrict__ row, int t0,
                                                uint32_t (&w)[ITEMS / 4])
{
    if constexpr ((VEC & kWideLoads) && ITEMS % 8 == 0) {
#pragma unroll
        for (int k = 0; k < ITEMS / 8; ++k) {
            const uint2 q = ld_stream(reinterpret_cast<const uint2 *>(row + t0) + k);
            w[2 * k] = q.x;
            w[2 * k + 1] = q.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < ITEMS / 4; ++k)
            w[k] = ld_stream(reinterpret_cast<const uint32_t *>(row + t0) + k);
    }
}

// Issue the loads of one full chunk of a row (thread's first step t0, t0 + ITEMS <= T).
// Thread 31 also reads the next chunk's first step, if the row has one.
template <Est E, int ITEMS, int VEC, bool TRUNC, typename TIn>
__device__ __forceinline__ void load_raw(const Params &p, int64_t off, int t0, int lane,
                                         RawChunk<E, ITEMS, TIn> &w)
{
    using Tr = EstTraits<E>;
    constexpr int kW = RawChunk<E, ITEMS, TIn>::kWords;
    load_words<kW, VEC>(in_row<TIn>(p.reward, off), t0, w.r);
    if constexpr (Tr::kValue) load_words<kW, VEC>(in_row<TIn>(p.value, off), t0, w.v);
    if constexpr (Tr::kAux) load_words<kW, VEC>(in_row<TIn>(p.aux, off), t0, w.x);
    if constexpr (Tr::kRho) load_words<kW, VEC>(in_row<TIn>(p.rho, off), t0, w.y);
    load_flag_words<ITEMS, VEC>(p.term + off, t0, w.term);
    if constexpr (TRUNC) load_flag_words<ITEMS, VEC>(p.trunc + off, t0, w.trunc);
    const int tn = t0 + ITEMS;
    if (lane == 31 && tn < p.T) {
        if constexpr (Tr::kNextValue) w.v_next = InType<TIn>::cached(in_row<TIn>(p.value, off) + tn);
        if constexpr (Tr::kNextAux) w.x_next = InType<TIn>::cached(in_row<TIn>(p.aux, off) + tn);
        if constexpr (Tr::kNextRho) w.y_next = InType<TIn>::cached(in_row<TIn>(p.rho, off) + tn);
    }
}

template <typename TIn, int ITEMS, int kWords>
__device__ __forceinline__ void widen_words(const uint32_t (&w)[kWords], float (&x)[ITEMS])
{
    constexpr int PV = InType<TIn>::kPerVec;
#pragma unroll
    for (int k = 0; k < ITEMS / PV; ++k)
        InType<TIn>::unpack(make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]),
                            x + PV * k);
}

// A full chunk's Chunk from its raw words (what load_chunk forms from its loads);
// boot_v: load_boot of the thread's items, read when the raw words were requested.
// Every thread of the warp must call this (it shuffles).
template <Est E, int ITEMS, bool TRUNC, typename TIn>
__device__ __forceinline__ void unpack_raw(const RawChunk<E, ITEMS, TIn> &w, int T, int t0,
                                           int lane, float boot_v, Chunk<ITEMS> &c)
{
    using Tr = EstTraits<E>;
    c.boot_v = boot_v;
    c.boot_late = false;
    widen_words<TIn>(w.r, c.r);
    if constexpr (Tr::kValue) widen_words<TIn>(w.v, c.v);
    if constexpr (Tr::kAux) widen_words<TIn>(w.x, c.x);
    if constexpr (Tr::kRho) widen_words<TIn>(w.y, c.y);
    unsigned term = 0, trunc = 0;
#pragma unroll
    for (int k = 0; k < ITEMS / 4; ++k) {
        term |= nonzero_bytes(w.term[k]) << (4 * k);
        if constexpr (TRUNC) trunc |= nonzero_bytes(w.trunc[k]) << (4 * k);
    }
    c.term = term;
    c.trunc = trunc;
    c.valid = all_items<ITEMS>();
    const int last = T - 1 - t0;
    const unsigned window_end = (last >= 0 && last < ITEMS) ? (1u << last) : 0u;
    c.stop = (term | trunc | window_end) & all_items<ITEMS>();
    const bool need = t0 + ITEMS < T;  // false only for the row's last thread
    if constexpr (Tr::kNextValue) {
        const float s = __shfl_down_sync(kFullMask, c.v[0], 1);
        c.v_next = need ? (lane == 31 ? w.v_next : s) : 0.f;
    }
    if constexpr (Tr::kNextAux) {
        const float s = __shfl_down_sync(kFullMask, c.x[0], 1);
        c.x_next = need ? (lane == 31 ? w.x_next : s) : 0.f;
    }
    if constexpr (Tr::kNextRho) {
        const float s = __shfl_down_sync(kFullMask, c.y[0], 1);
        c.y_next = need ? (lane == 31 ? w.y_next : s) : 0.f;
    }
}

template <int ITEMS>
__device__ __forceinline__ float at_or_next(const float (&a)[ITEMS], float next, int j)
{
    return (j + 1 < ITEMS) ? a[j + 1] : next;
}

// Forms (alpha, beta) of every item: one select picks the value of the state after the
// step (the next step's value inside an episode, the successor value where it stops),
// one picks beta or the reset marker. Successor values that need a load (truncated
// steps, and the window end where its bootstrap was not read with the data, boot_late)
// are fetched in a branch that few threads take.
// V-trace keeps rho_t in c.x for the epilogue.
template <Est E, int ITEMS, typename TIn = float>
__device__ __forceinline__ void build(const Params &p, int64_t row, int t0, Chunk<ITEMS> &c,
                                      Affine (&e)[ITEMS])
{
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) c.sv[j] = 0.f;
    // Steps whose successor value is loaded (Method section 3): truncated -> the supplied
    // truncation value (read only there), window end -> the per-env bootstrap.
    const unsigned load_sv = c.stop & c.valid & ~c.term;
    if (load_sv) {
        const int64_t off = row * p.ld;
#pragma unroll
        for (int j = 0; j < ITEMS; ++j)
            if (load_sv & (1u << j))
                c.sv[j] = (c.trunc & (1u << j))
                              ? InType<TIn>::cached(in_row<TIn>(p.trunc_value, off) + t0 + j)
                              : c.boot_late ? (p.boot ? __ldg(p.boot + row) : 0.f)
                                            : c.boot_v;
    }
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        const bool stop = (c.stop >> j) & 1u;
        const float r = c.r[j];
        if (E == Est::kReturn) {
            e[j] = Affine{fmaf(p.gamma, c.sv[j], r), 0.f};  // beta: const_beta + stop bit
        } else if (E == Est::kTdLambda) {
            const float nxt = stop ? c.sv[j] : at_or_next(c.v, c.v_next, j);
            e[j] = Affine{fmaf(stop ? p.gamma : p.gamma_one_m_lambda, nxt, r), 0.f};
        } else if (E == Est::kGae) {
            const float nxt = stop ? c.sv[j] : at_or_next(c.v, c.v_next, j);
            e[j] = Affine{fmaf(p.gamma, nxt, r) - c.v[j], 0.f};
        } else if (E == Est::kVtrace) {
            const float rho = expf(c.x[j]);
            c.x[j] = rho;
            const float rho_hat = rho < p.rho_bar ? rho : p.rho_bar;
            const float cmin = rho < p.c_bar ? rho : p.c_bar;
            const float nxt = stop ? c.sv[j] : at_or_next(c.v, c.v_next, j);
            const float delta = fmaf(p.gamma, nxt, r) - c.v[j];
            c.sv[j] = delta;  // the policy-gradient target reuses the TD error
            e[j] = Affine{rho_hat * delta, stop ? kResetB : p.gamma_lambda * cmin};
        } else {  // Retrace: beta_t uses the trace of step t+1
            const float rho1 = at_or_next(c.y, c.y_next, j);
            const float c1 = p.lambda * (rho1 < 1.f ? rho1 : 1.f);
            const float nxt = stop ? c.sv[j] : at_or_next(c.x, c.x_next, j);
            e[j] = Affine{fmaf(p.gamma, nxt, r) - c.v[j], stop ? kResetB : p.gamma * c1};
        }
    }
}

// The constant beta of the constant-beta estimators.
template <Est E>
__device__ __forceinline__ float const_beta(const Params &p)
{
    return E == Est::kReturn ? p.gamma : p.gamma_lambda;
}

// A at item j from A at item j+1 (x). With a constant beta the reset test reads the stop
// bit and the multiplier is the scalar beta, so per-item betas are never formed.
template <Est E, int ITEMS>
__device__ __forceinline__ float step_apply(const Params &p, const Chunk<ITEMS> &c,
                                            const Affine (&e)[ITEMS], int j, float x)
{
    if (EstTraits<E>::kConstBeta)
        return ((c.stop >> j) & 1u) ? e[j].a : fmaf(const_beta<E>(p), x, e[j].a);
    return affine_apply(e[j], x);
}

// Composite of a thread's items, e_0 (+) e_1 (+) ... (+) e_{ITEMS-1}. With a constant
// beta the composite beta is beta^ITEMS, or a reset if any item resets.
template <Est E, int ITEMS>
__device__ __forceinline__ Affine thread_aggregate(const Params &p, const Chunk<ITEMS> &c,
                                                   const Affine (&e)[ITEMS])
{
    float a = e[ITEMS - 1].a;
#pragma unroll
    for (int j = ITEMS - 2; j >= 0; --j) a = step_apply<E, ITEMS>(p, c, e, j, a);
    float b;
    if (EstTraits<E>::kConstBeta) {
        b = c.stop ? kResetB : p.beta_pow;
    } else {
        b = e[ITEMS - 1].b;
#pragma unroll
        for (int j = ITEMS - 2; j >= 0; --j) b = is_reset(e[j].b) ? e[j].b : e[j].b * b;
    }
    return Affine{a, b};
}

// Every A_t of the thread's items from A after the last item (a_after).
template <Est E, int ITEMS>
__device__ __forceinline__ void replay(const Params &p, const Chunk<ITEMS> &c,
                                       const Affine (&e)[ITEMS], float a_after, float (&A)[ITEMS])
{
    A[ITEMS - 1] = step_apply<E, ITEMS>(p, c, e, ITEMS - 1, a_after);
#pragma unroll
    for (int j = ITEMS - 2; j >= 0; --j) A[j] = step_apply<E, ITEMS>(p, c, e, j, A[j + 1]);
}

// Outputs of every item from A_t (A[j]) and A at the step after the chunk (a_after).
template <Est E, int ITEMS, int VEC>
__device__ __forceinline__ void epilogue(const Params &p, const Chunk<ITEMS> &c,
                                         const float (&A)[ITEMS], float a_after, int64_t row,
                                         int t0)
{
    if (!c.valid) return;
    const int64_t off = row * p.ld;
    float o0[ITEMS];
    float o1[ITEMS];
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        if (E == Est::kReturn || E == Est::kTdLambda) {
            o0[j] = A[j];
        } else if (E == Est::kGae) {
            o0[j] = A[j];
            o1[j] = A[j] + c.v[j];
        } else if (E == Est::kVtrace) {
            // pg_t = rho_pg (r_t + gamma vs_{t+1} - V_t) = rho_pg (delta_t + gamma A_{t+1})
            // inside an episode (vs_{t+1} = V_{t+1} + A_{t+1}), rho_pg delta_t at its last
            // step (the successor value already in delta_t); build() left delta_t in sv.
            const bool stop = (c.stop >> j) & 1u;
            const float rho = c.x[j];
            const float a_next = (j + 1 < ITEMS) ? A[j + 1] : a_after;
            const float rho_pg = rho < p.pg_rho_bar ? rho : p.pg_rho_bar;
            o0[j] = c.v[j] + A[j];
            o1[j] = rho_pg * (stop ? c.sv[j] : fmaf(p.gamma, a_next, c.sv[j]));
        } else {
            o0[j] = A[j] + c.v[j];
        }
    }
    store_items<ITEMS, VEC>(p.out0 + off, t0, c.valid, o0);
    if (EstTraits<E>::kTwoOutputs && p.out1) store_items<ITEMS, VEC>(p.out1 + off, t0, c.valid, o1);
}

}  // namespace rlca
