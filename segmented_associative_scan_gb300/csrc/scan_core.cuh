// Segmented reverse affine scan: the on-chip core shared by every estimator kernel.
//
// Method section 1 of "rl-triton: High-Performance Triton GPU Kernels for Reinforcement
// Learning Credit Assignment": every estimator is A_t = alpha_t + beta_t * A_{t+1}, an
// associative scan over pairs (alpha, beta) with
//   (aB, bB) (+) (aA, bA) = (aB + bB * aA, bA * bB),   B the earlier step, A the later.
// Method section 3 (episode boundaries) enters as an explicit reset: a step whose
// episode ends there takes nothing from t+1. The reset is a select, not a multiply by 0,
// so a NaN or Inf in a later episode never reaches an earlier one.
//
// Encoding: every beta of the estimators is >= 0 (gamma >= 0, lambda in [0,1], clipped
// ratios >= 0), so the sign bit of b is free and carries the reset. A reset element has
// b = -1; composing a non-reset element (b >= 0) with a reset one multiplies the signs,
// so the composite is negative, i.e. reset, too (0 * -1 = -0 keeps the sign bit).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace rlca {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kResetB = -1.0f;

// The map x -> a + b * x, or the constant a when b's sign bit is set (reset inside).
struct Affine {
    float a;
    float b;
};

__device__ __forceinline__ bool is_reset(float b) { return __float_as_int(b) < 0; }

__device__ __forceinline__ Affine affine_identity() { return Affine{0.f, 1.f}; }

__device__ __forceinline__ float affine_apply(const Affine &e, float x)
{
    return is_reset(e.b) ? e.a : fmaf(e.b, x, e.a);
}

// The pages' operator: `early` applied after `late` (early covers smaller t).
__device__ __forceinline__ Affine affine_compose(const Affine &early, const Affine &late)
{
    const bool r = is_reset(early.b);
    return Affine{r ? early.a : fmaf(early.b, late.a, early.a), r ? early.b : early.b * late.b};
}

__device__ __forceinline__ Affine shfl_down(const Affine &x, int d)
{
    return Affine{__shfl_down_sync(kFullMask, x.a, d), __shfl_down_sync(kFullMask, x.b, d)};
}

__device__ __forceinline__ Affine shfl_idx(const Affine &x, int lane)
{
    return Affine{__shfl_sync(kFullMask, x.a, lane), __shfl_sync(kFullMask, x.b, lane)};
}

// Inclusive suffix scan across a warp: lane i gets x_i (+) x_{i+1} (+) ... (+) x_31.
__device__ __forceinline__ Affine warp_suffix_scan(Affine x, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Affine y = shfl_down(x, d);
        if (lane + d < 32) x = affine_compose(x, y);
    }
    return x;
}

// ---------------------------------------------------------------- memory access

// Streaming loads/stores: every input is read once and every output written once.
__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ float ld_stream(const float *p) { return __ldcs(p); }
__device__ __forceinline__ uint32_t ld_stream(const uint32_t *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(float *p, float v) { __stcs(p, v); }

// Access widths, the VEC template argument of the load/store helpers (bit flags):
//   0 scalar; bit 0: 128-bit access (16-byte aligned rows);
//   bit 1: 256-bit loads of fp32 data and 64-bit loads of the 8 flag bytes of 8 steps;
//   bit 2: 256-bit stores of fp32 outputs.
// Bits 1 and 2 need 32-byte aligned rows (sm_100 and later). A 256-bit access moves one
// whole 32-byte sector per thread, so a warp's store fills every sector it touches in
// one instruction instead of writing two half sectors.
constexpr int kVec16 = 1;
constexpr int kWideLoads = 2;
constexpr int kWideStores = 4;
__device__ __forceinline__ void ld_stream8(const float *p, float *x)
{
    asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]),
                   "=f"(x[6]), "=f"(x[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_stream8(float *p, const float *x)
{
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                 "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                 "f"(x[7])
                 : "memory");
}

__device__ __forceinline__ uint2 ld_stream(const uint2 *p) { return __ldcs(p); }

// Ask L2 to fetch the 16-byte granules inside [p, p + bytes) of global memory, without
// waiting and without touching registers or L1 (one bulk prefetch; a hint only). L2 is
// the point of coherence for global memory, so a later load still sees any write that
// lands after the prefetch: a kernel may issue it before its grid dependency wait.
__device__ __forceinline__ void prefetch_l2(const void *p, int64_t bytes)
{
    if (bytes > (1 << 24)) bytes = 1 << 24;  // a hint: at most 16 MiB per call
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uintptr_t lo = (a + 15) & ~(uintptr_t)15;
    const uintptr_t hi = (a + (uintptr_t)bytes) & ~(uintptr_t)15;
    if (bytes > 0 && hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo),
                     "r"((unsigned)(hi - lo))
                     : "memory");
}

template <int ITEMS>
__device__ __forceinline__ constexpr unsigned all_items()
{
    return ITEMS == 32 ? 0xffffffffu : ((1u << ITEMS) - 1u);
}

// Bit j set for the items t0 + j < T.
template <int ITEMS>
__device__ __forceinline__ unsigned valid_items(int t0, int T)
{
    const int n = T - t0;
    return n >= ITEMS ? all_items<ITEMS>() : (n > 0 ? (1u << n) - 1u : 0u);
}

// ------------------------------------------------------------- input element types

// Per-step inputs are fp32, bf16 (`uint16_t` holding the bf16 bit pattern) or fp16
// (`__half`); the arithmetic is fp32 either way. A bf16 value widens to fp32 exactly (its
// bits are the high half of the fp32 pattern), and so does every fp16 value, subnormals
// and infinities included (CUDA's half-to-float conversion). `kPerVec` elements fill one
// 128-bit load.
template <typename TIn>
struct InType;

template <>
struct InType<float> {
    static constexpr int kPerVec = 4;
    __device__ static __forceinline__ float stream(const float *p) { return __ldcs(p); }
    __device__ static __forceinline__ float cached(const float *p) { return __ldg(p); }
    __device__ static __forceinline__ void unpack(const uint4 &q, float *x)
    {
        x[0] = __uint_as_float(q.x);
        x[1] = __uint_as_float(q.y);
        x[2] = __uint_as_float(q.z);
        x[3] = __uint_as_float(q.w);
    }
    __device__ static __forceinline__ void unpack64(const uint2 &q, float *x)
    {
        x[0] = __uint_as_float(q.x);
        x[1] = __uint_as_float(q.y);
    }
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits)
{
    return __uint_as_float(bits << 16);
}

template <>
struct InType<uint16_t> {
    static constexpr int kPerVec = 8;
    __device__ static __forceinline__ float stream(const uint16_t *p)
    {
        return bf16_bits_to_float(__ldcs(reinterpret_cast<const unsigned short *>(p)));
    }
    __device__ static __forceinline__ float cached(const uint16_t *p)
    {
        return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short *>(p)));
    }
    __device__ static __forceinline__ void unpack(const uint4 &q, float *x)
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ void unpack64(const uint2 &q, float *x)
    {
        x[0] = __uint_as_float(q.x << 16);
        x[1] = __uint_as_float(q.x & 0xffff0000u);
        x[2] = __uint_as_float(q.y << 16);
        x[3] = __uint_as_float(q.y & 0xffff0000u);
    }
};

template <>
struct InType<__half> {
    static constexpr int kPerVec = 8;
    __device__ static __forceinline__ float stream(const __half *p)
    {
        return __half2float(__ldcs(p));
    }
    __device__ static __forceinline__ float cached(const __half *p)
    {
        return __half2float(__ldg(p));
    }
    __device__ static __forceinline__ void unpack(const uint4 &q, float *x)
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // Word i holds steps 2i (low half) and 2i + 1 (high half).
            const float2 f = __half22float2(__halves2half2(
                __ushort_as_half((unsigned short)(w[i] & 0xffffu)),
                __ushort_as_half((unsigned short)(w[i] >> 16))));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    __device__ static __forceinline__ void unpack64(const uint2 &q, float *x)
    {
        const uint32_t w[2] = {q.x, q.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float2 f = __half22float2(__halves2half2(
                __ushort_as_half((unsigned short)(w[i] & 0xffffu)),
                __ushort_as_half((unsigned short)(w[i] >> 16))));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
};

// Whether a pointer sits on an n-byte boundary (n a power of two).
template <int N>
__device__ __forceinline__ bool on_boundary(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & (N - 1)) == 0;
}

// ITEMS consecutive inputs of one row starting at column t0, widened to fp32; columns
// >= T read as 0. VEC 1: 128-bit loads (the row start and t0 are 16-byte aligned);
// VEC bit 1: 256-bit loads for fp32 data (32-byte aligned), 128-bit for bf16. VEC 0
// (rows not aligned as a whole): 128-bit or 64-bit loads where this thread's items
// happen to sit on such a boundary (measured on GB300: bf16 GAE [4096, 700] 30.2 ->
// 15.2 us, fp32 GAE [4096, 1001] 35.2 -> 25.8), element loads otherwise.
template <int ITEMS, int VEC, typename TIn = float>
__device__ __forceinline__ void load_items(const TIn *__restrict__ row, int t0, int T,
                                           float (&x)[ITEMS])
{
    constexpr int PV = InType<TIn>::kPerVec;
    static_assert(ITEMS % PV == 0, "a thread's items fill whole 128-bit loads");
    constexpr bool kWide = (VEC & kWideLoads) && sizeof(TIn) == 4 && ITEMS % 8 == 0;
    if (kWide && t0 + ITEMS <= T) {
#pragma unroll
        for (int k = 0; k < ITEMS / 8; ++k)
            ld_stream8(reinterpret_cast<const float *>(row + t0) + 8 * k, x + 8 * k);
    } else if (VEC && t0 + ITEMS <= T) {
#pragma unroll
        for (int k = 0; k < ITEMS / PV; ++k) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(row + t0) + k);
            InType<TIn>::unpack(q, x + PV * k);
        }
    } else if (!VEC && t0 + ITEMS <= T && on_boundary<16>(row + t0)) {
        // Rows not aligned as a whole, this thread's items on a 16-byte boundary.
#pragma unroll
        for (int k = 0; k < ITEMS / PV; ++k) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(row + t0) + k);
            InType<TIn>::unpack(q, x + PV * k);
        }
    } else if (!VEC && t0 + ITEMS <= T && on_boundary<8>(row + t0)) {
        constexpr int P8 = 8 / (int)sizeof(TIn);  // items per 64-bit load
#pragma unroll
        for (int k = 0; k < ITEMS / P8; ++k) {
            const uint2 q = __ldcs(reinterpret_cast<const uint2 *>(row + t0) + k);
            InType<TIn>::unpack64(q, x + P8 * k);
        }
    } else {
#pragma unroll
        for (int j = 0; j < ITEMS; ++j)
            x[j] = (t0 + j < T) ? InType<TIn>::stream(row + t0 + j) : 0.f;
    }
}

// 4 flag bytes -> 4 bits (bit i set when byte i is nonzero), branch-free: bit 7 of each
// byte becomes "any bit set" without carries across bytes, then one multiply gathers the
// four bit-7s into bits 24..27 (the partial products land on distinct bit positions).
__device__ __forceinline__ unsigned nonzero_bytes(uint32_t w)
{
    const uint32_t hi = ((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w;
    const uint32_t b = (hi & 0x80808080u) >> 7;
    return (b * 0x01020408u) >> 24;
}

// Bit j set when flag byte (t0 + j) is nonzero; columns >= T read as clear. VEC bit 1
// reads the 8 bytes of 8 steps with one 64-bit load (row start and t0 8-byte aligned).
template <int ITEMS, int VEC>
__device__ __forceinline__ unsigned load_flag_bits(const uint8_t *__restrict__ row, int t0,
                                                   int T)
{
    unsigned bits = 0;
    if ((VEC & kWideLoads) && ITEMS % 8 == 0 && t0 + ITEMS <= T) {
#pragma unroll
        for (int k = 0; k < ITEMS / 8; ++k) {
            const uint2 w = ld_stream(reinterpret_cast<const uint2 *>(row + t0) + k);
            bits |= (nonzero_bytes(w.x) | (nonzero_bytes(w.y) << 4)) << (8 * k);
        }
    } else if ((VEC || on_boundary<4>(row + t0)) && t0 + ITEMS <= T) {
#pragma unroll
        for (int k = 0; k < ITEMS / 4; ++k)
            bits |= nonzero_bytes(ld_stream(reinterpret_cast<const uint32_t *>(row + t0) + k))
                    << (4 * k);
    } else {
#pragma unroll
        for (int j = 0; j < ITEMS; ++j)
            if (t0 + j < T && row[t0 + j] != 0) bits |= 1u << j;
    }
    return bits;
}

// Bit j set when either flag byte (t0 + j) of row_a or row_b is nonzero: the two flag
// words are OR-ed before a single decode.
template <int ITEMS, int VEC>
__device__ __forceinline__ unsigned load_flag_bits_or(const uint8_t *__restrict__ row_a,
                                                      const uint8_t *__restrict__ row_b, int t0,
                                                      int T)
{
    unsigned bits = 0;
    if ((VEC & kWideLoads) && ITEMS % 8 == 0 && t0 + ITEMS <= T) {
#pragma unroll
        for (int k = 0; k < ITEMS / 8; ++k) {
            const uint2 a = ld_stream(reinterpret_cast<const uint2 *>(row_a + t0) + k);
            const uint2 b = ld_stream(reinterpret_cast<const uint2 *>(row_b + t0) + k);
            bits |= (nonzero_bytes(a.x | b.x) | (nonzero_bytes(a.y | b.y) << 4)) << (8 * k);
        }
    } else if ((VEC || (on_boundary<4>(row_a + t0) && on_boundary<4>(row_b + t0))) &&
               t0 + ITEMS <= T) {
#pragma unroll
        for (int k = 0; k < ITEMS / 4; ++k)
            bits |= nonzero_bytes(ld_stream(reinterpret_cast<const uint32_t *>(row_a + t0) + k) |
                                  ld_stream(reinterpret_cast<const uint32_t *>(row_b + t0) + k))
                    << (4 * k);
    } else {
#pragma unroll
        for (int j = 0; j < ITEMS; ++j)
            if (t0 + j < T && (row_a[t0 + j] | row_b[t0 + j]) != 0) bits |= 1u << j;
    }
    return bits;
}

// Store the valid items (bit j of `valid`) of ITEMS consecutive floats.
template <int ITEMS, int VEC>
__device__ __forceinline__ void store_items(float *__restrict__ row, int t0, unsigned valid,
                                            const float (&x)[ITEMS])
{
    if ((VEC & kWideStores) && ITEMS % 8 == 0 && valid == all_items<ITEMS>()) {
#pragma unroll
        for (int k = 0; k < ITEMS / 8; ++k) st_stream8(row + t0 + 8 * k, x + 8 * k);
    } else if ((VEC || on_boundary<16>(row + t0)) && valid == all_items<ITEMS>()) {
#pragma unroll
        for (int k = 0; k < ITEMS / 4; ++k)
            st_stream(reinterpret_cast<float4 *>(row + t0) + k,
                      make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]));
    } else if (!VEC && on_boundary<8>(row + t0) && valid == all_items<ITEMS>()) {
#pragma unroll
        for (int k = 0; k < ITEMS / 2; ++k)
            __stcs(reinterpret_cast<float2 *>(row + t0) + k, make_float2(x[2 * k], x[2 * k + 1]));
    } else {
#pragma unroll
        for (int j = 0; j < ITEMS; ++j)
            if (valid & (1u << j)) st_stream(row + t0 + j, x[j]);
    }
}

}  // namespace rlca
