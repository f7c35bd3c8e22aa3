// Copy ceiling of an access pattern (declared in include/rlca_measure.h): the bytes an
// estimator moves per step, moved by a kernel that does nothing else, in the estimator
// kernels' launch shape. Measurement only; no estimator uses it.
#include "../../include/rlca.h"
#include "../../include/rlca_measure.h"
#include "launch.cuh"

namespace {

struct CopyArgs {
    const void *in[RLCA_MEASURE_MAX_ARRAYS];
    const uint8_t *flags[2];
    float *out[RLCA_MEASURE_MAX_ARRAYS];
    int n_in, n_flags, n_out, chunks;
    int64_t total;
};

// 8 consecutive input elements from element i: fp32 (one 256-bit load) or a 16-bit format
// (one 128-bit load; the bits are widened as bf16, which keeps every load's data in use).
template <int EB>
__device__ __forceinline__ void load8(const void *base, int64_t i, float *x)
{
    if constexpr (EB == 4) {
        rlca::ld_stream8(static_cast<const float *>(base) + i, x);
    } else {
        const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + i));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
}

template <int EB>
__device__ __forceinline__ float load1(const void *base, int64_t i)
{
    if constexpr (EB == 4) return rlca::ld_stream(static_cast<const float *>(base) + i);
    return __uint_as_float((uint32_t)__ldcs(static_cast<const unsigned short *>(base) + i) << 16);
}

constexpr int kChunk = 256;  // elements per warp chunk (32 lanes x 8)

// NI fp32 inputs, NF flag arrays and CHUNKS chunks per warp are compile-time, so every
// load of a warp's chunks is issued before the first one is used: the best a copy can do
// in this launch shape. The output count stays a run-time value (stores never wait).
template <int NI, int NF, int CHUNKS, int EB>
__global__ void __launch_bounds__(128) copy_pattern_kernel(const CopyArgs a)
{
    const int lane = threadIdx.x & 31;
    constexpr int64_t span = (int64_t)CHUNKS * kChunk;
    const int64_t w0 = ((int64_t)blockIdx.x * 4 + (threadIdx.x >> 5)) * span;
    if (lane == 0 && w0 < a.total) {
        const int64_t n = (w0 + span <= a.total ? span : a.total - w0);
#pragma unroll
        for (int k = 0; k < NI; ++k)
            rlca::prefetch_l2(static_cast<const char *>(a.in[k]) + EB * w0, EB * n);
#pragma unroll
        for (int k = 0; k < NF; ++k) rlca::prefetch_l2(a.flags[k] + w0, n);
    }
    rlca::grid_dependency_sync();
    if (w0 + span <= a.total) {
        float x[CHUNKS][NI][8];
        uint2 f[CHUNKS][NF > 0 ? NF : 1];
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
            const int64_t i = w0 + (int64_t)c * kChunk + lane * 8;
#pragma unroll
            for (int k = 0; k < NI; ++k) load8<EB>(a.in[k], i, x[c][k]);
#pragma unroll
            for (int k = 0; k < NF; ++k)
                f[c][k] = rlca::ld_stream(reinterpret_cast<const uint2 *>(a.flags[k] + i));
        }
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                acc[j] = 0.f;
#pragma unroll
                for (int k = 0; k < NI; ++k) acc[j] += x[c][k][j];
            }
#pragma unroll
            for (int k = 0; k < NF; ++k) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[j] += (float)((f[c][k].x >> (8 * j)) & 0xffu);
                    acc[4 + j] += (float)((f[c][k].y >> (8 * j)) & 0xffu);
                }
            }
            const int64_t i = w0 + (int64_t)c * kChunk + lane * 8;
#pragma unroll
            for (int k = 0; k < RLCA_MEASURE_MAX_ARRAYS; ++k)
                if (k < a.n_out) rlca::st_stream8(a.out[k] + i, acc);
        }
        return;
    }
    // The ragged end of the array, element by element.
    for (int64_t i = w0 + lane; i < w0 + span && i < a.total; i += 32) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NI; ++k) s += load1<EB>(a.in[k], i);
#pragma unroll
        for (int k = 0; k < NF; ++k) s += (float)a.flags[k][i];
#pragma unroll
        for (int k = 0; k < RLCA_MEASURE_MAX_ARRAYS; ++k)
            if (k < a.n_out) rlca::st_stream(a.out[k] + i, s);
    }
}

template <int NI, int NF, int EB>
cudaError_t launch_copy_ni_nf(const CopyArgs &a, unsigned grid, cudaStream_t stream)
{
    if (a.chunks == 1)
        return rlca::launch_pdl(copy_pattern_kernel<NI, NF, 1, EB>, grid, 128, 0, stream, a);
    if (a.chunks == 2)
        return rlca::launch_pdl(copy_pattern_kernel<NI, NF, 2, EB>, grid, 128, 0, stream, a);
    return rlca::launch_pdl(copy_pattern_kernel<NI, NF, 4, EB>, grid, 128, 0, stream, a);
}

template <int NI, int EB>
cudaError_t launch_copy_ni(const CopyArgs &a, unsigned grid, cudaStream_t stream)
{
    if (a.n_flags == 0) return launch_copy_ni_nf<NI, 0, EB>(a, grid, stream);
    if (a.n_flags == 1) return launch_copy_ni_nf<NI, 1, EB>(a, grid, stream);
    return launch_copy_ni_nf<NI, 2, EB>(a, grid, stream);
}

template <int EB>
cudaError_t launch_copy_eb(const CopyArgs &a, unsigned grid, cudaStream_t stream)
{
    switch (a.n_in) {
    case 1: return launch_copy_ni<1, EB>(a, grid, stream);
    case 2: return launch_copy_ni<2, EB>(a, grid, stream);
    case 3: return launch_copy_ni<3, EB>(a, grid, stream);
    default: return launch_copy_ni<4, EB>(a, grid, stream);
    }
}

bool aligned_to(const void *p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" int rlca_measure_copy(const void *const *inputs, int n_inputs, int input_bytes,
                                 const uint8_t *const *flags, int n_flags,
                                 float *const *outputs, int n_outputs, int64_t n_elements,
                                 int chunks, void *stream)
{
    if (n_inputs < 1 || n_inputs > RLCA_MEASURE_MAX_ARRAYS || n_outputs < 1 ||
        n_outputs > RLCA_MEASURE_MAX_ARRAYS || n_flags < 0 || n_flags > 2 ||
        (chunks != 1 && chunks != 2 && chunks != 4) || n_elements < 0 ||
        (input_bytes != 4 && input_bytes != 2))
        return RLCA_ERR_PARAM;
    if (!inputs || !outputs || (n_flags > 0 && !flags)) return RLCA_ERR_NULL;
    if (n_elements == 0) return RLCA_OK;
    CopyArgs a = {};
    for (int k = 0; k < n_inputs; ++k) {
        if (!inputs[k]) return RLCA_ERR_NULL;
        if (!aligned_to(inputs[k], 8 * input_bytes)) return RLCA_ERR_WORKSPACE;
        a.in[k] = inputs[k];
    }
    for (int k = 0; k < n_flags; ++k) {
        if (!flags[k]) return RLCA_ERR_NULL;
        if (!aligned_to(flags[k], 8)) return RLCA_ERR_WORKSPACE;
        a.flags[k] = flags[k];
    }
    for (int k = 0; k < n_outputs; ++k) {
        if (!outputs[k]) return RLCA_ERR_NULL;
        if (!aligned_to(outputs[k], 32)) return RLCA_ERR_WORKSPACE;
        a.out[k] = outputs[k];
    }
    a.n_in = n_inputs;
    a.n_flags = n_flags;
    a.n_out = n_outputs;
    a.chunks = chunks;
    a.total = n_elements;
    const int64_t per_cta = 4LL * kChunk * chunks;
    const int64_t grid = (n_elements + per_cta - 1) / per_cta;
    if (grid > 0x7fffffffLL) return RLCA_ERR_PARAM;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t err = input_bytes == 4 ? launch_copy_eb<4>(a, (unsigned)grid, s)
                                             : launch_copy_eb<2>(a, (unsigned)grid, s);
    return err == cudaSuccess ? RLCA_OK : RLCA_ERR_LAUNCH;
}
