/*
 * rlca_measure.h - measurement-only entry point of librlca: the copy ceiling of an access
 * pattern, against which the credit-assignment kernels of rlca.h are judged.
 *
 * The estimators are bound by HBM traffic (technical summary of "rl-triton:
 * High-Performance Triton GPU Kernels for Reinforcement Learning Credit Assignment",
 * Method section 2: inputs read once, outputs written once). How close a kernel gets to
 * the bandwidth of the memory is limited not only by the peak but also by the size and
 * shape of one launch (ramp-up, tail, partial waves). A plain copy with the same bytes
 * per step and the same launch shape measures that limit directly; the ratio of the
 * kernel's time to the copy's time says how much the scan itself costs.
 */
#ifndef RLCA_MEASURE_H
#define RLCA_MEASURE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RLCA_MEASURE_MAX_ARRAYS 4

/*
 * Streams n_elements elements (a contiguous [N, T] problem, N * T elements) through one
 * kernel launch on `stream`: reads every element of the n_inputs data arrays inputs[k]
 * (input_bytes = 4: fp32; 2: a 16-bit format, widened as bf16 bits) and of the n_flags
 * uint8 arrays flags[k], and writes every element of the n_outputs fp32 arrays
 * outputs[k], each output element being the sum of the inputs at that element (flag
 * bytes counted as their integer value), so no read can be skipped.
 *
 * Launch shape, as the estimator kernels: CTAs of 4 warps; each warp walks `chunks`
 * consecutive chunks of 256 elements (8 per lane, one 256-bit load per fp32 input,
 * one 64-bit load per flag array, one 256-bit store per output; 128-bit loads for 16-bit
 * inputs). chunks = 1 is the
 * shape of the warp-owned rows and of one 1024-step row per CTA; chunks = 4 that of a
 * warp walking a 1024-step row. Launched with programmatic stream serialization, and
 * each warp asks L2 for its elements before its grid dependency wait, as the estimator
 * kernels do.
 *
 * inputs, flags, outputs: host arrays of device pointers (current device). Every input
 * array must be aligned to 8 elements (32 bytes for fp32, 16 for 16-bit), every output
 * to 32 bytes and every flag array to 8 bytes. Outputs may not overlap inputs (not
 * checked: measurement only).
 * Every load of a warp's chunks is issued before the first one is used.
 * Returns 0, RLCA_ERR_PARAM (-3) for counts outside [0, RLCA_MEASURE_MAX_ARRAYS] (at
 * least one input and one output; flags at most 2), chunks not 1, 2 or 4 or input_bytes
 * not 4 or 2, RLCA_ERR_NULL (-1)
 * for a NULL array, RLCA_ERR_WORKSPACE (-5) for a misaligned array, RLCA_ERR_LAUNCH (-6)
 * if the launch fails. n_elements == 0 enqueues nothing.
 */
int rlca_measure_copy(const void *const *inputs, int n_inputs, int input_bytes,
                      const uint8_t *const *flags, int n_flags, float *const *outputs,
                      int n_outputs, int64_t n_elements, int chunks, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* RLCA_MEASURE_H */
