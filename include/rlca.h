/*
 * rlca.h - C ABI of librlca: reinforcement-learning credit assignment on one GB300
 * (sm_103a), each estimator computed as one fused, segmented, reverse affine scan.
 *
 * Source: "rl-triton: High-Performance Triton GPU Kernels for Reinforcement Learning
 * Credit Assignment" (technical summary).
 *   - Problem statement: credit-assignment quantities (advantages, value targets,
 *     returns) over [num_envs, seq_len] tensors of rewards, values and done flags.
 *   - Method section 1: every estimator is the first-order recurrence
 *     A_t = alpha_t + beta_t * A_{t+1}, solved as an associative scan over the pairs
 *     (alpha_t, beta_t) with (aB, bB) (+) (aA, bA) = (aB + bB * aA, bA * bB).
 *   - Method section 2: the pairs are built on chip from the raw inputs; inputs are
 *     read from HBM once and outputs written once.
 *   - Method section 3: a terminated step has successor value 0; a truncated step
 *     bootstraps from a supplied value; the last step of the window (t = T-1)
 *     bootstraps from a supplied per-env value, counted exactly once.
 *
 * Common conventions (all entry points)
 *   Layout    Every per-step array is row-major [N, ld]: row n holds
 *             env n, steps t = 0..T-1 in columns 0..T-1 (T contiguous), ld >= T.
 *             Outputs use the same layout and ld; their columns T..ld-1 are not
 *             written. Data are float32; flags are uint8 (0 = clear, nonzero = set;
 *             a torch.bool tensor qualifies). Per-env bootstrap values are float32 [N].
 *   Flags     terminated[n,t]: the episode ended at step t (successor value 0, no credit
 *             from t+1). truncated[n,t] (nullable = none truncated): the episode was
 *             cut at t; its successor value is trunc_value[n,t], which is read only
 *             where truncated is set. If both are set, termination wins. At t = T-1 the
 *             successor value is bootstrap[n] (nullable = 0) unless the step is
 *             terminated or truncated.
 *   Memory    Every buffer is either device memory of the current device (cudaMalloc,
 *             a stream-ordered pool, managed memory) or pinned host memory
 *             (cudaHostAlloc, cudaMallocHost, cudaHostRegister; torch pin_memory). On
 *             GB300 the kernels read and write pinned host memory directly over
 *             NVLink-C2C, so a caller whose rollouts sit in host memory needs no
 *             staging copies: inputs cross the link once and outputs once, inside the
 *             kernel. Pageable host memory and another device's memory are rejected
 *             with RLCA_ERR_MEMORY (each pointer is classified with
 *             cudaPointerGetAttributes on every call). The look-back workspace must be
 *             device memory.
 *   Stream    `stream` is a cudaStream_t (NULL = the legacy default stream) of the
 *             current device; all work is enqueued on it, asynchronously.
 *   Ownership The caller owns every buffer. The library never allocates or frees
 *             memory, never changes the current device and never synchronises (except
 *             rlca_workspace_check, which says so). Inputs are read only. Outputs must
 *             not overlap any input or each other.
 *   Errors    0 = RLCA_OK. A negative code means nothing was enqueued, except
 *             RLCA_ERR_LAUNCH (the launch itself failed; cudaGetLastError is cleared).
 *             N == 0 or T == 0 is a valid empty problem: RLCA_OK, nothing enqueued.
 *   Precision fp32 arithmetic, round to nearest, no fast-math; exp is the CUDA libm
 *             expf. The scan reassociates the recurrence, so results differ from a
 *             sequential loop by rounding only.
 */
#ifndef RLCA_H
#define RLCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum rlca_status {
    RLCA_OK = 0,
    RLCA_ERR_NULL = -1,      /* a required pointer is NULL */
    RLCA_ERR_SHAPE = -2,     /* N < 0, T < 0, ld < T, T > RLCA_MAX_T, or N*ld overflows */
    RLCA_ERR_PARAM = -3,     /* gamma < 0 or not finite; lambda outside [0,1]; a clip <= 0 or NaN */
    RLCA_ERR_ALIAS = -4,     /* an output overlaps an input or another output */
    RLCA_ERR_WORKSPACE = -5, /* workspace too small or misaligned */
    RLCA_ERR_LAUNCH = -6,    /* the CUDA launch failed */
    RLCA_ERR_TIMEOUT = -7,   /* a bounded cross-block wait gave up (see rlca_workspace_check) */
    RLCA_ERR_MEMORY = -8     /* a buffer is neither current-device memory nor pinned host memory */
};

/* Largest supported seq_len. */
#define RLCA_MAX_T (1 << 30)

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int rlca_version(void);

/* Static, NUL-terminated description of a status code. */
const char *rlca_status_string(int status);

/*
 * Discounted return G_t = r_t + gamma * G_{t+1} inside an episode, and
 * G_t = r_t + gamma * (successor value) at its last step.
 * Scan form: alpha_t = r_t (+ gamma * successor value at the episode's last step),
 * beta_t = gamma.
 * Inputs: reward, terminated [N,ld]; truncated, trunc_value [N,ld] (nullable, together);
 * bootstrap [N] (nullable). Output: returns [N,ld].
 */
int rlca_discounted_return(const float *reward, const uint8_t *terminated,
                           const uint8_t *truncated, const float *trunc_value,
                           const float *bootstrap, float gamma, int64_t N, int64_t T,
                           int64_t ld, float *returns, void *stream);

/*
 * TD(lambda) lambda-returns (Sutton & Barto):
 * G_t = r_t + gamma * ((1 - lambda) V_{t+1} + lambda G_{t+1}) inside an episode,
 * G_t = r_t + gamma * (successor value) at its last step.
 * Scan form: alpha_t = r_t + gamma (1 - lambda) V_{t+1}, beta_t = gamma lambda.
 * Inputs as rlca_discounted_return plus value [N,ld]. Output: targets [N,ld].
 */
int rlca_td_lambda(const float *reward, const float *value, const uint8_t *terminated,
                   const uint8_t *truncated, const float *trunc_value,
                   const float *bootstrap, float gamma, float lambda, int64_t N,
                   int64_t T, int64_t ld, float *targets, void *stream);

/*
 * GAE (Schulman et al. 2016): delta_t = r_t + gamma V(s_{t+1}) - V_t,
 * A_t = delta_t + gamma lambda A_{t+1} inside an episode (A_t = delta_t at its last
 * step); returns_t = A_t + V_t. V(s_{t+1}) is V_{t+1} inside an episode and the
 * successor value at its last step.
 * Scan form: alpha_t = delta_t, beta_t = gamma lambda.
 * Outputs: advantages [N,ld]; returns [N,ld] (nullable: not written).
 */
int rlca_gae(const float *reward, const float *value, const uint8_t *terminated,
             const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
             float gamma, float lambda, int64_t N, int64_t T, int64_t ld,
             float *advantages, float *returns, void *stream);

/*
 * V-trace (Espeholt et al. 2018, IMPALA), from log importance ratios log_rho [N,ld]:
 * rho_t = exp(log_rho_t), rho_hat_t = min(rho_bar, rho_t), c_t = lambda min(c_bar, rho_t),
 * vs_t - V_t = rho_hat_t (r_t + gamma V(s_{t+1}) - V_t) + gamma c_t (vs_{t+1} - V_{t+1})
 * inside an episode (last term absent at its last step);
 * pg_t = min(pg_rho_bar, rho_t) (r_t + gamma q_{t+1} - V_t), q_{t+1} = vs_{t+1} inside an
 * episode, the successor value at its last step.
 * Scan form: A_t = vs_t - V_t, alpha_t = rho_hat_t delta_t, beta_t = gamma c_t.
 * Outputs: vs [N,ld]; pg_advantages [N,ld] (nullable: not written).
 */
int rlca_vtrace(const float *reward, const float *value, const float *log_rho,
                const uint8_t *terminated, const uint8_t *truncated,
                const float *trunc_value, const float *bootstrap, float gamma,
                float lambda, float rho_bar, float c_bar, float pg_rho_bar, int64_t N,
                int64_t T, int64_t ld, float *vs, float *pg_advantages, void *stream);

/*
 * Retrace(lambda) (Munos et al. 2016), from importance ratios rho [N,ld],
 * Q(s_t, a_t) = q_taken [N,ld] and E_pi Q(s_t, .) = expected_q [N,ld]:
 * c_t = lambda min(1, rho_t),
 * Q^ret_t = r_t + gamma E_pi Q(s_{t+1},.) + gamma c_{t+1} (Q^ret_{t+1} - Q(s_{t+1},a_{t+1}))
 * inside an episode (last term absent at its last step). At the episode's last step
 * E_pi Q(s_{t+1},.) is 0 (terminated), trunc_value (truncated) or bootstrap_ev[n]
 * (window end; nullable = 0).
 * Scan form: A_t = Q^ret_t - Q_t, alpha_t = r_t + gamma E_pi Q(s_{t+1},.) - Q_t,
 * beta_t = gamma c_{t+1}. Output: q_ret [N,ld].
 * Domain: rho is a ratio of probabilities, rho >= +0. rho_{t+1} = +0 gives c_{t+1} = 0,
 * exactly as the formula (a NaN or Inf in Q^ret_{t+1} - Q(s_{t+1},a_{t+1}) still turns
 * Q^ret_t into NaN, since 0 * NaN and 0 * Inf are NaN). A negative ratio, and -0.0, lie
 * outside the domain and are read as the end of the trace: Q^ret_t then takes nothing
 * from step t+1 on, not even a NaN or Inf (the scan carries its reset in the sign bit
 * of beta_t). With finite values that equals the formula with the ratio replaced by +0.
 */
int rlca_retrace(const float *reward, const float *q_taken, const float *expected_q,
                 const float *rho, const uint8_t *terminated, const uint8_t *truncated,
                 const float *trunc_value, const float *bootstrap_ev, float gamma,
                 float lambda, int64_t N, int64_t T, int64_t ld, float *q_ret,
                 void *stream);

/*
 * TD(lambda) for several lambdas in one pass (fused): the inputs are read from HBM once
 * and every lambda's targets are scanned on chip and written once (Method section 2:
 * HBM traffic, not arithmetic, bounds these scans, so sharing the load is what pays).
 * Each targets[k] equals rlca_td_lambda with lambdas[k] (lambda = 1 gives the discounted
 * return). lambdas: host array of n_lambdas values in [0, 1]; targets: host array of
 * n_lambdas output pointers [N, ld] (device or pinned host memory), none NULL, overlapping
 * no input and no other target.
 * 1 <= n_lambdas <= RLCA_TD_LAMBDA_MAX, else RLCA_ERR_PARAM.
 */
#define RLCA_TD_LAMBDA_MAX 4
int rlca_td_lambda_multi(const float *reward, const float *value, const uint8_t *terminated,
                         const uint8_t *truncated, const float *trunc_value,
                         const float *bootstrap, float gamma, const float *lambdas,
                         int n_lambdas, int64_t N, int64_t T, int64_t ld,
                         float *const *targets, void *stream);

/*
 * GAE and V-trace in one pass (fused): reward, value, log_rho and the flags are read from
 * HBM once; both estimators are scanned on chip and their four outputs written once
 * (Method section 2: the load, not the arithmetic, is what costs). The outputs equal
 * rlca_gae with lambda_gae (advantages, returns) and rlca_vtrace with lambda_vtrace,
 * rho_bar, c_bar, pg_rho_bar (vs, pg_advantages), for the same value estimates.
 * advantages and vs are required; returns and pg_advantages are nullable (not written).
 * No output may overlap an input or another output.
 */
int rlca_gae_vtrace(const float *reward, const float *value, const float *log_rho,
                    const uint8_t *terminated, const uint8_t *truncated,
                    const float *trunc_value, const float *bootstrap, float gamma,
                    float lambda_gae, float lambda_vtrace, float rho_bar, float c_bar,
                    float pg_rho_bar, int64_t N, int64_t T, int64_t ld, float *advantages,
                    float *returns, float *vs, float *pg_advantages, void *stream);

/*
 * Forward-time scans (Method section 1: eligibility traces are the forward-time mirror
 * of the recurrence; episodic prefix sums are among the estimators it covers).
 *   A_t = x_t + decay * A_{t-1} inside an episode; A_t = x_t at a step whose previous
 *   step terminated or truncated (a new episode); A_{-1} = init[n] at the window start
 *   (nullable = 0), the value carried in from the previous window.
 * Inputs: x, terminated [N,ld]; truncated [N,ld] (nullable; no values needed: a
 * truncation only ends the episode here); init [N] (nullable). Output [N,ld].
 * Errors as above; decay must be finite and >= 0 (RLCA_ERR_PARAM otherwise).
 */

/* Accumulating eligibility trace e_t = x_t + decay * e_{t-1} (decay = gamma * lambda). */
int rlca_eligibility_trace(const float *x, const uint8_t *terminated,
                           const uint8_t *truncated, const float *init, float decay, int64_t N,
                           int64_t T, int64_t ld, float *traces, void *stream);

/* Episodic prefix sum S_t = x_t + S_{t-1} (decay 1). */
int rlca_episodic_prefix_sum(const float *x, const uint8_t *terminated,
                             const uint8_t *truncated, const float *init, int64_t N, int64_t T,
                             int64_t ld, float *sums, void *stream);

/*
 * 16-bit inputs: bf16 (the _bf16 entry points) and fp16 (the _fp16 entry points). The
 * same estimators with every per-step data input (rewards, values, log-ratios, ratios,
 * Q-values, truncation values, x) given as 16-bit floats: uint16_t holding the bit
 * pattern (a torch.bfloat16 or torch.float16 tensor qualifies). Each value widens to fp32
 * exactly (fp16 subnormals and infinities included; NaN stays NaN) and all arithmetic is
 * fp32, so the results equal the fp32 entry points' on the widened inputs up to rounding
 * order. Per-env bootstrap / init values and all outputs stay fp32. Rows take 128-bit
 * loads when ld % 8 == 0 and every input base is 16-byte aligned. Arguments, layouts
 * and errors otherwise as the fp32 entry points.
 * This halves the bytes of each data input; the pages note that data formats other
 * than the standard one need more work (technical summary, lay text on limitations).
 */
int rlca_discounted_return_bf16(const uint16_t *reward, const uint8_t *terminated,
                                const uint8_t *truncated, const uint16_t *trunc_value,
                                const float *bootstrap, float gamma, int64_t N, int64_t T,
                                int64_t ld, float *returns, void *stream);
int rlca_td_lambda_bf16(const uint16_t *reward, const uint16_t *value,
                        const uint8_t *terminated, const uint8_t *truncated,
                        const uint16_t *trunc_value, const float *bootstrap, float gamma,
                        float lambda, int64_t N, int64_t T, int64_t ld, float *targets,
                        void *stream);
int rlca_gae_bf16(const uint16_t *reward, const uint16_t *value, const uint8_t *terminated,
                  const uint8_t *truncated, const uint16_t *trunc_value, const float *bootstrap,
                  float gamma, float lambda, int64_t N, int64_t T, int64_t ld,
                  float *advantages, float *returns, void *stream);
int rlca_vtrace_bf16(const uint16_t *reward, const uint16_t *value, const uint16_t *log_rho,
                     const uint8_t *terminated, const uint8_t *truncated,
                     const uint16_t *trunc_value, const float *bootstrap, float gamma,
                     float lambda, float rho_bar, float c_bar, float pg_rho_bar, int64_t N,
                     int64_t T, int64_t ld, float *vs, float *pg_advantages, void *stream);
int rlca_retrace_bf16(const uint16_t *reward, const uint16_t *q_taken,
                      const uint16_t *expected_q, const uint16_t *rho,
                      const uint8_t *terminated, const uint8_t *truncated,
                      const uint16_t *trunc_value, const float *bootstrap_ev, float gamma,
                      float lambda, int64_t N, int64_t T, int64_t ld, float *q_ret,
                      void *stream);
int rlca_eligibility_trace_bf16(const uint16_t *x, const uint8_t *terminated,
                                const uint8_t *truncated, const float *init, float decay,
                                int64_t N, int64_t T, int64_t ld, float *traces, void *stream);
int rlca_episodic_prefix_sum_bf16(const uint16_t *x, const uint8_t *terminated,
                                  const uint8_t *truncated, const float *init, int64_t N,
                                  int64_t T, int64_t ld, float *sums, void *stream);

int rlca_discounted_return_fp16(const uint16_t *reward, const uint8_t *terminated,
                                const uint8_t *truncated, const uint16_t *trunc_value,
                                const float *bootstrap, float gamma, int64_t N, int64_t T,
                                int64_t ld, float *returns, void *stream);
int rlca_td_lambda_fp16(const uint16_t *reward, const uint16_t *value,
                        const uint8_t *terminated, const uint8_t *truncated,
                        const uint16_t *trunc_value, const float *bootstrap, float gamma,
                        float lambda, int64_t N, int64_t T, int64_t ld, float *targets,
                        void *stream);
int rlca_gae_fp16(const uint16_t *reward, const uint16_t *value, const uint8_t *terminated,
                  const uint8_t *truncated, const uint16_t *trunc_value, const float *bootstrap,
                  float gamma, float lambda, int64_t N, int64_t T, int64_t ld,
                  float *advantages, float *returns, void *stream);
int rlca_vtrace_fp16(const uint16_t *reward, const uint16_t *value, const uint16_t *log_rho,
                     const uint8_t *terminated, const uint8_t *truncated,
                     const uint16_t *trunc_value, const float *bootstrap, float gamma,
                     float lambda, float rho_bar, float c_bar, float pg_rho_bar, int64_t N,
                     int64_t T, int64_t ld, float *vs, float *pg_advantages, void *stream);
int rlca_retrace_fp16(const uint16_t *reward, const uint16_t *q_taken,
                      const uint16_t *expected_q, const uint16_t *rho,
                      const uint8_t *terminated, const uint8_t *truncated,
                      const uint16_t *trunc_value, const float *bootstrap_ev, float gamma,
                      float lambda, int64_t N, int64_t T, int64_t ld, float *q_ret,
                      void *stream);
int rlca_eligibility_trace_fp16(const uint16_t *x, const uint8_t *terminated,
                                const uint8_t *truncated, const float *init, float decay,
                                int64_t N, int64_t T, int64_t ld, float *traces, void *stream);
int rlca_episodic_prefix_sum_fp16(const uint16_t *x, const uint8_t *terminated,
                                  const uint8_t *truncated, const float *init, int64_t N,
                                  int64_t T, int64_t ld, float *sums, void *stream);

/*
 * Long sequences: tiles scanned in parallel with decoupled look-back.
 *
 * The kernels scan tiles of 1024 steps. When T > 1024 a row spans several tiles. The
 * entry points above walk the tiles of a row one after another inside one CTA, carrying
 * A between them in registers. The _ex variants below take a caller-owned device
 * workspace and, when N is below twice the SM count (rows alone cannot fill the GPU),
 * launch one CTA per tile for all tiles of all rows at once; a tile finds its carry-in
 * from the later tiles of its row by decoupled look-back (Merrill & Garland 2016). On a
 * GB300 this is 16x faster at [16, 524288] and 60x at [4, 2097152]. With more rows the
 * _ex call walks rows like the plain call (faster there) and leaves the workspace alone.
 * This realises Method section 1's O(log T)-depth scan across CTAs with one HBM read
 * and one write (Method section 2).
 *
 * Workspace: rlca_workspace_bytes(N, T) bytes of device memory, 256-byte aligned,
 * zero-filled once before its first use (e.g. cudaMemsetAsync to 0). Each call leaves
 * it ready for the next, so it is zeroed only once. Calls that share a workspace must
 * not run concurrently on the GPU (use one stream, or order the streams). The workspace
 * may overlap no input or output (RLCA_ERR_ALIAS).
 * When rlca_workspace_bytes returns 0 (T <= 1024: rows never span tiles) an _ex call
 * ignores the workspace and behaves exactly as the plain call.
 *
 * Bounded waits: a tile polls the state of a later tile at most about a second; if it
 * gives up it marks its outputs NaN and records RLCA_ERR_TIMEOUT in the workspace. No
 * wait can hang the GPU. rlca_workspace_check reports and clears that record.
 */

/* Bytes of workspace an _ex call needs for [N, T]: 256 + 32 * N * ceil(T / 1024) when
 * T > 1024, else 0. Returns 0 for invalid shapes. */
size_t rlca_workspace_bytes(int64_t N, int64_t T);

/* Synchronises `stream`, then returns RLCA_OK, or RLCA_ERR_TIMEOUT if a look-back wait
 * on this workspace gave up since the last check (the record is then cleared), or
 * RLCA_ERR_LAUNCH if a CUDA call failed. This is the only entry point that blocks. */
int rlca_workspace_check(void *workspace, void *stream);

int rlca_discounted_return_ex(const float *reward, const uint8_t *terminated,
                              const uint8_t *truncated, const float *trunc_value,
                              const float *bootstrap, float gamma, int64_t N, int64_t T,
                              int64_t ld, float *returns, void *workspace,
                              size_t workspace_bytes, void *stream);

int rlca_td_lambda_ex(const float *reward, const float *value, const uint8_t *terminated,
                      const uint8_t *truncated, const float *trunc_value,
                      const float *bootstrap, float gamma, float lambda, int64_t N,
                      int64_t T, int64_t ld, float *targets, void *workspace,
                      size_t workspace_bytes, void *stream);

int rlca_gae_ex(const float *reward, const float *value, const uint8_t *terminated,
                const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
                float gamma, float lambda, int64_t N, int64_t T, int64_t ld,
                float *advantages, float *returns, void *workspace, size_t workspace_bytes,
                void *stream);

int rlca_vtrace_ex(const float *reward, const float *value, const float *log_rho,
                   const uint8_t *terminated, const uint8_t *truncated,
                   const float *trunc_value, const float *bootstrap, float gamma,
                   float lambda, float rho_bar, float c_bar, float pg_rho_bar, int64_t N,
                   int64_t T, int64_t ld, float *vs, float *pg_advantages, void *workspace,
                   size_t workspace_bytes, void *stream);

int rlca_retrace_ex(const float *reward, const float *q_taken, const float *expected_q,
                    const float *rho, const uint8_t *terminated, const uint8_t *truncated,
                    const float *trunc_value, const float *bootstrap_ev, float gamma,
                    float lambda, int64_t N, int64_t T, int64_t ld, float *q_ret,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Testing only: runs the look-back discounted return (gamma 0.99, no truncation, no
 * bootstrap, ld = T) with every tile withholding its state, so each waiting tile gives
 * up after `spin_limit` empty polls. Afterwards rlca_workspace_check returns
 * RLCA_ERR_TIMEOUT and the workspace is ready for normal calls again. Needs T > 1024
 * and spin_limit > 0 (else RLCA_ERR_WORKSPACE).
 */
int rlca_testing_lookback_stall(const float *reward, const uint8_t *terminated, int64_t N,
                                int64_t T, float *returns, void *workspace,
                                size_t workspace_bytes, int spin_limit, void *stream);

/*
 * GAE that allocates nothing, for callers that cannot allocate device memory: code
 * that a host framework hands only its input and output buffers (the framework plans
 * all device memory itself), or a loop running under a fixed memory budget where a
 * cudaMalloc could fail or stall the device. The paper has no counterpart to this
 * entry point.
 *
 * Same arguments and results as rlca_gae. Calls that rlca_gae would run without a
 * workspace anyway go to it unchanged, with its error codes: T <= 1024, N at least twice
 * the SM count (304 on GB300: the rows fill the GPU one CTA per row), and malformed
 * shapes. Other calls (T > 1024 and fewer rows) run the look-back path of rlca_gae_ex
 * on a workspace the library keeps in a static device array of
 * 256 + 32 * RLCA_NOALLOC_MAX_TILES bytes (about 1 MiB), which every GPU that loads the
 * library holds until the process exits. They get rlca_gae_ex's checks, in its order;
 * a look-back call of more than RLCA_NOALLOC_MAX_TILES tiles (N * ceil(T / 1024)) fails
 * with RLCA_ERR_WORKSPACE. A call that fails a check enqueues nothing. It calls no
 * allocator.
 *   - Set-up: a look-back call looks up the array's device address with the current
 *     device (cheap; host code cannot use the symbol itself). When the address is new
 *     to the library (the first such call on a device, or after cudaDeviceReset moved
 *     the array) it zeroes the whole array first, synchronously. Make the first call on
 *     each device before any stream capture.
 *   - Every call on a device shares the one array, and the array keeps the previous
 *     call's contents (each call clears, on its stream, the parts that must start at
 *     zero). Calls whose kernels overlap on the GPU race on it: issue them on one
 *     stream, or order them.
 *   - A look-back wait that gives up (about a second without progress) marks the
 *     affected outputs NaN, and the call still returned RLCA_OK: its timeout record sits
 *     in the library's array, which no entry point reads. Callers that must detect it
 *     check the outputs for NaN.
 */
#define RLCA_NOALLOC_MAX_TILES 32768
int rlca_gae_noalloc(const float *reward, const float *value, const uint8_t *terminated,
                     const uint8_t *truncated, const float *trunc_value,
                     const float *bootstrap, float gamma, float lambda, int64_t N, int64_t T,
                     int64_t ld, float *advantages, float *returns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* RLCA_H */
