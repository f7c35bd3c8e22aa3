// C ABI of librlca (declared in include/rlca.h): argument validation, then one fused
// kernel launch on the caller's stream. No allocation, no synchronisation (except in
// rlca_workspace_check, which says so), no change of the current device.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/rlca.h"
#include "launch.cuh"

namespace {

using rlca::Est;
using rlca::Fmt;
using rlca::Params;

// Bytes of one per-step data element in format f.
size_t in_bytes(Fmt f) { return f == Fmt::kF32 ? 4 : 2; }

// The launch function of reverse estimator E in format f, for validate_and_launch.
template <Est E>
auto launcher(Fmt f)
{
    return [f](const Params &q, int vec, cudaStream_t s) {
        return rlca::launch_in_format<E>(f, q, vec, s);
    };
}

struct Range {
    uintptr_t lo, hi;
};

// Bytes spanned by a [N, ld] array of which the first T columns are used.
Range span(const void *p, int64_t N, int64_t T, int64_t ld, size_t elem)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + (uintptr_t)(((N - 1) * ld + T) * (int64_t)elem)};
}

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape check shared by every entry point. Sets *empty for N == 0 or T == 0.
int check_shape(int64_t N, int64_t T, int64_t ld, bool *empty)
{
    if (N < 0 || T < 0 || ld < T || T > RLCA_MAX_T) return RLCA_ERR_SHAPE;
    *empty = (N == 0 || T == 0);
    if (*empty) return RLCA_OK;
    if (ld > INT64_MAX / 8 / N) return RLCA_ERR_SHAPE;
    return RLCA_OK;
}

bool bad_gamma(float g) { return !std::isfinite(g) || g < 0.f; }
bool bad_lambda(float l) { return !(l >= 0.f && l <= 1.f); }
bool bad_clip(float c) { return std::isnan(c) || !(c > 0.f); }

struct Workspace {
    void *ptr;
    size_t bytes;
};

// Where a buffer lives, as the kernels see it.
enum class Mem { kDevice, kManaged, kHost, kBad };

// Device memory of the current device (including managed memory) or pinned host memory
// mapped into the device's address space at the same address (unified addressing).
// Pageable host memory and other devices' memory are kBad.
Mem classify(const void *ptr, int device)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return Mem::kBad;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
        return a.device == device ? Mem::kDevice : Mem::kBad;
    case cudaMemoryTypeManaged:
        return Mem::kManaged;
    case cudaMemoryTypeHost:
        return a.devicePointer == ptr ? Mem::kHost : Mem::kBad;
    default:
        return Mem::kBad;
    }
}

// Common validation of inputs, outputs and workspace, then launch.
// `f32_in` are the required float inputs, `outs` the outputs (outs[0] required).
// `in_elem`: bytes per element of the per-step data inputs (4 = fp32, 2 = bf16 or fp16).
template <typename LaunchFn>
int validate_and_launch(Params &p, const float *const *f32_in, int n_in, float *const *outs,
                        int n_out, Workspace ws, LaunchFn launch, void *stream,
                        size_t in_elem = 4)
{
    // An empty problem is valid whatever the pointers (an empty tensor may have none).
    bool empty = false;
    int st = check_shape(p.N, p.T, p.ld, &empty);
    if (st != RLCA_OK || empty) return st;

    for (int i = 0; i < n_in; ++i)
        if (!f32_in[i]) return RLCA_ERR_NULL;
    if (!p.term || !outs[0]) return RLCA_ERR_NULL;
    if (p.trunc && !p.trunc_value && !p.forward) return RLCA_ERR_NULL;

    // Outputs may overlap neither an input nor each other.
    Range in_ranges[8];
    int k = 0;
    for (int i = 0; i < n_in; ++i) in_ranges[k++] = span(f32_in[i], p.N, p.T, p.ld, in_elem);
    in_ranges[k++] = span(p.term, p.N, p.T, p.ld, 1);
    if (p.trunc) in_ranges[k++] = span(p.trunc, p.N, p.T, p.ld, 1);
    if (p.trunc_value) in_ranges[k++] = span(p.trunc_value, p.N, p.T, p.ld, in_elem);
    if (p.boot) in_ranges[k++] = span(p.boot, 1, p.N, p.N, 4);
    for (int o = 0; o < n_out; ++o) {
        if (!outs[o]) continue;
        const Range ro = span(outs[o], p.N, p.T, p.ld, 4);
        for (int i = 0; i < k; ++i)
            if (overlaps(ro, in_ranges[i])) return RLCA_ERR_ALIAS;
        for (int q = o + 1; q < n_out; ++q)
            if (outs[q] && overlaps(ro, span(outs[q], p.N, p.T, p.ld, 4))) return RLCA_ERR_ALIAS;
    }

    // The workspace is used only when a row spans several tiles.
    p.ws = nullptr;
    const size_t need = rlca::workspace_bytes(p.N, p.T);
    if (ws.ptr && need > 0 && rlca::lookback_tiles(p.N, p.T) <= INT32_MAX) {
        if (ws.bytes < need || !aligned(ws.ptr, 256)) return RLCA_ERR_WORKSPACE;
        const Range rw{reinterpret_cast<uintptr_t>(ws.ptr),
                       reinterpret_cast<uintptr_t>(ws.ptr) + need};
        for (int i = 0; i < k; ++i)
            if (overlaps(rw, in_ranges[i])) return RLCA_ERR_ALIAS;
        for (int o = 0; o < n_out; ++o)
            if (outs[o] && overlaps(rw, span(outs[o], p.N, p.T, p.ld, 4))) return RLCA_ERR_ALIAS;
        p.ws = ws.ptr;
        if (p.spin_limit <= 0) p.spin_limit = rlca::kDefaultSpinLimit;
    }

    // Checked last, as it asks the CUDA runtime: every buffer must be reachable from the
    // current device. Pinned host memory is read and written in place (no bulk copies
    // from it: the kernels then use plain loads and stores).
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        (void)cudaGetLastError();
        return RLCA_ERR_LAUNCH;
    }
    {
        const void *bufs[12];
        int nb = 0;
        for (int i = 0; i < n_in; ++i) bufs[nb++] = f32_in[i];
        bufs[nb++] = p.term;
        if (p.trunc) bufs[nb++] = p.trunc;
        if (p.trunc_value) bufs[nb++] = p.trunc_value;
        if (p.boot) bufs[nb++] = p.boot;
        for (int o = 0; o < n_out; ++o)
            if (outs[o]) bufs[nb++] = outs[o];
        p.host = 0;
        p.prefetch = 1;
        for (int i = 0; i < nb; ++i) {
            const Mem m = classify(bufs[i], device);
            if (m == Mem::kBad) return RLCA_ERR_MEMORY;
            if (m == Mem::kHost) p.host = 1;
            if (m != Mem::kDevice) p.prefetch = 0;  // L2 prefetches: device memory only
        }
        // The look-back state lives in device memory (its waits poll it).
        if (p.ws) {
            const Mem m = classify(p.ws, device);
            if (m != Mem::kDevice && m != Mem::kManaged) return RLCA_ERR_MEMORY;
        }
    }

    // 128-bit loads/stores need 16-byte aligned rows: ld a multiple of 16 bytes of every
    // array (ld % 4 == 0 for fp32, ld % 8 == 0 for 16-bit inputs) and aligned bases.
    bool vec16 = (p.ld % (int64_t)(16 / in_elem)) == 0 && aligned(p.term, 4) &&
                 (!p.trunc || aligned(p.trunc, 4));
    for (int i = 0; i < n_in; ++i) vec16 = vec16 && aligned(f32_in[i], 16);
    for (int o = 0; o < n_out; ++o) vec16 = vec16 && (!outs[o] || aligned(outs[o], 16));
    // 256-bit access to fp32 rows (8 steps per thread in one access) needs 32-byte
    // aligned rows: ld % 8 == 0, fp32 bases 32-byte aligned, flag bases 8-byte aligned
    // (16-bit inputs keep 128-bit loads; only the fp32 outputs widen then).
    bool vec32 = vec16 && (p.ld % 8) == 0 && aligned(p.term, 8) &&
                 (!p.trunc || aligned(p.trunc, 8));
    for (int i = 0; i < n_in; ++i) vec32 = vec32 && (in_elem == 2 || aligned(f32_in[i], 32));
    for (int o = 0; o < n_out; ++o) vec32 = vec32 && (!outs[o] || aligned(outs[o], 32));
    const int vec = vec32 ? 2 : (vec16 ? 1 : 0);

    const cudaError_t err = launch(p, vec, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? RLCA_OK : RLCA_ERR_LAUNCH;
}

Params base_params(const float *reward, const uint8_t *term, const uint8_t *trunc,
                   const float *tv, const float *boot, float gamma, float lambda, int64_t N,
                   int64_t T, int64_t ld)
{
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.reward = reward;
    p.term = term;
    p.trunc = trunc;
    p.trunc_value = trunc ? tv : nullptr;
    p.boot = boot;
    p.N = N;
    p.T = (T < 0 || T > RLCA_MAX_T) ? -1 : (int)T;  // out of range -> RLCA_ERR_SHAPE
    p.ld = ld;
    p.gamma = gamma;
    p.lambda = lambda;
    p.gamma_lambda = gamma * lambda;
    p.gamma_one_m_lambda = gamma * (1.f - lambda);
    p.rho_bar = p.c_bar = p.pg_rho_bar = 1.f;
    return p;
}

// fmt: the format of the per-step data inputs (16-bit formats take no workspace).

int discounted_return(const float *reward, const uint8_t *terminated, const uint8_t *truncated,
                      const float *trunc_value, const float *bootstrap, float gamma, int64_t N,
                      int64_t T, int64_t ld, float *returns, Workspace ws, void *stream,
                      int spin_limit = 0, int stall = 0, Fmt fmt = Fmt::kF32)
{
    if (bad_gamma(gamma)) return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma, 1.f,
                           N, T, ld);
    p.out0 = returns;
    p.spin_limit = spin_limit;
    p.stall = stall;
    const float *in[] = {reward};
    float *out[] = {returns};
    return validate_and_launch(p, in, 1, out, 1, ws, launcher<Est::kReturn>(fmt), stream,
                               in_bytes(fmt));
}

int td_lambda(const float *reward, const float *value, const uint8_t *terminated,
              const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
              float gamma, float lambda, int64_t N, int64_t T, int64_t ld, float *targets,
              Workspace ws, void *stream, Fmt fmt = Fmt::kF32)
{
    if (bad_gamma(gamma) || bad_lambda(lambda)) return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                           lambda, N, T, ld);
    p.value = value;
    p.out0 = targets;
    const float *in[] = {reward, value};
    float *out[] = {targets};
    return validate_and_launch(p, in, 2, out, 1, ws, launcher<Est::kTdLambda>(fmt), stream,
                               in_bytes(fmt));
}

int gae(const float *reward, const float *value, const uint8_t *terminated,
        const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
        float gamma, float lambda, int64_t N, int64_t T, int64_t ld, float *advantages,
        float *returns, Workspace ws, void *stream, Fmt fmt = Fmt::kF32)
{
    if (bad_gamma(gamma) || bad_lambda(lambda)) return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                           lambda, N, T, ld);
    p.value = value;
    p.out0 = advantages;
    p.out1 = returns;
    const float *in[] = {reward, value};
    float *out[] = {advantages, returns};
    return validate_and_launch(p, in, 2, out, 2, ws, launcher<Est::kGae>(fmt), stream,
                               in_bytes(fmt));
}

int vtrace(const float *reward, const float *value, const float *log_rho,
           const uint8_t *terminated, const uint8_t *truncated, const float *trunc_value,
           const float *bootstrap, float gamma, float lambda, float rho_bar, float c_bar,
           float pg_rho_bar, int64_t N, int64_t T, int64_t ld, float *vs,
           float *pg_advantages, Workspace ws, void *stream, Fmt fmt = Fmt::kF32)
{
    if (bad_gamma(gamma) || bad_lambda(lambda) || bad_clip(rho_bar) || bad_clip(c_bar) ||
        bad_clip(pg_rho_bar))
        return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                           lambda, N, T, ld);
    p.value = value;
    p.aux = log_rho;
    p.rho_bar = rho_bar;
    p.c_bar = c_bar;
    p.pg_rho_bar = pg_rho_bar;
    p.out0 = vs;
    p.out1 = pg_advantages;
    const float *in[] = {reward, value, log_rho};
    float *out[] = {vs, pg_advantages};
    return validate_and_launch(p, in, 3, out, 2, ws, launcher<Est::kVtrace>(fmt), stream,
                               in_bytes(fmt));
}

int retrace(const float *reward, const float *q_taken, const float *expected_q,
            const float *rho, const uint8_t *terminated, const uint8_t *truncated,
            const float *trunc_value, const float *bootstrap_ev, float gamma, float lambda,
            int64_t N, int64_t T, int64_t ld, float *q_ret, Workspace ws, void *stream,
            Fmt fmt = Fmt::kF32)
{
    if (bad_gamma(gamma) || bad_lambda(lambda)) return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap_ev, gamma,
                           lambda, N, T, ld);
    p.value = q_taken;
    p.aux = expected_q;
    p.rho = rho;
    p.out0 = q_ret;
    const float *in[] = {reward, q_taken, expected_q, rho};
    float *out[] = {q_ret};
    return validate_and_launch(p, in, 4, out, 1, ws, launcher<Est::kRetrace>(fmt), stream,
                               in_bytes(fmt));
}

int gae_vtrace(const float *reward, const float *value, const float *log_rho,
               const uint8_t *terminated, const uint8_t *truncated, const float *trunc_value,
               const float *bootstrap, float gamma, float lambda_gae, float lambda_vtrace,
               float rho_bar, float c_bar, float pg_rho_bar, int64_t N, int64_t T, int64_t ld,
               float *advantages, float *returns, float *vs, float *pg_advantages, void *stream)
{
    if (bad_gamma(gamma) || bad_lambda(lambda_gae) || bad_lambda(lambda_vtrace) ||
        bad_clip(rho_bar) || bad_clip(c_bar) || bad_clip(pg_rho_bar))
        return RLCA_ERR_PARAM;
    Params pv = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                            lambda_vtrace, N, T, ld);
    pv.value = value;
    pv.aux = log_rho;
    pv.rho_bar = rho_bar;
    pv.c_bar = c_bar;
    pv.pg_rho_bar = pg_rho_bar;
    pv.out0 = vs;
    pv.out1 = pg_advantages;
    Params pg = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                            lambda_gae, N, T, ld);
    pg.value = value;
    pg.out0 = advantages;
    pg.out1 = returns;
    bool empty = false;
    if (check_shape(N, T, ld, &empty) == RLCA_OK && !empty && !advantages) return RLCA_ERR_NULL;
    const float *in[] = {reward, value, log_rho};
    float *out[] = {vs, advantages, returns, pg_advantages};
    auto launch = [&pg](const Params &q, int vec, cudaStream_t s) {
        Params g = pg;  // the same validated shape and memory kind as the V-trace half
        g.host = q.host;
        g.prefetch = q.prefetch;
        return rlca::launch_gae_vtrace(g, q, vec, s);
    };
    return validate_and_launch(pv, in, 3, out, 4, Workspace{nullptr, 0}, launch, stream);
}

int td_lambda_multi(const float *reward, const float *value, const uint8_t *terminated,
                    const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
                    float gamma, const float *lambdas, int n_lambdas, int64_t N, int64_t T,
                    int64_t ld, float *const *targets, void *stream)
{
    if (bad_gamma(gamma)) return RLCA_ERR_PARAM;
    if (n_lambdas < 1 || n_lambdas > RLCA_TD_LAMBDA_MAX) return RLCA_ERR_PARAM;
    if (!lambdas || !targets) return RLCA_ERR_NULL;
    for (int k = 0; k < n_lambdas; ++k)
        if (bad_lambda(lambdas[k])) return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                           lambdas[0], N, T, ld);
    p.value = value;
    p.multi.count = n_lambdas;
    float *outs[RLCA_TD_LAMBDA_MAX] = {};
    for (int k = 0; k < n_lambdas; ++k) {
        p.multi.gamma_lambda[k] = gamma * lambdas[k];
        p.multi.gamma_one_m_lambda[k] = gamma * (1.f - lambdas[k]);
        p.multi.out[k] = outs[k] = targets[k];
    }
    p.out0 = targets[0];
    // Every target is required (an empty problem needs none).
    bool empty = false;
    if (check_shape(N, T, ld, &empty) == RLCA_OK && !empty)
        for (int k = 0; k < n_lambdas; ++k)
            if (!outs[k]) return RLCA_ERR_NULL;
    const float *in[] = {reward, value};
    auto launch = [](const Params &q, int vec, cudaStream_t s) {
        return rlca::launch_td_multi(q, vec, s);
    };
    return validate_and_launch(p, in, 2, outs, n_lambdas, Workspace{nullptr, 0}, launch,
                               stream);
}

// Forward scans: x and flags as the reverse estimators' reward and flags; `init` is the
// per-env value carried into the window (nullable); decay >= 0 and finite.
int forward_scan(const float *x, const uint8_t *terminated, const uint8_t *truncated,
                 const float *init, float decay, int64_t N, int64_t T, int64_t ld, float *out,
                 void *stream, Fmt fmt = Fmt::kF32)
{
    if (!std::isfinite(decay) || decay < 0.f) return RLCA_ERR_PARAM;
    Params p = base_params(x, terminated, truncated, nullptr, init, decay, 1.f, N, T, ld);
    p.trunc = truncated;  // truncation needs no successor values here
    p.forward = 1;
    p.out0 = out;
    const float *in[] = {x};
    float *outs[] = {out};
    auto launch = [fmt](const Params &q, int vec, cudaStream_t s) {
        return rlca::launch_forward_in_format(fmt, q, vec, s);
    };
    return validate_and_launch(p, in, 1, outs, 1, Workspace{nullptr, 0}, launch, stream,
                               in_bytes(fmt));
}

constexpr Workspace kNoWorkspace{nullptr, 0};

}  // namespace

namespace rlca {

int gae_on_library_workspace(const float *reward, const float *value, const uint8_t *terminated,
                             const uint8_t *truncated, const float *trunc_value,
                             const float *bootstrap, float gamma, float lambda, int64_t N,
                             int64_t T, int64_t ld, float *advantages, float *returns,
                             void *ws, size_t ws_bytes,
                             cudaError_t (*prepare)(void *ws, cudaStream_t stream), void *stream)
{
    if (bad_gamma(gamma) || bad_lambda(lambda)) return RLCA_ERR_PARAM;
    Params p = base_params(reward, terminated, truncated, trunc_value, bootstrap, gamma,
                           lambda, N, T, ld);
    p.value = value;
    p.out0 = advantages;
    p.out1 = returns;
    const float *in[] = {reward, value};
    float *out[] = {advantages, returns};
    // Every check has passed once the launch function runs: only then is the workspace
    // prepared, on the same stream, right before the kernel.
    auto launch = [prepare](const Params &q, int vec, cudaStream_t s) {
        if (q.ws) {
            const cudaError_t e = prepare(q.ws, s);
            if (e != cudaSuccess) return e;
        }
        return launch_unit<Est::kGae, Fmt::kF32>(q, vec, s);
    };
    return validate_and_launch(p, in, 2, out, 2, Workspace{ws, ws_bytes}, launch, stream);
}

}  // namespace rlca

extern "C" {

int rlca_version(void) { return 200; }

const char *rlca_status_string(int status)
{
    switch (status) {
    case RLCA_OK: return "ok";
    case RLCA_ERR_NULL: return "a required pointer is NULL";
    case RLCA_ERR_SHAPE: return "invalid shape (N < 0, T < 0, ld < T, T too large, or N*ld overflows)";
    case RLCA_ERR_PARAM: return "invalid parameter (gamma < 0 or not finite, lambda outside [0,1], or a clip <= 0)";
    case RLCA_ERR_ALIAS: return "an output or the workspace overlaps an input or another output";
    case RLCA_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case RLCA_ERR_LAUNCH: return "CUDA call failed";
    case RLCA_ERR_TIMEOUT: return "a bounded cross-block wait timed out";
    case RLCA_ERR_MEMORY: return "a buffer is neither current-device memory nor pinned host memory";
    default: return "unknown status";
    }
}

size_t rlca_workspace_bytes(int64_t N, int64_t T)
{
    if (N <= 0 || T <= 0 || T > RLCA_MAX_T) return 0;
    return rlca::workspace_bytes(N, T);
}

int rlca_workspace_check(void *workspace, void *stream)
{
    if (!workspace) return RLCA_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int *err_dev = &static_cast<rlca::LookbackHeader *>(workspace)->error;
    int err = 0;
    if (cudaMemcpyAsync(&err, err_dev, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return RLCA_ERR_LAUNCH;
    if (err != 0) {
        if (cudaMemsetAsync(err_dev, 0, sizeof(int), s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return RLCA_ERR_LAUNCH;
        return RLCA_ERR_TIMEOUT;
    }
    return RLCA_OK;
}

int rlca_discounted_return(const float *reward, const uint8_t *terminated,
                           const uint8_t *truncated, const float *trunc_value,
                           const float *bootstrap, float gamma, int64_t N, int64_t T,
                           int64_t ld, float *returns, void *stream)
{
    return discounted_return(reward, terminated, truncated, trunc_value, bootstrap, gamma, N, T,
                             ld, returns, kNoWorkspace, stream);
}

int rlca_discounted_return_ex(const float *reward, const uint8_t *terminated,
                              const uint8_t *truncated, const float *trunc_value,
                              const float *bootstrap, float gamma, int64_t N, int64_t T,
                              int64_t ld, float *returns, void *workspace,
                              size_t workspace_bytes, void *stream)
{
    return discounted_return(reward, terminated, truncated, trunc_value, bootstrap, gamma, N, T,
                             ld, returns, Workspace{workspace, workspace_bytes}, stream);
}

int rlca_td_lambda(const float *reward, const float *value, const uint8_t *terminated,
                   const uint8_t *truncated, const float *trunc_value,
                   const float *bootstrap, float gamma, float lambda, int64_t N,
                   int64_t T, int64_t ld, float *targets, void *stream)
{
    return td_lambda(reward, value, terminated, truncated, trunc_value, bootstrap, gamma,
                     lambda, N, T, ld, targets, kNoWorkspace, stream);
}

int rlca_td_lambda_ex(const float *reward, const float *value, const uint8_t *terminated,
                      const uint8_t *truncated, const float *trunc_value,
                      const float *bootstrap, float gamma, float lambda, int64_t N,
                      int64_t T, int64_t ld, float *targets, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    return td_lambda(reward, value, terminated, truncated, trunc_value, bootstrap, gamma,
                     lambda, N, T, ld, targets, Workspace{workspace, workspace_bytes}, stream);
}

int rlca_gae(const float *reward, const float *value, const uint8_t *terminated,
             const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
             float gamma, float lambda, int64_t N, int64_t T, int64_t ld,
             float *advantages, float *returns, void *stream)
{
    return gae(reward, value, terminated, truncated, trunc_value, bootstrap, gamma, lambda, N,
               T, ld, advantages, returns, kNoWorkspace, stream);
}

int rlca_gae_ex(const float *reward, const float *value, const uint8_t *terminated,
                const uint8_t *truncated, const float *trunc_value, const float *bootstrap,
                float gamma, float lambda, int64_t N, int64_t T, int64_t ld,
                float *advantages, float *returns, void *workspace, size_t workspace_bytes,
                void *stream)
{
    return gae(reward, value, terminated, truncated, trunc_value, bootstrap, gamma, lambda, N,
               T, ld, advantages, returns, Workspace{workspace, workspace_bytes}, stream);
}

int rlca_vtrace(const float *reward, const float *value, const float *log_rho,
                const uint8_t *terminated, const uint8_t *truncated,
                const float *trunc_value, const float *bootstrap, float gamma,
                float lambda, float rho_bar, float c_bar, float pg_rho_bar, int64_t N,
                int64_t T, int64_t ld, float *vs, float *pg_advantages, void *stream)
{
    return vtrace(reward, value, log_rho, terminated, truncated, trunc_value, bootstrap, gamma,
                  lambda, rho_bar, c_bar, pg_rho_bar, N, T, ld, vs, pg_advantages,
                  kNoWorkspace, stream);
}

int rlca_vtrace_ex(const float *reward, const float *value, const float *log_rho,
                   const uint8_t *terminated, const uint8_t *truncated,
                   const float *trunc_value, const float *bootstrap, float gamma,
                   float lambda, float rho_bar, float c_bar, float pg_rho_bar, int64_t N,
                   int64_t T, int64_t ld, float *vs, float *pg_advantages, void *workspace,
                   size_t workspace_bytes, void *stream)
{
    return vtrace(reward, value, log_rho, terminated, truncated, trunc_value, bootstrap, gamma,
                  lambda, rho_bar, c_bar, pg_rho_bar, N, T, ld, vs, pg_advantages,
                  Workspace{workspace, workspace_bytes}, stream);
}

int rlca_retrace(const float *reward, const float *q_taken, const float *expected_q,
                 const float *rho, const uint8_t *terminated, const uint8_t *truncated,
                 const float *trunc_value, const float *bootstrap_ev, float gamma,
                 float lambda, int64_t N, int64_t T, int64_t ld, float *q_ret,
                 void *stream)
{
    return retrace(reward, q_taken, expected_q, rho, terminated, truncated, trunc_value,
                   bootstrap_ev, gamma, lambda, N, T, ld, q_ret, kNoWorkspace, stream);
}

int rlca_retrace_ex(const float *reward, const float *q_taken, const float *expected_q,
                    const float *rho, const uint8_t *terminated, const uint8_t *truncated,
                    const float *trunc_value, const float *bootstrap_ev, float gamma,
                    float lambda, int64_t N, int64_t T, int64_t ld, float *q_ret,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    return retrace(reward, q_taken, expected_q, rho, terminated, truncated, trunc_value,
                   bootstrap_ev, gamma, lambda, N, T, ld, q_ret,
                   Workspace{workspace, workspace_bytes}, stream);
}

int rlca_td_lambda_multi(const float *reward, const float *value, const uint8_t *terminated,
                         const uint8_t *truncated, const float *trunc_value,
                         const float *bootstrap, float gamma, const float *lambdas,
                         int n_lambdas, int64_t N, int64_t T, int64_t ld,
                         float *const *targets, void *stream)
{
    return td_lambda_multi(reward, value, terminated, truncated, trunc_value, bootstrap, gamma,
                           lambdas, n_lambdas, N, T, ld, targets, stream);
}

int rlca_gae_vtrace(const float *reward, const float *value, const float *log_rho,
                    const uint8_t *terminated, const uint8_t *truncated,
                    const float *trunc_value, const float *bootstrap, float gamma,
                    float lambda_gae, float lambda_vtrace, float rho_bar, float c_bar,
                    float pg_rho_bar, int64_t N, int64_t T, int64_t ld, float *advantages,
                    float *returns, float *vs, float *pg_advantages, void *stream)
{
    return gae_vtrace(reward, value, log_rho, terminated, truncated, trunc_value, bootstrap,
                      gamma, lambda_gae, lambda_vtrace, rho_bar, c_bar, pg_rho_bar, N, T, ld,
                      advantages, returns, vs, pg_advantages, stream);
}

int rlca_eligibility_trace(const float *x, const uint8_t *terminated,
                           const uint8_t *truncated, const float *init, float decay, int64_t N,
                           int64_t T, int64_t ld, float *traces, void *stream)
{
    return forward_scan(x, terminated, truncated, init, decay, N, T, ld, traces, stream);
}

int rlca_episodic_prefix_sum(const float *x, const uint8_t *terminated,
                             const uint8_t *truncated, const float *init, int64_t N, int64_t T,
                             int64_t ld, float *sums, void *stream)
{
    return forward_scan(x, terminated, truncated, init, 1.f, N, T, ld, sums, stream);
}

// ---- 16-bit per-step inputs (bf16 or fp16 bit patterns), fp32 bootstrap values and
// outputs: the same seven entry points for each format, SUFFIX _bf16 or _fp16.

#define RLCA_IN(p) reinterpret_cast<const float *>(p)
#define RLCA_NARROW_ENTRY_POINTS(SUFFIX, FMT)                                                   \
    int rlca_discounted_return##SUFFIX(const uint16_t *reward, const uint8_t *terminated,       \
                                       const uint8_t *truncated, const uint16_t *trunc_value,   \
                                       const float *bootstrap, float gamma, int64_t N,          \
                                       int64_t T, int64_t ld, float *returns, void *stream)     \
    {                                                                                           \
        return discounted_return(RLCA_IN(reward), terminated, truncated, RLCA_IN(trunc_value), \
                                 bootstrap, gamma, N, T, ld, returns, kNoWorkspace, stream, 0, \
                                 0, FMT);                                                       \
    }                                                                                           \
    int rlca_td_lambda##SUFFIX(const uint16_t *reward, const uint16_t *value,                   \
                               const uint8_t *terminated, const uint8_t *truncated,             \
                               const uint16_t *trunc_value, const float *bootstrap,             \
                               float gamma, float lambda, int64_t N, int64_t T, int64_t ld,     \
                               float *targets, void *stream)                                    \
    {                                                                                           \
        return td_lambda(RLCA_IN(reward), RLCA_IN(value), terminated, truncated,                \
                         RLCA_IN(trunc_value), bootstrap, gamma, lambda, N, T, ld, targets,     \
                         kNoWorkspace, stream, FMT);                                            \
    }                                                                                           \
    int rlca_gae##SUFFIX(const uint16_t *reward, const uint16_t *value,                         \
                         const uint8_t *terminated, const uint8_t *truncated,                   \
                         const uint16_t *trunc_value, const float *bootstrap, float gamma,      \
                         float lambda, int64_t N, int64_t T, int64_t ld, float *advantages,     \
                         float *returns, void *stream)                                          \
    {                                                                                           \
        return gae(RLCA_IN(reward), RLCA_IN(value), terminated, truncated,                      \
                   RLCA_IN(trunc_value), bootstrap, gamma, lambda, N, T, ld, advantages,        \
                   returns, kNoWorkspace, stream, FMT);                                         \
    }                                                                                           \
    int rlca_vtrace##SUFFIX(const uint16_t *reward, const uint16_t *value,                      \
                            const uint16_t *log_rho, const uint8_t *terminated,                 \
                            const uint8_t *truncated, const uint16_t *trunc_value,              \
                            const float *bootstrap, float gamma, float lambda, float rho_bar,   \
                            float c_bar, float pg_rho_bar, int64_t N, int64_t T, int64_t ld,    \
                            float *vs, float *pg_advantages, void *stream)                      \
    {                                                                                           \
        return vtrace(RLCA_IN(reward), RLCA_IN(value), RLCA_IN(log_rho), terminated,           \
                      truncated, RLCA_IN(trunc_value), bootstrap, gamma, lambda, rho_bar,       \
                      c_bar, pg_rho_bar, N, T, ld, vs, pg_advantages, kNoWorkspace, stream,     \
                      FMT);                                                                     \
    }                                                                                           \
    int rlca_retrace##SUFFIX(const uint16_t *reward, const uint16_t *q_taken,                   \
                             const uint16_t *expected_q, const uint16_t *rho,                   \
                             const uint8_t *terminated, const uint8_t *truncated,               \
                             const uint16_t *trunc_value, const float *bootstrap_ev,            \
                             float gamma, float lambda, int64_t N, int64_t T, int64_t ld,       \
                             float *q_ret, void *stream)                                        \
    {                                                                                           \
        return retrace(RLCA_IN(reward), RLCA_IN(q_taken), RLCA_IN(expected_q), RLCA_IN(rho),   \
                       terminated, truncated, RLCA_IN(trunc_value), bootstrap_ev, gamma,        \
                       lambda, N, T, ld, q_ret, kNoWorkspace, stream, FMT);                     \
    }                                                                                           \
    int rlca_eligibility_trace##SUFFIX(const uint16_t *x, const uint8_t *terminated,            \
                                       const uint8_t *truncated, const float *init,             \
                                       float decay, int64_t N, int64_t T, int64_t ld,           \
                                       float *traces, void *stream)                             \
    {                                                                                           \
        return forward_scan(RLCA_IN(x), terminated, truncated, init, decay, N, T, ld, traces,   \
                            stream, FMT);                                                       \
    }                                                                                           \
    int rlca_episodic_prefix_sum##SUFFIX(const uint16_t *x, const uint8_t *terminated,          \
                                         const uint8_t *truncated, const float *init,           \
                                         int64_t N, int64_t T, int64_t ld, float *sums,         \
                                         void *stream)                                          \
    {                                                                                           \
        return forward_scan(RLCA_IN(x), terminated, truncated, init, 1.f, N, T, ld, sums,       \
                            stream, FMT);                                                       \
    }

RLCA_NARROW_ENTRY_POINTS(_bf16, Fmt::kBF16)
RLCA_NARROW_ENTRY_POINTS(_fp16, Fmt::kF16)

#undef RLCA_NARROW_ENTRY_POINTS
#undef RLCA_IN

int rlca_testing_lookback_stall(const float *reward, const uint8_t *terminated, int64_t N,
                                int64_t T, float *returns, void *workspace,
                                size_t workspace_bytes, int spin_limit, void *stream)
{
    if (!workspace || rlca::workspace_bytes(N, T) == 0 || spin_limit <= 0)
        return RLCA_ERR_WORKSPACE;
    return discounted_return(reward, terminated, nullptr, nullptr, nullptr, 0.99f, N, T, T,
                             returns, Workspace{workspace, workspace_bytes}, stream, spin_limit,
                             1);
}

}  // extern "C"
