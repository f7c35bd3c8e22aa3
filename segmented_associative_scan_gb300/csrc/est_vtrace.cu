// Kernels of one estimator (instantiated in a translation unit of its own so the
// library builds in parallel).
#include "launch.cuh"

namespace rlca {
cudaError_t launch_vtrace(const Params &p, int vec, bool streamable, cudaStream_t stream)
{
    return launch_estimator<Est::kVtrace>(p, vec, streamable, stream);
}

cudaError_t launch_vtrace_bf16(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator_bf16<Est::kVtrace>(p, vec, stream);
}
}  // namespace rlca
