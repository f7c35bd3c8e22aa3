// Kernels of one estimator (instantiated in a translation unit of its own so the
// library builds in parallel).
#include "launch.cuh"

namespace rlca {
cudaError_t launch_retrace(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator<Est::kRetrace>(p, vec, stream);
}

cudaError_t launch_retrace_bf16(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator_bf16<Est::kRetrace>(p, vec, stream);
}
}  // namespace rlca
