// Kernels of one estimator (instantiated in a translation unit of its own so the
// library builds in parallel).
#include "launch.cuh"

namespace rlca {
cudaError_t launch_gae(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator<Est::kGae>(p, vec, stream);
}

cudaError_t launch_gae_bf16(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator_bf16<Est::kGae>(p, vec, stream);
}
}  // namespace rlca
