// Kernels of one estimator (instantiated in a translation unit of its own so the
// library builds in parallel).
#include "launch.cuh"

namespace rlca {
cudaError_t launch_return(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator<Est::kReturn>(p, vec, stream);
}

cudaError_t launch_return_bf16(const Params &p, int vec, cudaStream_t stream)
{
    return launch_estimator_bf16<Est::kReturn>(p, vec, stream);
}
}  // namespace rlca
