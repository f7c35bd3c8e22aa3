// One reverse estimator in one input format, compiled once per (estimator, format) pair
// with RLCA_UNIT_EST (the Est value) and RLCA_UNIT_FMT (the Fmt value) set by the build,
// so the library's kernels compile in parallel.
#include "launch.cuh"

#if !defined(RLCA_UNIT_EST) || !defined(RLCA_UNIT_FMT)
#error "reverse_unit.cu is compiled with -DRLCA_UNIT_EST=<0..4> -DRLCA_UNIT_FMT=<0..2>"
#endif

namespace rlca {

template <Est E, Fmt F>
cudaError_t launch_unit(const Params &p, int vec, cudaStream_t stream)
{
    if constexpr (F == Fmt::kF32)
        return launch_estimator<E>(p, vec, stream);
    else
        return launch_estimator_narrow<E, typename FmtType<F>::type>(p, vec, stream);
}

template cudaError_t launch_unit<static_cast<Est>(RLCA_UNIT_EST), static_cast<Fmt>(RLCA_UNIT_FMT)>(
    const Params &, int, cudaStream_t);

}  // namespace rlca
