// Instantiation of the vectorised SpMV kernel for the 2:8 pattern
// (one file per pattern so the instantiations compile in parallel).
#include "nm_fast.cuh"

namespace nm {
cudaError_t launch_fast_2_8(const SpmvProblem &p, cudaStream_t s)
{
    return launch_fast_pattern<2, 8>(p, s);
}
}  // namespace nm
