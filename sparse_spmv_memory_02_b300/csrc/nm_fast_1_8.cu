// Instantiation of the vectorised SpMV kernel for the 1:8 pattern
// (one file per pattern so the instantiations compile in parallel).
#include "nm_fast.cuh"

namespace nm {
cudaError_t launch_fast_1_8(const SpmvProblem &p, cudaStream_t s)
{
    return launch_fast_pattern<1, 8>(p, s);
}
}  // namespace nm
