// Instantiation of the vectorised SpMV kernel for the 1:4 pattern
// (one file per pattern so the instantiations compile in parallel).
#include "nm_fast.cuh"

namespace nm {
cudaError_t launch_fast_1_4(const SpmvProblem &p, cudaStream_t s)
{
    return launch_fast_pattern<1, 4>(p, s);
}
}  // namespace nm
