// Instantiation of the vectorised SpMV kernel for the 1:4 pattern
// and of the bulk-staged kernels
// (one file per pattern so the instantiations compile in parallel).
#include "nm_bulk.cuh"
#include "nm_rows.cuh"

namespace nm {
cudaError_t launch_fast_1_4(const SpmvProblem &p, cudaStream_t s)
{
    return launch_fast_pattern<1, 4>(p, s);
}
cudaError_t launch_bulk_1_4(const SpmvProblem &p, cudaStream_t s)
{
    return launch_bulk_pattern<1, 4>(p, s);
}
cudaError_t launch_rows_1_4(const SpmvGroup &g, cudaStream_t s)
{
    return launch_rows_pattern<1, 4>(g, s);
}
}  // namespace nm
