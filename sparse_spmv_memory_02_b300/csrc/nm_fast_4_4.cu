// Instantiation of the vectorised SpMV kernel for the 4:4 pattern
// and of the bulk-staged kernels
// (one file per pattern so the instantiations compile in parallel).
#include "nm_bulk.cuh"
#include "nm_rows.cuh"

namespace nm {
cudaError_t launch_fast_4_4(const SpmvProblem &p, cudaStream_t s)
{
    return launch_fast_pattern<4, 4>(p, s);
}
cudaError_t launch_bulk_4_4(const SpmvProblem &p, cudaStream_t s)
{
    return launch_bulk_pattern<4, 4>(p, s);
}
cudaError_t launch_rows_4_4(const SpmvGroup &g, cudaStream_t s)
{
    return launch_rows_pattern<4, 4>(g, s);
}
}  // namespace nm
