/* A plain C (C99) program that uses libnm through its public headers only:
 * it must compile as C, link against libnm.so and get the host-only calls'
 * answers without a GPU (built and run by tests/test_c_consumer.py). */
#include <stdio.h>
#include <string.h>

#include "nm.h"
#include "nm_probe.h"

int main(void)
{
    size_t vb = 0, mb = 0;
    int fails = 0;
    if (nm_version() != NM_VERSION) { printf("version %d\n", nm_version()); ++fails; }
    if (nm_packed_sizes(4096, 4096, 2, 4, &vb, &mb) != NM_OK || vb != 4096u * 2048u * 2u ||
        mb != 4096u * 128u * 4u) { printf("sizes %zu %zu\n", vb, mb); ++fails; }
    if (nm_packed_sizes(4, 18, 2, 4, &vb, &mb) != NM_ERR_INVALID_ARG) { printf("K %% M\n"); ++fails; }
    if (strcmp(nm_status_str(NM_ERR_BAD_MASK), "NM_ERR_BAD_MASK") != 0) { printf("str\n"); ++fails; }
    /* argument checks happen on the host before any CUDA call */
    nm_matrix A = {64, 256, 2, 4, NULL, NULL};
    if (nm_spmv(&A, NULL, NULL, NM_F16, NULL) != NM_ERR_INVALID_ARG) { printf("spmv\n"); ++fails; }
    if (nm_last_error()[0] == 0) { printf("no message\n"); ++fails; }
    if (nm_probe_read_stream(NULL, 64, NULL, NULL) != NM_ERR_INVALID_ARG) { printf("probe\n"); ++fails; }
    printf(fails ? "FAIL\n" : "OK\n");
    return fails ? 1 : 0;
}
