/*
 * nm_probe.h -- measurement aid shipped in libnm: a read-only HBM stream.
 *
 * The N:M sparse matrix-vector product of "SparseDecoding: Decoding-Aware
 * Pruning for Accurate and Efficient LLM Inference" (Abstract) is a pure
 * weight stream during decoding, so its speed is judged against the rate at
 * which this GPU can read memory at all.  A copy benchmark moves as many
 * bytes in as out; the product only reads, so the library carries its own
 * read-only stream to time beside it.  The pages have no counterpart to this
 * call.  Same conventions as nm.h (device pointers owned by the caller,
 * status codes, no exception crosses the interface).
 */
#ifndef NM_PROBE_H_
#define NM_PROBE_H_

#include "nm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Read `bytes` of `buf` once with 16-byte loads that bypass L1 (one CTA of
 * 1024 threads per SM, four loads in flight per thread) and write the XOR of
 * all words read into *sink, so that no load can be dropped.
 *   buf    device, 16-byte aligned; bytes a multiple of 16 (0: no effect).
 *   sink   device, 4 bytes, overwritten.
 * Asynchronous on `stream`, allocates nothing, may be captured in a CUDA
 * graph.  Time it over a buffer several times larger than L2 so that the
 * reads come from HBM.
 * Errors: NM_ERR_INVALID_ARG (NULL or misaligned pointer, bytes not a
 * multiple of 16), NM_ERR_CUDA.
 */
nm_status nm_probe_read_stream(const void *buf, size_t bytes, uint32_t *sink,
                               nm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NM_PROBE_H_ */
