/*
 * nm.h -- C ABI of libnm: N:M structured-sparse matrix-vector products for
 * token-by-token LLM decoding on NVIDIA B300 (sm_103a).
 *
 * What the library computes.  "SparseDecoding: Decoding-Aware Pruning for
 * Accurate and Efficient LLM Inference" (Abstract) states that decoding is
 * memory-bound and dominated by sparse matrix-vector (SpMV) products, and
 * that its system contribution is an N:M sparse matrix-vector kernel with
 * bitmask indexing and fixed-step traversal; "SparseDecoding Makes LLM
 * Pruning Aware of Generation" (Key points) says the same.  The bedrocknews
 * summary of arXiv 2610.12327v1 defines N:M structured sparsity as a fixed
 * ratio of zeros inside small blocks and the product as a sparse matrix times
 * a single vector.  The pages give no layout, interface or code; everything
 * below that they do not state is this library's own reading of them.
 *
 * Packed layout (the "canonical layout"; pack output, SpMV input):
 *   - W is rows x K (output features x input features), K a multiple of M.
 *   - values: fp16, row-major [rows][K/M*N].  The N kept weights of group g
 *     (positions g*M .. g*M+M-1 along K) sit at values[row][g*N + j],
 *     j = 0..N-1, in increasing k.  Every group advances the value index by
 *     exactly N, so no per-row offsets exist (fixed step).
 *   - masks: uint32, row-major [rows][ceil(K/32)].  Bit b of word w is the
 *     keep bit of position k = 32*w + b (least significant bit first); bits
 *     past K are zero.  Because M divides 32, a group never spans two words.
 *   - A valid matrix has exactly N set bits in every group.
 *
 * Conventions shared by every call:
 *   - Pointers named W, mask, values, masks, x, y are DEVICE pointers of the
 *     calling thread's current CUDA device; the caller allocates, owns and
 *     frees them.  The library keeps no pointer after a call returns.
 *   - `stream` is a CUDA stream of that device (the same type as
 *     cudaStream_t; NULL means the legacy default stream).  Work is ordered
 *     on it.
 *   - Supported patterns: M in {4, 8} and 1 <= N <= M.  Patterns with 8 % N
 *     == 0 and K a multiple of 8*M/N take the vectorised kernel; the others
 *     take a scalar kernel with the same results.
 *   - Arguments are checked on the host before anything is launched; a
 *     failing check returns NM_ERR_INVALID_ARG or NM_ERR_UNSUPPORTED and has
 *     no effect.  A failing CUDA call returns NM_ERR_CUDA.  nm_last_error()
 *     then describes the failure.  No C++ exception crosses this interface.
 *   - rows == 0 is an empty problem: the call succeeds and does nothing.
 *   - Per-device state: on its first use on a device the library caches
 *     device attributes and the device addresses of its static device
 *     variables (the error word, nm_pack_noalloc's scratch).  After
 *     cudaDeviceReset on a device, libnm must not be called on that device
 *     again in the same process.
 */
#ifndef NM_H_
#define NM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NM_VERSION 170 /* 1.7.0 */
#define NM_MAX_BATCH 8     /* vectors a product takes on every path */
#define NM_MAX_BATCH_TC 32 /* vectors a 2:4 product on the tensor cores takes */
#define NM_MAX_GROUP 8

/* A CUDA stream handle; identical to cudaStream_t. */
typedef struct CUstream_st *nm_stream_t;

typedef enum nm_status {
    NM_OK = 0,
    NM_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or stride    */
    NM_ERR_UNSUPPORTED = 2, /* N:M pattern outside M in {4,8}, 1 <= N <= M    */
    NM_ERR_BAD_MASK = 3,    /* nm_pack: some group does not keep exactly N     */
    NM_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed     */
} nm_status;

typedef enum nm_dtype {
    NM_F16 = 0, /* IEEE binary16, rounded to nearest even */
    NM_F32 = 1  /* IEEE binary32                          */
} nm_dtype;

/* A packed N:M matrix (see "Packed layout" above).  `values` and `masks`
 * are device pointers owned by the caller; both must be 16-byte aligned. */
typedef struct nm_matrix {
    int64_t rows;            /* output features, >= 0                */
    int64_t K;               /* input features, >= 0, multiple of M  */
    int32_t N;               /* kept weights per group               */
    int32_t M;               /* group length along K: 4 or 8         */
    const void *values;      /* fp16 [rows][K/M*N]                   */
    const uint32_t *masks;   /* uint32 [rows][ceil(K/32)]            */
} nm_matrix;

/*
 * Byte sizes of the packed arrays for a rows x K matrix with pattern N:M
 * (host only; no CUDA call).  values_bytes = rows*(K/M)*N*2,
 * mask_bytes = rows*ceil(K/32)*4.  Either output pointer may be NULL.
 * Errors: NM_ERR_INVALID_ARG for negative sizes, K not a multiple of M or
 * a size that overflows size_t; NM_ERR_UNSUPPORTED for the pattern.
 */
nm_status nm_packed_sizes(int64_t rows, int64_t K, int N, int M,
                          size_t *values_bytes, size_t *mask_bytes);

/*
 * Compress a dense fp16 matrix and its keep-mask into the packed layout
 * (the representation step that "SparseDecoding: Why Pruning Should Account
 * for How LLMs Generate", section 6, leaves open; bit-exact copy of the kept
 * fp16 bit patterns, including -0.0, subnormals and NaN payloads).
 *   W      fp16 [rows][K], row-major, device.
 *   mask   uint8 [rows][K], row-major, device; nonzero = keep.  The mask, not
 *          the value, decides what is kept: a kept zero is stored.
 *   values fp16 [rows][K/M*N] and masks uint32 [rows][ceil(K/32)], device,
 *          written completely (16-byte aligned).
 * The call allocates a 4-byte device counter, validates every group and
 * SYNCHRONISES `stream` to read it back, so it cannot be captured in a CUDA
 * graph (capturing streams are refused with NM_ERR_INVALID_ARG).
 * Returns NM_ERR_BAD_MASK if any group does not hold exactly N set bits; the
 * outputs are then fully written but their contents are unspecified.
 */
nm_status nm_pack(const void *W, const uint8_t *mask, int64_t rows, int64_t K,
                  int N, int M, void *values, uint32_t *masks, nm_stream_t stream);

/*
 * nm_pack for callers that cannot let a library allocate device memory.
 * The pages have no counterpart to this call; it exists for deployment.
 * Who needs it: an engine that reserves almost all device memory for its
 * own pools before loading this library (an extra allocation would fail or
 * fragment them), a runtime with a fixed device-memory budget, or code that
 * must not risk the implicit device synchronisation an allocation or a free
 * can cause.  nm_pack needs four bytes of device scratch (its bad-group
 * counter) and allocates them on every call; this variant counts into a
 * static array of NM_NOALLOC_SCRATCH_BYTES bytes compiled into the library
 * (present on every GPU that loads the library, until the process exits)
 * and calls no allocating routine.
 *   Arguments, layout, results and errors are those of nm_pack, plus:
 *   - rows*(K/M) above NM_PACK_NOALLOC_MAX_GROUPS (what the 32-bit counter
 *     can count) is rejected with NM_ERR_INVALID_ARG;
 *   - like nm_pack it SYNCHRONISES `stream` to read the counter back, so it
 *     cannot be captured in a CUDA graph: a capturing stream is refused with
 *     NM_ERR_INVALID_ARG before anything is queued (the capture stays valid);
 *   - the first call on a device, made with that device current, looks up
 *     the array's device address (cudaGetSymbolAddress) and caches it (see
 *     "Per-device state" above);
 *   - every call on a device shares the array and clears the counter first;
 *     two calls that overlap on the GPU (for example on different streams)
 *     race on it and may report wrong counts.
 */
#define NM_NOALLOC_SCRATCH_BYTES 256
#define NM_PACK_NOALLOC_MAX_GROUPS 4294967295LL
nm_status nm_pack_noalloc(const void *W, const uint8_t *mask, int64_t rows, int64_t K,
                          int N, int M, void *values, uint32_t *masks, nm_stream_t stream);

/*
 * Expand a packed matrix back to dense fp16 [rows][K] (dropped positions
 * become +0.0).  A test and debugging aid; asynchronous on `stream`.
 * W_out: device, 2-byte aligned, rows*K*2 bytes, overwritten.
 */
nm_status nm_unpack(const nm_matrix *A, void *W_out, nm_stream_t stream);

/*
 * The decode-step product y = A x for one vector ("SparseDecoding:
 * Decoding-Aware Pruning for Accurate and Efficient LLM Inference",
 * Abstract: the N:M sparse matrix-vector kernel; bedrocknews summary of
 * arXiv 2610.12327v1: a sparse matrix times a single vector).
 *   A      packed matrix (host struct, device arrays).
 *   x      fp16 [K], device, 16-byte aligned.
 *   y      [rows] of y_type, device, naturally aligned; overwritten
 *          (no alpha/beta).  If K == 0, y is set to zero.
 * Products and sums are carried in fp32; y is rounded once at the end.
 * Asynchronous: never synchronises, allocates nothing, and may be captured
 * in a CUDA graph.  Results for a matrix with invalid groups are unspecified
 * (never out of bounds).
 * Overlap with the preceding kernel: the call is launched with programmatic
 * dependent launch, so it may start streaming A's packed arrays while the
 * kernel before it in `stream` is still running; it reads x and writes y only
 * after that kernel has completed.  A's arrays must therefore not be written
 * by the kernel immediately before the call.  The library's own writers are
 * safe to precede it: nm_pack and nm_pack_noalloc synchronise, and
 * nm_prune_pack ends with a launch that does not overlap.  A caller's own
 * kernel that writes the packed arrays needs something in between (an event
 * wait, a memcpy, or any ordinary kernel launch).  NM_BULK_TUNE=pdl=0 in the
 * environment turns the overlap off.
 */
nm_status nm_spmv(const nm_matrix *A, const void *x, void *y, nm_dtype y_type,
                  nm_stream_t stream);

/*
 * The same product for 1 <= batch <= NM_MAX_BATCH vectors sharing one pass
 * over A (each weight byte is read once and used `batch` times).  A 2:4
 * matrix that the tensor-core path can run (below) takes up to
 * NM_MAX_BATCH_TC vectors; above NM_MAX_BATCH any other matrix returns
 * NM_ERR_UNSUPPORTED (as does NM_BULK_TUNE=tc=0), and a batch outside
 * [1, NM_MAX_BATCH_TC] NM_ERR_INVALID_ARG.
 *   x  fp16 [batch][ldx], device; ldx >= K; with batch > 1, ldx must be a
 *      multiple of 8 so that every vector starts 16-byte aligned.
 *   y  y_type [batch][ldy], device; ldy >= rows.  Row b of y receives A x_b.
 * Same semantics and errors as nm_spmv.  A 2:4 matrix with K a multiple of
 * 128, at most 256 rows per SM and x and the packed arrays 16-byte aligned
 * is multiplied on the tensor cores when that is faster: from batch 5 on
 * layers of at least 4 Mi weights (rows x K), at batch 3-4 above 24 M, at
 * batch 2 from 128 Mi with at most 128 rows per SM, and always above
 * NM_MAX_BATCH.  Layers of at most one
 * 128-row tile per SM then split K over thread-block clusters of 2, 4 or 8
 * CTAs.  The packed values are then the compressed operand of the
 * sparse tensor-core MMA (the mask bits become its metadata on chip) and
 * products are summed with fp32 accumulation in another order, within the
 * same error bound and deterministic from call to call; that path overlaps
 * the preceding kernel as nm_spmv does.  NM_BULK_TUNE=tc=0 turns it off, tc=1
 * takes it for every 2:4 product it can run; tc_sp=0 selects the earlier
 * variant that expands the groups to dense fp16 in tensor memory.
 */
nm_status nm_spmv_batched(const nm_matrix *A, const void *x, int64_t ldx,
                          void *y, int64_t ldy, int batch, nm_dtype y_type,
                          nm_stream_t stream);

/*
 * Several independent products in one launch: y_i = A_i x_i for i < count
 * (0 <= count <= NM_MAX_GROUP), for the decode-step layers that share an
 * input -- the query, key and value projections of a block all read the
 * attention input, the gate and up projections the MLP input -- so that one
 * launch streams all their weights (fewer launch boundaries per token).
 *   A     host array of `count` packed matrices with the same N, M and K;
 *         rows may differ.
 *   x     host array of `count` device pointers, x[i] fp16 [batch][ldx]
 *         (the same vector may appear several times).
 *   y     host array of `count` device pointers, y[i] y_type [batch][ldy[i]].
 *   ldy   host array of `count` leading dimensions (NULL: ldy[i] = rows_i).
 *   batch, ldx, y_type, stream: as nm_spmv_batched, shared by all products.
 * Each product's arguments are checked as by nm_spmv_batched (errors name
 * the matrix); matrices that differ in N, M or K are NM_ERR_INVALID_ARG.
 * A 2:4 group that the tensor-core path of nm_spmv_batched can run as a
 * whole (every member within its limits, the group's rows together meeting
 * its routing rule) is one launch of that path; otherwise the products share
 * one CUDA-core launch when they can, or are launched one by one (then each
 * on the kernel nm_spmv_batched picks).  Results are within the same error
 * bound and deterministic for a given group; a batch above NM_MAX_BATCH needs
 * every product to be one the tensor-core path runs.
 * Asynchronous, allocates nothing, may be captured in a CUDA graph; the
 * products' y must not overlap.
 */
nm_status nm_spmv_group(const nm_matrix *A, int count, const void *const *x, int64_t ldx,
                        void *const *y, const int64_t *ldy, int batch, nm_dtype y_type,
                        nm_stream_t stream);

/*
 * Decode-only calibration accumulation: H[i][j] += sum_t X[t][i] * X[t][j]
 * for i, j < K, t < T.  SparseDecoding builds each layer's pruning
 * calibration matrix from the layer inputs collected while the dense model
 * generates, the prefill excluded ("SparseDecoding: Decoding-Aware Pruning
 * for Accurate and Efficient LLM Inference", Abstract); the caller passes
 * only decode-step activations, batch by batch, and H accumulates X^T X.
 * Runs on the tensor cores (fp16 products exact, fp32 sums; H is added to
 * with fp32 reductions, so concurrent calls on one H add up, in an
 * unspecified order).
 *   X    fp16 [T][ldx], device, 16-byte aligned; K % 8 == 0, ldx >= K and a
 *        multiple of 8.
 *   H    fp32 [K][ldh], device, 16-byte aligned; ldh >= K, multiple of 4.
 * Errors: NM_ERR_INVALID_ARG for bad sizes, strides or pointers;
 * NM_ERR_UNSUPPORTED if the driver has no tensor-map encoder; NM_ERR_CUDA.
 * Asynchronous, allocates nothing, may be captured in a CUDA graph (the
 * call's tensor map is built on the host at call time).
 */
nm_status nm_calib_accumulate(const void *X, int64_t T, int64_t K, int64_t ldx, float *H,
                              int64_t ldh, nm_stream_t stream);

/*
 * N:M keep-mask from scores, the step before nm_pack in a pruning flow.  In
 * every group of M consecutive weights of a row keep the N of largest score
 * s(r, k) = |W[r][k]| (col_scale NULL: magnitude pruning) or
 * |W[r][k]| * col_scale[k] (a per-input-channel importance, e.g. the norm of
 * input feature k over calibration activations: the activation-weighted
 * magnitude of the Wanda family of training-free pruning methods, the
 * baseline named by the bedrocknews summary of arXiv 2610.12327v1).  Scores
 * are fp32: |w| is exact, the product rounds to nearest.  Position q of a
 * group is kept iff fewer than N positions beat it, q' beating q when
 * s(q') > s(q), or s(q') == s(q) and q' < q (ties go to the lower k), so
 * exactly N are kept unless a score is NaN (then the group is unspecified).
 *   W          fp16 [rows][K], device, 16-byte aligned; K % M == 0.
 *   col_scale  fp32 [K], device, 16-byte aligned, or NULL.
 *   mask       u8 [rows][K], device, 16-byte aligned; 1 = keep, 0 = drop
 *              (the mask nm_pack takes).
 * Errors: as nm_pack's shape checks; NM_ERR_INVALID_ARG for NULL or
 * misaligned pointers.  Asynchronous, allocates nothing, capturable.
 */
nm_status nm_select_mask(const void *W, const float *col_scale, int64_t rows, int64_t K, int N,
                         int M, uint8_t *mask, nm_stream_t stream);

/*
 * nm_select_mask and nm_pack in one pass over W: writes the packed layout
 * (values, masks as for nm_pack) of W pruned by the same rule, without the
 * u8 mask.  Same arguments and errors as nm_select_mask, values and masks as
 * nm_pack (16-byte aligned).  Asynchronous, allocates nothing, capturable
 * (unlike nm_pack it has no invalid groups to report).  An nm_spmv* call
 * made right after it on the same stream may read the packed arrays it
 * writes: the call ends with an ordinary (non-overlapping) launch, so the
 * next call's early weight copies (see nm_spmv) start only after the packed
 * arrays are complete.
 */
nm_status nm_prune_pack(const void *W, const float *col_scale, int64_t rows, int64_t K, int N,
                        int M, void *values, uint32_t *masks, nm_stream_t stream);

/*
 * The gated MLP input of a decoder layer in one pass over both weight
 * matrices: h[b][i] = silu(gate_i . x_b) * (up_i . x_b), silu(g) =
 * g / (1 + exp(-g)), for i < rows and b < batch.  The decoder layers of the
 * model families the pages measure (Llama-3.1, Llama-3.3, Qwen3:
 * "SparseDecoding Makes LLM Pruning Aware of Generation", Introduction)
 * feed their down projection with this product of the gate and up
 * projections, which both read the MLP input; computing it in the SpMV's
 * epilogue saves the two intermediate vectors and a kernel boundary.
 *   gate, up  packed matrices with the same rows, K, N and M.
 *   x         fp16 [batch][ldx], device (as nm_spmv_batched).
 *   h         h_type [batch][ldh], device; ldh >= rows.
 * Both dot products are carried in fp32 as by nm_spmv; silu and the product
 * are evaluated in fp32 and h is rounded once.  Errors as nm_spmv_batched
 * (batch at most NM_MAX_BATCH: a larger one is NM_ERR_UNSUPPORTED);
 * in addition NM_ERR_INVALID_ARG if gate and up differ in shape, and
 * NM_ERR_UNSUPPORTED unless K is a multiple of 128 and 8 % N == 0 (the
 * shapes the streaming kernel takes).  Asynchronous, allocates nothing, may
 * be captured in a CUDA graph; overlaps the preceding kernel as nm_spmv.
 */
nm_status nm_spmv_gate_up_silu(const nm_matrix *gate, const nm_matrix *up, const void *x,
                               int64_t ldx, void *h, int64_t ldh, int batch, nm_dtype h_type,
                               nm_stream_t stream);

/*
 * Read the device error word of the calling thread's current device into
 * *flags and, if `clear` is nonzero, reset it to zero.  A kernel of this
 * library sets NM_DEVERR_PIPE_TIMEOUT when one of its internal pipeline
 * waits (shared-memory barriers between its copy and compute warps) has not
 * completed within about two seconds; the kernel then stops waiting, ends,
 * and the y it wrote is unspecified.  This never happens in a correct run;
 * the word lets a caller check for it after the fact.  The tensor-core
 * product sets NM_DEVERR_SMEM_ALIGN, and writes nothing, if its dynamic
 * shared memory does not start on a 1024-byte boundary (its swizzled copies
 * need that; CUDA places it there).  Synchronises `stream` (so it cannot be
 * captured in a CUDA graph).  A test aid exercises the time-out path without
 * a fault: with NM_BULK_TUNE=wait_fault_test=1 in the environment the
 * streaming SpMV kernel issues no copies and gives up its waits after 2 ms.
 * Errors: NM_ERR_INVALID_ARG (flags NULL, capturing stream), NM_ERR_CUDA.
 */
#define NM_DEVERR_PIPE_TIMEOUT 1u
#define NM_DEVERR_SMEM_ALIGN 2u
nm_status nm_device_errors(uint32_t *flags, int clear, nm_stream_t stream);

/* Static, human-readable name of a status code. */
const char *nm_status_str(nm_status status);

/* Description of the last failing call on the calling thread ("" if none).
 * The pointer stays valid until the thread's next libnm call. */
const char *nm_last_error(void);

/* NM_VERSION of the loaded library. */
int nm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NM_H_ */
