// C entry points of libnm (declared in include/nm.h): argument checks on the
// host, then one kernel launch.  No exception crosses this file's functions.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>

#include "nm.h"
#include "nm_internal.h"

namespace nm {
cudaError_t launch_fast_1_4(const SpmvProblem &, cudaStream_t);
cudaError_t launch_fast_2_4(const SpmvProblem &, cudaStream_t);
cudaError_t launch_fast_4_4(const SpmvProblem &, cudaStream_t);
cudaError_t launch_fast_1_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_fast_2_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_fast_4_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_fast_8_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_1_4(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_2_4(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_4_4(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_1_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_2_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_4_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_bulk_8_8(const SpmvProblem &, cudaStream_t);
cudaError_t launch_rows_1_4(const SpmvGroup &, cudaStream_t);
cudaError_t launch_rows_2_4(const SpmvGroup &, cudaStream_t);
cudaError_t launch_rows_4_4(const SpmvGroup &, cudaStream_t);
cudaError_t launch_rows_1_8(const SpmvGroup &, cudaStream_t);
cudaError_t launch_rows_2_8(const SpmvGroup &, cudaStream_t);
cudaError_t launch_rows_4_8(const SpmvGroup &, cudaStream_t);
cudaError_t launch_rows_8_8(const SpmvGroup &, cudaStream_t);

bool fast_path_applies(int N, int M, int64_t K)
{
    if (M != 4 && M != 8) return false;
    if (N < 1 || N > M || 8 % N != 0) return false;
    const int64_t ck = 8 * M / N;  // positions covered by one 16-byte value chunk
    return K > 0 && K % ck == 0 && K / ck <= INT_MAX / 2;
}

bool bulk_path_applies(int N, int M, int64_t K)
{
    return fast_path_applies(N, M, K) && K % 128 == 0;
}

cudaError_t launch_rows(const SpmvGroup &g, cudaStream_t s)
{
    switch (g.p[0].M * 16 + g.p[0].N) {
    case 4 * 16 + 1: return launch_rows_1_4(g, s);
    case 4 * 16 + 2: return launch_rows_2_4(g, s);
    case 4 * 16 + 4: return launch_rows_4_4(g, s);
    case 8 * 16 + 1: return launch_rows_1_8(g, s);
    case 8 * 16 + 2: return launch_rows_2_8(g, s);
    case 8 * 16 + 4: return launch_rows_4_8(g, s);
    case 8 * 16 + 8: return launch_rows_8_8(g, s);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_bulk(const SpmvProblem &p, cudaStream_t s)
{
    switch (p.M * 16 + p.N) {
    case 4 * 16 + 1: return launch_bulk_1_4(p, s);
    case 4 * 16 + 2: return launch_bulk_2_4(p, s);
    case 4 * 16 + 4: return launch_bulk_4_4(p, s);
    case 8 * 16 + 1: return launch_bulk_1_8(p, s);
    case 8 * 16 + 2: return launch_bulk_2_8(p, s);
    case 8 * 16 + 4: return launch_bulk_4_8(p, s);
    case 8 * 16 + 8: return launch_bulk_8_8(p, s);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_fast(const SpmvProblem &p, cudaStream_t s)
{
    switch (p.M * 16 + p.N) {
    case 4 * 16 + 1: return launch_fast_1_4(p, s);
    case 4 * 16 + 2: return launch_fast_2_4(p, s);
    case 4 * 16 + 4: return launch_fast_4_4(p, s);
    case 8 * 16 + 1: return launch_fast_1_8(p, s);
    case 8 * 16 + 2: return launch_fast_2_8(p, s);
    case 8 * 16 + 4: return launch_fast_4_8(p, s);
    case 8 * 16 + 8: return launch_fast_8_8(p, s);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace nm

namespace {

thread_local char g_last_error[512];

// The device error word: kernels set bits in it when an internal pipeline
// wait gives up (see nm_device_errors).  Its device address is looked up
// once per device.
__device__ unsigned int g_device_error;
constexpr int kMaxDevices = 64;
std::atomic<unsigned int *> g_error_ptr[kMaxDevices];

cudaError_t device_error_word(unsigned int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned int *p = g_error_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        void *v = nullptr;
        e = cudaGetSymbolAddress(&v, g_device_error);
        if (e != cudaSuccess) return e;
        p = static_cast<unsigned int *>(v);
        g_error_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

nm_status fail(nm_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

nm_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(NM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// rows and K bounds keep every index of the kernels inside int64 and the
// per-launch row count inside int.
constexpr int64_t kMaxRows = INT_MAX;
constexpr int64_t kMaxK = INT_MAX;

nm_status check_shape(int64_t rows, int64_t K, int N, int M)
{
    if (M != 4 && M != 8) return fail(NM_ERR_UNSUPPORTED, "M=%d: only M in {4, 8} is supported", M);
    if (N < 1 || N > M)
        return fail(NM_ERR_UNSUPPORTED, "N=%d: need 1 <= N <= M (M=%d)", N, M);
    if (rows < 0 || K < 0) return fail(NM_ERR_INVALID_ARG, "negative size rows=%lld K=%lld",
                                       (long long)rows, (long long)K);
    if (rows > kMaxRows || K > kMaxK)
        return fail(NM_ERR_INVALID_ARG, "size too large rows=%lld K=%lld (max %lld each)",
                    (long long)rows, (long long)K, (long long)INT_MAX);
    if (K % M != 0)
        return fail(NM_ERR_INVALID_ARG, "K=%lld is not a multiple of M=%d", (long long)K, M);
    return NM_OK;
}

nm_status check_matrix(const nm_matrix *A)
{
    if (!A) return fail(NM_ERR_INVALID_ARG, "matrix descriptor is NULL");
    nm_status st = check_shape(A->rows, A->K, A->N, A->M);
    if (st != NM_OK) return st;
    if (A->rows > 0 && A->K > 0) {
        if (!A->values || !A->masks) return fail(NM_ERR_INVALID_ARG, "values or masks is NULL");
        if (!aligned(A->values, 16) || !aligned(A->masks, 16))
            return fail(NM_ERR_INVALID_ARG, "values and masks must be 16-byte aligned");
    }
    return NM_OK;
}

bool takes_tensor_cores(const nm::SpmvProblem &p, uint32_t *lbo_enc);

// Checks the arguments of one product y = A x (batch vectors) and fills `p`.
// Sets *empty, having done the whole job, when rows == 0 (nothing to do) or
// K == 0 (y is zeroed on `s`).
nm_status prepare_product(const nm_matrix *A, const void *x, int64_t ldx, void *y, int64_t ldy,
                          int batch, nm_dtype y_type, nm::SpmvProblem *p, bool *empty,
                          cudaStream_t s)
{
    *empty = false;
    nm_status st = check_matrix(A);
    if (st != NM_OK) return st;
    if (batch < 1 || batch > NM_MAX_BATCH_TC)
        return fail(NM_ERR_INVALID_ARG, "batch=%d outside [1, %d]", batch, NM_MAX_BATCH_TC);
    // more than NM_MAX_BATCH vectors: only the 2:4 tensor-core product (the
    // rest of its conditions is checked below, once the device is known)
    if (batch > NM_MAX_BATCH && !(A->N == 2 && A->M == 4 && A->K % 128 == 0))
        return fail(NM_ERR_UNSUPPORTED,
                    "batch=%d > %d needs a 2:4 matrix with K a multiple of 128 (the tensor-core "
                    "path)", batch, NM_MAX_BATCH);
    if (y_type != NM_F16 && y_type != NM_F32)
        return fail(NM_ERR_INVALID_ARG, "unknown y_type %d", (int)y_type);
    const size_t esize = y_type == NM_F32 ? 4 : 2;
    if (ldy < A->rows)
        return fail(NM_ERR_INVALID_ARG, "ldy=%lld < rows=%lld", (long long)ldy, (long long)A->rows);
    if (A->K > 0) {
        if (ldx < A->K)
            return fail(NM_ERR_INVALID_ARG, "ldx=%lld < K=%lld", (long long)ldx, (long long)A->K);
        if (batch > 1 && ldx % 8 != 0)
            return fail(NM_ERR_INVALID_ARG, "ldx=%lld must be a multiple of 8 when batch > 1",
                        (long long)ldx);
    }
    if (A->rows == 0) {
        *empty = true;
        return NM_OK;
    }
    if (!y) return fail(NM_ERR_INVALID_ARG, "y is NULL");
    if (!aligned(y, esize)) return fail(NM_ERR_INVALID_ARG, "y is not %zu-byte aligned", esize);
    if (ldy > (INT64_MAX / 16) / batch) return fail(NM_ERR_INVALID_ARG, "ldy too large");
    if (A->K == 0) {  // empty sums: y = 0
        cudaError_t e = cudaMemset2DAsync(y, static_cast<size_t>(ldy) * esize, 0,
                                          static_cast<size_t>(A->rows) * esize, batch, s);
        if (e != cudaSuccess) return cuda_fail(e, "nm_spmv: cudaMemset2DAsync");
        *empty = true;
        return NM_OK;
    }
    if (!x) return fail(NM_ERR_INVALID_ARG, "x is NULL");
    if (!aligned(x, 16)) return fail(NM_ERR_INVALID_ARG, "x must be 16-byte aligned");
    if (ldx > (INT64_MAX / 16) / batch) return fail(NM_ERR_INVALID_ARG, "ldx too large");

    p->rows = A->rows;
    p->K = A->K;
    p->N = A->N;
    p->M = A->M;
    p->values = A->values;
    p->masks = A->masks;
    p->x = x;
    p->ldx = ldx;
    p->y = y;
    p->ldy = ldy;
    p->batch = batch;
    p->y_f32 = y_type == NM_F32;
    if (batch > NM_MAX_BATCH) {
        uint32_t lbo = 0;
        if (!takes_tensor_cores(*p, &lbo))
            return fail(NM_ERR_UNSUPPORTED,
                        "batch=%d > %d: the tensor-core path does not apply (at most 256 rows "
                        "per SM, x, values and masks 16-byte aligned, not turned off)",
                        batch, NM_MAX_BATCH);
    }
    cudaError_t e = device_error_word(&p->err);
    if (e != cudaSuccess) return cuda_fail(e, "nm_spmv: device error word");
    return NM_OK;
}

// One product on the best kernel that applies: the row kernel (any batch;
// K a multiple of 128), the chunk-column kernel (when no row plan fits in
// shared memory), the direct-load kernel, the scalar kernel.
// 2:4 products with several vectors go to the tensor-core product where it
// is faster (measured on the decode shapes, each layer alone).  Its time
// hardly depends on the batch (up to 8): ~4.5 us a launch plus the weights
// at up to ~6.1 TB/s (layers of at most one 128-row tile a SM split K over
// clusters of 2-8 CTAs).  The CUDA-core row kernel is instruction-bound from
// batch 3 and slows with every vector.  Measured crossovers: from batch 5
// the tensor cores win on every layer of at least 4 Mi weights; at batch 3
// and 4 on layers above 24 M (5120 x 5120 and larger; 4096 x 4096 and
// 1024 x 8192 stay on the row kernel); at batch 2 only on the largest split
// layers (8192 x 28672: 43 against 58 us; 8192 x 8192 is a tie, 28672 x
// 8192 slightly slower).  Tuning key tc forces it on (1) or off (0).
// The rule alone, for a product (or a group, p.rows its rows together) that
// the tensor-core product can run.
bool takes_tensor_cores_rule(const nm::SpmvProblem &p, uint32_t *lbo_enc)
{
    const int tc = nm::spmm_tc_mode(lbo_enc);
    const int nsm = nm::sm_count();
    if (tc == 0 || nsm <= 0) return false;
    if (tc == 1 || p.batch > NM_MAX_BATCH) return true;
    const int64_t weights = p.rows * p.K;
    const int64_t per_sm = (p.rows + nsm - 1) / nsm;
    if (p.batch >= 5) return weights >= (4ll << 20);
    if (p.batch >= 3) return weights > 24ll * 1000 * 1000;
    if (p.batch == 2) return weights >= (128ll << 20) && per_sm <= 128;
    return false;
}

bool takes_tensor_cores(const nm::SpmvProblem &p, uint32_t *lbo_enc)
{
    const int nsm = nm::sm_count();
    if (nsm <= 0 || !nm::spmm_tc_applies(p, nsm)) {
        nm::spmm_tc_mode(lbo_enc);
        return false;
    }
    return takes_tensor_cores_rule(p, lbo_enc);
}

nm_status run_product(const nm::SpmvProblem &p, cudaStream_t s)
{
    cudaError_t e = cudaErrorNotSupported;
    uint32_t tc_lbo = 0;
    if (takes_tensor_cores(p, &tc_lbo))
        e = nm::launch_spmm_tc(p, nm::spmm_tc_desc_hi(tc_lbo), s);
    if (e == cudaErrorNotSupported && p.batch > NM_MAX_BATCH)  // no other kernel takes it
        return fail(NM_ERR_UNSUPPORTED, "batch=%d: no tensor-core plan fits", p.batch);
    if (e == cudaErrorNotSupported && nm::bulk_path_applies(p.N, p.M, p.K)) {
        nm::SpmvGroup g;
        g.count = 1;
        g.p[0] = p;
        e = nm::launch_rows(g, s);
        if (e == cudaErrorNotSupported) e = nm::launch_bulk(p, s);
    }
    if (e == cudaErrorNotSupported)
        e = nm::fast_path_applies(p.N, p.M, p.K) ? nm::launch_fast(p, s) : nm::launch_generic(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "nm_spmv launch");
    return NM_OK;
}

}  // namespace

void nm::set_last_error(const char *msg)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

extern "C" {

int nm_version(void) { return NM_VERSION; }

const char *nm_last_error(void) { return g_last_error; }

const char *nm_status_str(nm_status status)
{
    switch (status) {
    case NM_OK: return "NM_OK";
    case NM_ERR_INVALID_ARG: return "NM_ERR_INVALID_ARG";
    case NM_ERR_UNSUPPORTED: return "NM_ERR_UNSUPPORTED";
    case NM_ERR_BAD_MASK: return "NM_ERR_BAD_MASK";
    case NM_ERR_CUDA: return "NM_ERR_CUDA";
    default: return "NM_ERR_UNKNOWN";
    }
}

nm_status nm_packed_sizes(int64_t rows, int64_t K, int N, int M, size_t *values_bytes,
                          size_t *mask_bytes)
{
    g_last_error[0] = 0;
    nm_status st = check_shape(rows, K, N, M);
    if (st != NM_OK) return st;
    // rows, K < 2^31, so every product below stays under 2^63.
    const int64_t vb = rows * ((K / M) * N) * 2;
    const int64_t mb = rows * ((K + 31) / 32) * 4;
    if (values_bytes) *values_bytes = static_cast<size_t>(vb);
    if (mask_bytes) *mask_bytes = static_cast<size_t>(mb);
    return NM_OK;
}

nm_status nm_pack(const void *W, const uint8_t *mask, int64_t rows, int64_t K, int N, int M,
                  void *values, uint32_t *masks, nm_stream_t stream)
{
    g_last_error[0] = 0;
    nm_status st = check_shape(rows, K, N, M);
    if (st != NM_OK) return st;
    if (rows == 0 || K == 0) return NM_OK;
    if (!W || !mask || !values || !masks)
        return fail(NM_ERR_INVALID_ARG, "W, mask, values and masks must be non-NULL");
    if (!aligned(W, 2)) return fail(NM_ERR_INVALID_ARG, "W must be 2-byte aligned");
    if (!aligned(values, 16) || !aligned(masks, 16))
        return fail(NM_ERR_INVALID_ARG, "values and masks must be 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "nm_pack: cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return fail(NM_ERR_INVALID_ARG, "nm_pack synchronises its stream and cannot be captured");

    unsigned int *d_bad = nullptr;
    e = cudaMallocAsync(reinterpret_cast<void **>(&d_bad), sizeof(unsigned int), s);
    if (e != cudaSuccess) return cuda_fail(e, "nm_pack: cudaMallocAsync");
    unsigned int h_bad = 0;
    e = cudaMemsetAsync(d_bad, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess)
        e = nm::launch_pack(static_cast<const uint16_t *>(W), mask, rows, K, N, M,
                            static_cast<uint16_t *>(values), masks, d_bad, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&h_bad, d_bad, sizeof(unsigned int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaError_t ef = cudaFreeAsync(d_bad, s);
    if (e != cudaSuccess) return cuda_fail(e, "nm_pack");
    if (ef != cudaSuccess) return cuda_fail(ef, "nm_pack: cudaFreeAsync");
    if (h_bad != 0)
        return fail(NM_ERR_BAD_MASK, "%u group(s) do not keep exactly N=%d of M=%d", h_bad, N, M);
    return NM_OK;
}

nm_status nm_unpack(const nm_matrix *A, void *W_out, nm_stream_t stream)
{
    g_last_error[0] = 0;
    nm_status st = check_matrix(A);
    if (st != NM_OK) return st;
    if (A->rows == 0 || A->K == 0) return NM_OK;
    if (!W_out) return fail(NM_ERR_INVALID_ARG, "W_out is NULL");
    if (!aligned(W_out, 2)) return fail(NM_ERR_INVALID_ARG, "W_out must be 2-byte aligned");
    cudaError_t e = nm::launch_unpack(static_cast<const uint16_t *>(A->values), A->masks, A->rows,
                                      A->K, A->N, A->M, static_cast<uint16_t *>(W_out),
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "nm_unpack launch");
    return NM_OK;
}

nm_status nm_spmv_batched(const nm_matrix *A, const void *x, int64_t ldx, void *y, int64_t ldy,
                          int batch, nm_dtype y_type, nm_stream_t stream)
{
    g_last_error[0] = 0;
    nm::SpmvProblem p;
    bool empty = false;
    nm_status st = prepare_product(A, x, ldx, y, ldy, batch, y_type, &p, &empty,
                                   reinterpret_cast<cudaStream_t>(stream));
    if (st != NM_OK || empty) return st;
    return run_product(p, reinterpret_cast<cudaStream_t>(stream));
}

nm_status nm_calib_accumulate(const void *X, int64_t T, int64_t K, int64_t ldx, float *H,
                              int64_t ldh, nm_stream_t stream)
{
    g_last_error[0] = 0;
    if (T < 0 || K < 0) return fail(NM_ERR_INVALID_ARG, "negative size T=%lld K=%lld",
                                    (long long)T, (long long)K);
    if (T == 0 || K == 0) return NM_OK;
    if (T > INT_MAX || K > (1 << 20))
        return fail(NM_ERR_INVALID_ARG, "size too large T=%lld K=%lld", (long long)T,
                    (long long)K);
    if (K % 8 != 0) return fail(NM_ERR_INVALID_ARG, "K=%lld must be a multiple of 8", (long long)K);
    if (ldx < K || ldx % 8 != 0)
        return fail(NM_ERR_INVALID_ARG, "ldx=%lld must be >= K and a multiple of 8", (long long)ldx);
    if (ldh < K || ldh % 4 != 0)
        return fail(NM_ERR_INVALID_ARG, "ldh=%lld must be >= K and a multiple of 4", (long long)ldh);
    if (!X || !H) return fail(NM_ERR_INVALID_ARG, "X and H must be non-NULL");
    if (!aligned(X, 16) || !aligned(H, 16))
        return fail(NM_ERR_INVALID_ARG, "X and H must be 16-byte aligned");
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e, "nm_calib_accumulate: device error word");
    e = nm::launch_calib(static_cast<const uint16_t *>(X), T, K, ldx, H, ldh, err,
                         nm::calib_idesc(), nm::calib_desc_hi(8192, 1024),
                         reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported)
        return fail(NM_ERR_UNSUPPORTED, "nm_calib_accumulate: no tensor-map encoder in the driver");
    if (e != cudaSuccess) return cuda_fail(e, "nm_calib_accumulate launch");
    return NM_OK;
}

nm_status nm_select_mask(const void *W, const float *col_scale, int64_t rows, int64_t K, int N,
                         int M, uint8_t *mask, nm_stream_t stream)
{
    g_last_error[0] = 0;
    nm_status st = check_shape(rows, K, N, M);
    if (st != NM_OK) return st;
    if (rows == 0 || K == 0) return NM_OK;
    if (!W || !mask) return fail(NM_ERR_INVALID_ARG, "W and mask must be non-NULL");
    if (!aligned(W, 16) || !aligned(mask, 16) || (col_scale && !aligned(col_scale, 16)))
        return fail(NM_ERR_INVALID_ARG, "W, mask and col_scale must be 16-byte aligned");
    const cudaError_t e = nm::launch_select(static_cast<const uint16_t *>(W), col_scale, rows, K,
                                            N, M, mask, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "nm_select_mask launch");
    return NM_OK;
}

nm_status nm_prune_pack(const void *W, const float *col_scale, int64_t rows, int64_t K, int N,
                        int M, void *values, uint32_t *masks, nm_stream_t stream)
{
    g_last_error[0] = 0;
    nm_status st = check_shape(rows, K, N, M);
    if (st != NM_OK) return st;
    if (rows == 0 || K == 0) return NM_OK;
    if (!W || !values || !masks)
        return fail(NM_ERR_INVALID_ARG, "W, values and masks must be non-NULL");
    if (!aligned(W, 16) || !aligned(values, 16) || !aligned(masks, 16) ||
        (col_scale && !aligned(col_scale, 16)))
        return fail(NM_ERR_INVALID_ARG, "W, values, masks and col_scale must be 16-byte aligned");
    const cudaError_t e = nm::launch_prune_pack(static_cast<const uint16_t *>(W), col_scale, rows,
                                                K, N, M, static_cast<uint16_t *>(values), masks,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "nm_prune_pack launch");
    return NM_OK;
}

nm_status nm_spmv_gate_up_silu(const nm_matrix *gate, const nm_matrix *up, const void *x,
                               int64_t ldx, void *h, int64_t ldh, int batch, nm_dtype h_type,
                               nm_stream_t stream)
{
    g_last_error[0] = 0;
    if (!gate || !up) return fail(NM_ERR_INVALID_ARG, "gate and up must be non-NULL");
    if (gate->rows != up->rows || gate->K != up->K || gate->N != up->N || gate->M != up->M)
        return fail(NM_ERR_INVALID_ARG, "gate and up must have the same rows, K, N and M");
    nm_status st = check_matrix(gate);
    if (st != NM_OK) return st;
    if (batch > NM_MAX_BATCH && batch <= NM_MAX_BATCH_TC)
        return fail(NM_ERR_UNSUPPORTED, "nm_spmv_gate_up_silu: batch=%d > %d", batch,
                    NM_MAX_BATCH);
    if (gate->rows > 0 && gate->K > 0 && !nm::bulk_path_applies(gate->N, gate->M, gate->K))
        return fail(NM_ERR_UNSUPPORTED,
                    "nm_spmv_gate_up_silu: K must be a multiple of 128 and N:M one of 1:4, "
                    "2:4, 4:4, 1:8, 2:8, 4:8, 8:8 (K=%lld, %d:%d)",
                    (long long)gate->K, gate->N, gate->M);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    nm::SpmvGroup g;
    g.count = 2;
    g.pair = true;
    bool empty_gate = false, empty_up = false;
    st = prepare_product(gate, x, ldx, h, ldh, batch, h_type, &g.p[0], &empty_gate, s);
    if (st != NM_OK) {
        char msg[512];
        snprintf(msg, sizeof(msg), "gate: %s", g_last_error);
        return fail(st, "%s", msg);
    }
    st = prepare_product(up, x, ldx, h, ldh, batch, h_type, &g.p[1], &empty_up, s);
    if (st != NM_OK) {
        char msg[512];
        snprintf(msg, sizeof(msg), "up: %s", g_last_error);
        return fail(st, "%s", msg);
    }
    if (empty_gate) return NM_OK;  // rows == 0, or K == 0 and h zeroed (silu(0) * 0 = 0)
    const cudaError_t e = nm::launch_rows(g, s);
    if (e == cudaErrorNotSupported)
        return fail(NM_ERR_UNSUPPORTED, "nm_spmv_gate_up_silu: no kernel plan fits K=%lld",
                    (long long)gate->K);
    if (e != cudaSuccess) return cuda_fail(e, "nm_spmv_gate_up_silu launch");
    return NM_OK;
}

nm_status nm_spmv_group(const nm_matrix *A, int count, const void *const *x, int64_t ldx,
                        void *const *y, const int64_t *ldy, int batch, nm_dtype y_type,
                        nm_stream_t stream)
{
    g_last_error[0] = 0;
    if (count < 0 || count > NM_MAX_GROUP)
        return fail(NM_ERR_INVALID_ARG, "count=%d outside [0, %d]", count, NM_MAX_GROUP);
    if (count == 0) return NM_OK;
    if (!A || !x || !y) return fail(NM_ERR_INVALID_ARG, "A, x and y must be non-NULL arrays");
    for (int i = 1; i < count; ++i)
        if (A[i].N != A[0].N || A[i].M != A[0].M || A[i].K != A[0].K)
            return fail(NM_ERR_INVALID_ARG, "matrix %d: N, M and K must equal those of matrix 0", i);
    nm::SpmvGroup g;
    g.count = 0;
    bool fusable = true;
    for (int i = 0; i < count; ++i) {
        bool empty = false;
        nm_status st = prepare_product(&A[i], x[i], ldx, y[i], ldy ? ldy[i] : A[i].rows, batch,
                                       y_type, &g.p[g.count], &empty,
                                       reinterpret_cast<cudaStream_t>(stream));
        if (st != NM_OK) {
            char msg[512];
            snprintf(msg, sizeof(msg), "matrix %d: %s", i, g_last_error);
            return fail(st, "%s", msg);
        }
        if (empty) {  // rows == 0 (nothing) or K == 0 (y zeroed already)
            fusable = false;
            continue;
        }
        ++g.count;
    }
    // A group that the tensor-core product can run as a whole (every member
    // 2:4 within its limits, and the rule of takes_tensor_cores met by the
    // group's rows together) runs in one launch of it: the 70B-shaped q/k/v
    // (8192 + 1024 + 1024 rows, K = 8192) takes 24.3 us at batch 3-8 there,
    // against 25.6 / 29.2 us for one fused CUDA-core launch at batch 3 / 4
    // and 33.4 us for three tensor-core launches at batch 8.  Failing that
    // (no grouped plan fits: e.g. two 28672-row members), members that all
    // take the tensor-core product alone run one launch each, and other
    // groups one fused CUDA-core launch.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorNotSupported;
    uint32_t lbo = 0;
    if (g.count > 1) {
        nm::SpmvProblem whole = g.p[0];
        whole.rows = 0;
        const int nsm = nm::sm_count();
        bool runs = nsm > 0;
        for (int i = 0; i < g.count && runs; ++i) {
            whole.rows += g.p[i].rows;
            runs = nm::spmm_tc_applies(g.p[i], nsm);
        }
        if (runs && takes_tensor_cores_rule(whole, &lbo)) {
            e = nm::launch_spmm_tc_group(g, nm::spmm_tc_desc_hi(lbo), s);
            if (e == cudaSuccess) return NM_OK;
            if (e != cudaErrorNotSupported) return cuda_fail(e, "nm_spmv_group launch");
        }
    }
    bool all_tc = g.count > 0;
    for (int i = 0; i < g.count && all_tc; ++i) all_tc = takes_tensor_cores(g.p[i], &lbo);
    if (fusable && !all_tc && g.count > 1 &&
        nm::bulk_path_applies(g.p[0].N, g.p[0].M, g.p[0].K))
        e = nm::launch_rows(g, s);
    if (e == cudaSuccess) return NM_OK;
    if (e != cudaErrorNotSupported) return cuda_fail(e, "nm_spmv_group launch");
    for (int i = 0; i < g.count; ++i) {  // one launch per matrix
        nm_status st = run_product(g.p[i], s);
        if (st != NM_OK) return st;
    }
    return NM_OK;
}

nm_status nm_device_errors(uint32_t *flags, int clear, nm_stream_t stream)
{
    g_last_error[0] = 0;
    if (!flags) return fail(NM_ERR_INVALID_ARG, "flags is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "nm_device_errors: cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return fail(NM_ERR_INVALID_ARG, "nm_device_errors synchronises and cannot be captured");
    unsigned int *d = nullptr;
    e = device_error_word(&d);
    if (e != cudaSuccess) return cuda_fail(e, "nm_device_errors: device error word");
    unsigned int h = 0;
    e = cudaMemcpyAsync(&h, d, sizeof(h), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(d, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "nm_device_errors");
    *flags = h;
    return NM_OK;
}

nm_status nm_spmv(const nm_matrix *A, const void *x, void *y, nm_dtype y_type, nm_stream_t stream)
{
    if (!A) {
        g_last_error[0] = 0;
        return fail(NM_ERR_INVALID_ARG, "matrix descriptor is NULL");
    }
    return nm_spmv_batched(A, x, A->K, y, A->rows, 1, y_type, stream);
}

}  // extern "C"
