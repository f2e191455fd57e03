// Internal interface between the C entry points (nm_api.cu) and the kernel
// launchers.  Not installed; the public interface is include/nm.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "nm.h"

namespace nm {

// One product y[b] = A x[b] for b < batch, arguments already validated.
struct SpmvProblem {
    int64_t rows;
    int64_t K;
    int N;
    int M;
    const void *values;
    const uint32_t *masks;
    const void *x;
    int64_t ldx;
    void *y;
    int64_t ldy;
    int batch;
    bool y_f32;
    unsigned int *err;  // device error word (see nm_device_errors)
};

// Independent products fused into one launch: same N, M, K, batch, ldx and
// y type; rows, pointers and ldy per problem.
struct SpmvGroup {
    int count;
    SpmvProblem p[NM_MAX_GROUP];
    // Gate/up pair (count == 2, same shape): one output per row,
    // p[0].y = silu(p[0] x) * (p[1] x); p[1].y is unused.
    bool pair = false;
};

// Vectorised kernel: 8 % N == 0 and K a multiple of the k-span of one
// 16-byte value chunk (8*M/N positions), and at most kMaxFastChunks chunks
// per K tile sweep (any K is handled by tiling K inside a block).
bool fast_path_applies(int N, int M, int64_t K);
cudaError_t launch_fast(const SpmvProblem &p, cudaStream_t s);

// Bulk-staged kernels (the main path): a fast pattern and K a multiple of
// 128, so that every row's value and mask segments are 16-byte multiples.
// launch_rows (row-per-warp, batch <= 2) is tried first, then launch_bulk
// (chunk columns per thread, any batch).  Both return cudaErrorNotSupported,
// having launched nothing, if no tiling fits in shared memory.
bool bulk_path_applies(int N, int M, int64_t K);
cudaError_t launch_rows(const SpmvGroup &g, cudaStream_t s);  // batch <= 2
cudaError_t launch_bulk(const SpmvProblem &p, cudaStream_t s);

// Scalar kernel for every valid pattern and K (patterns like 3:4, or K not
// a multiple of the chunk span).
cudaError_t launch_generic(const SpmvProblem &p, cudaStream_t s);

// Pack / unpack kernels.  `bad` counts groups whose mask is not exactly N.
cudaError_t launch_pack(const uint16_t *W, const uint8_t *mask, int64_t rows, int64_t K,
                        int N, int M, uint16_t *values, uint32_t *masks,
                        unsigned int *bad, cudaStream_t s);
cudaError_t launch_unpack(const uint16_t *values, const uint32_t *masks, int64_t rows,
                          int64_t K, int N, int M, uint16_t *W, cudaStream_t s);

// N:M selection from scores |w| (scale null) or |w| * scale[k]: the keep-mask
// (u8 [rows][K]), or the packed layout directly (nm_select.cu).  W, scale,
// mask, values and masks 16-byte aligned; K % M == 0.
cudaError_t launch_select(const uint16_t *W, const float *scale, int64_t rows, int64_t K, int N,
                          int M, uint8_t *mask, cudaStream_t s);
cudaError_t launch_prune_pack(const uint16_t *W, const float *scale, int64_t rows, int64_t K,
                              int N, int M, uint16_t *values, uint32_t *masks, cudaStream_t s);

// H[i][j] += sum_t X[t][i] X[t][j] on the tensor cores (nm_calib.cu); X fp16
// [T][ldx] with K % 8 == 0, H fp32 [K][ldh] with ldh % 4 == 0, both 16-byte
// aligned.  idesc / desc_hi: the MMA instruction descriptor and the operands'
// shared-memory descriptor fields (calib_idesc(), calib_desc_hi(8192, 1024)).
cudaError_t launch_calib(const uint16_t *X, int64_t T, int64_t K, int64_t ldx, float *H,
                         int64_t ldh, unsigned int *err, uint32_t idesc, uint64_t desc_hi,
                         cudaStream_t s);
uint32_t calib_idesc();
uint64_t calib_desc_hi(uint32_t lbo, uint32_t sbo);

// 2:4 product for batches of 8 to 32 on the tensor cores (nm_spmm_tc.cu):
// applies to K % 128 == 0, ldx % 8 == 0, 16-byte aligned values, masks and
// x, and at most 256 rows per CTA with one CTA per SM.  desc_hi: the
// operands' shared-memory descriptor fields (spmm_tc_desc_hi(1)).
bool spmm_tc_applies(const SpmvProblem &p, int nsm);
cudaError_t launch_spmm_tc(const SpmvProblem &p, uint64_t desc_hi, cudaStream_t s);
// The products of a group (same K, batch, x stride and y type; each as
// spmm_tc_applies allows) in one launch of the sparse-operand product;
// cudaErrorNotSupported when that kernel is not the one selected (tc_sp=0,
// sp_group=0) or no plan fits: the caller then launches them one by one.
cudaError_t launch_spmm_tc_group(const SpmvGroup &g, uint64_t desc_hi, cudaStream_t s);
uint32_t spmm_tc_idesc(int N);
// When products take that path (tuning key tc: 1 wherever it applies, 0
// never, -1 by batch and layer size: takes_tensor_cores in nm_api.cu) and
// its descriptors' encoded leading-byte-offset field (tuning key tc_lbo).
int spmm_tc_mode(uint32_t *lbo_enc);
uint64_t spmm_tc_desc_hi(uint32_t lbo_enc);

// Cached device attributes of the current device.
int sm_count();
int max_dynamic_smem();

// Set the calling thread's message returned by nm_last_error().
void set_last_error(const char *msg);

}  // namespace nm
