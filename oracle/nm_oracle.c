/*
 * nm_oracle.c -- plain, slow, obviously correct CPU oracle for the N:M
 * sparse matrix-vector product of SparseDecoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include,
 * link or call this file; only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no header, helper,
 * table or constant with the CUDA path.
 *
 * What the method computes (sources, by page title and section):
 *   - "SparseDecoding: Decoding-Aware Pruning for Accurate and Efficient LLM
 *     Inference", Abstract: decoding is dominated by sparse matrix-vector
 *     (SpMV) products; the system contribution is an N:M sparse
 *     matrix-vector kernel with bitmask indexing and fixed-step traversal.
 *   - "SparseDecoding Makes LLM Pruning Aware of Generation", Key points:
 *     the same kernel, "bitmask indexing and fixed-step traversal".
 *   - bedrocknews, arXiv 2610.12327v1 (one-paragraph summary): N:M
 *     structured sparsity means a fixed ratio of zeros inside small blocks;
 *     the product is a sparse matrix times a single vector.
 *   - "SparseDecoding: Why Pruning Should Account for How LLMs Generate",
 *     section 6: how the pruned model is represented is left open.
 *
 * Readings taken where the pages are silent (each one is listed with its
 * reason in the design notes of the repository):
 *   - group = M consecutive weights along the input dimension K; a valid
 *     group keeps exactly N of them;
 *   - the bitmask is one bit per weight position: bit b of 32-bit word w of a
 *     row is position k = 32*w + b (least significant bit = lowest k); words
 *     per row = ceil(K/32); unused bits are zero;
 *   - the kept values of group g are stored at values[row][g*N + j],
 *     j = 0..N-1, in increasing k ("fixed step": every group advances the
 *     value pointer by exactly N, so no per-row offsets exist);
 *   - the mask, not the value, decides what is kept: a kept zero is stored,
 *     a dropped nonzero is not;
 *   - a group whose mask does not hold exactly N ones is invalid; the pack
 *     counts such groups (the first min(count, N) kept values are stored,
 *     missing slots are written as +0.0);
 *   - y = (W with dropped positions zeroed) . x, accumulated in fp64 here.
 *
 * fp16 values are handled as raw IEEE 754 binary16 bit patterns (uint16_t);
 * they are decoded to double by oracle_half_to_double below, written from the
 * binary16 definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction
 * bits; exponent 0 is zero/subnormal, exponent 31 is inf/NaN).
 *
 * Parity pins: every function here is pinned by the CPU tests against
 * numpy (binary16 conversion, boolean-mask gathers, dense fp64 matmul),
 * hand-worked examples stored under tests/golden/, closed forms (all-ones
 * and one-hot x, small integers) and invariants (pack then unpack, exactly
 * N per group, linearity).  No function here is "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* binary16 -> double, from the IEEE 754 definition. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);              /* zero or subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = (f != 0) ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x400), e - 25); /* (1024 + f) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

/* Number of values per row in the packed layout (K must be a multiple of M). */
int64_t oracle_values_per_row(int64_t K, int N, int M)
{
    return (K / M) * N;
}

/* Number of 32-bit mask words per row. */
int64_t oracle_mask_words_per_row(int64_t K)
{
    return (K + 31) / 32;
}

/*
 * Pack a dense fp16 matrix W[rows][K] and its keep-mask mask[rows][K]
 * (nonzero byte = keep) into values[rows][K/M*N] and masks[rows][ceil(K/32)].
 * Returns the number of groups whose mask does not hold exactly N ones.
 */
int64_t oracle_pack(int64_t rows, int64_t K, int N, int M,
                    const uint16_t *W, const uint8_t *mask,
                    uint16_t *values, uint32_t *masks)
{
    int64_t Lv = oracle_values_per_row(K, N, M);
    int64_t Wm = oracle_mask_words_per_row(K);
    int64_t groups = K / M;
    int64_t bad = 0;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t w = 0; w < Wm; ++w)
            masks[r * Wm + w] = 0u;
        for (int64_t g = 0; g < groups; ++g) {
            int kept = 0;
            for (int q = 0; q < M; ++q) {
                int64_t k = g * M + q;
                if (mask[r * K + k] != 0) {
                    masks[r * Wm + k / 32] |= (uint32_t)1u << (k % 32);
                    if (kept < N)
                        values[r * Lv + g * N + kept] = W[r * K + k];
                    ++kept;
                }
            }
            for (int j = kept; j < N; ++j)
                values[r * Lv + g * N + j] = 0; /* +0.0 in missing slots */
            if (kept != N)
                ++bad;
        }
    }
    return bad;
}

/* Is bit k of row r of the packed mask set? */
static int mask_bit(const uint32_t *masks, int64_t Wm, int64_t r, int64_t k)
{
    return (int)((masks[r * Wm + k / 32] >> (k % 32)) & 1u);
}

/*
 * Inverse of oracle_pack for a valid layout: W_out[rows][K] receives the kept
 * values at their positions and +0.0 (bits 0x0000) at every dropped position.
 * Within a group the j-th set bit (in increasing k) takes value j; at most N
 * values are read per group (fixed step).
 */
void oracle_unpack(int64_t rows, int64_t K, int N, int M,
                   const uint16_t *values, const uint32_t *masks,
                   uint16_t *W_out)
{
    int64_t Lv = oracle_values_per_row(K, N, M);
    int64_t Wm = oracle_mask_words_per_row(K);
    int64_t groups = K / M;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            int j = 0;
            for (int q = 0; q < M; ++q) {
                int64_t k = g * M + q;
                if (mask_bit(masks, Wm, r, k) && j < N) {
                    W_out[r * K + k] = values[r * Lv + g * N + j];
                    ++j;
                } else {
                    W_out[r * K + k] = 0;
                }
            }
        }
    }
}

/*
 * The plain definition of the product, from the dense inputs:
 *   y[b][i] = sum over k with mask[i][k] != 0 of W[i][k] * x[b][k]
 *   s[b][i] = sum over the same k of |W[i][k] * x[b][k]|
 * in fp64, for rows i in [row_begin, row_end) and b in [0, batch).
 * x is fp16 [batch][ldx]; y and s are double [batch][ldy] (s may be NULL).
 */
void oracle_spmv_dense_f64(int64_t rows, int64_t K,
                           const uint16_t *W, const uint8_t *mask,
                           int batch, const uint16_t *x, int64_t ldx,
                           double *y, double *s, int64_t ldy,
                           int64_t row_begin, int64_t row_end)
{
    (void)rows;
    for (int b = 0; b < batch; ++b) {
        for (int64_t i = row_begin; i < row_end; ++i) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                if (mask[i * K + k] != 0) {
                    double p = oracle_half_to_double(W[i * K + k]) *
                               oracle_half_to_double(x[(int64_t)b * ldx + k]);
                    acc += p;
                    sabs += fabs(p);
                }
            }
            y[(int64_t)b * ldy + i] = acc;
            if (s)
                s[(int64_t)b * ldy + i] = sabs;
        }
    }
}

/*
 * The same product computed the way the method reads its operand: from the
 * packed layout, walking each row group by group, decoding the group's bits
 * from the bitmask and advancing the value index by exactly N per group
 * (bitmask indexing with fixed-step traversal).  Same argument conventions as
 * oracle_spmv_dense_f64; the k order of the sum is the same, so for a valid
 * layout the two give identical results.
 */
void oracle_spmv_packed_f64(int64_t rows, int64_t K, int N, int M,
                            const uint16_t *values, const uint32_t *masks,
                            int batch, const uint16_t *x, int64_t ldx,
                            double *y, double *s, int64_t ldy,
                            int64_t row_begin, int64_t row_end)
{
    (void)rows;
    int64_t Lv = oracle_values_per_row(K, N, M);
    int64_t Wm = oracle_mask_words_per_row(K);
    int64_t groups = K / M;
    for (int b = 0; b < batch; ++b) {
        for (int64_t i = row_begin; i < row_end; ++i) {
            double acc = 0.0, sabs = 0.0;
            int64_t vbase = i * Lv; /* value pointer of the row */
            for (int64_t g = 0; g < groups; ++g) {
                int j = 0;
                for (int q = 0; q < M; ++q) {
                    int64_t k = g * M + q;
                    if (mask_bit(masks, Wm, i, k) && j < N) {
                        double p = oracle_half_to_double(values[vbase + j]) *
                                   oracle_half_to_double(x[(int64_t)b * ldx + k]);
                        acc += p;
                        sabs += fabs(p);
                        ++j;
                    }
                }
                vbase += N; /* fixed step: every group advances by N */
            }
            y[(int64_t)b * ldy + i] = acc;
            if (s)
                s[(int64_t)b * ldy + i] = sabs;
        }
    }
}

/*
 * Magnitude-pruning mask: in every group of M along K keep the N positions of
 * largest |w|; ties go to the lower k (so |-0| = |+0| ties resolve by k).
 * Used by tests to check the synthetic input generator's mask rule; the
 * generator itself lives outside this directory.
 * Position q of a group is kept iff fewer than N positions of the group beat
 * it, where q' beats q when |w_q'| > |w_q|, or |w_q'| == |w_q| and q' < q.
 */
void oracle_topn_mask(int64_t rows, int64_t K, int N, int M,
                      const uint16_t *W, uint8_t *mask)
{
    int64_t groups = K / M;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            for (int q = 0; q < M; ++q) {
                double aq = fabs(oracle_half_to_double(W[r * K + g * M + q]));
                int beaten = 0;
                for (int q2 = 0; q2 < M; ++q2) {
                    if (q2 == q)
                        continue;
                    double a2 = fabs(oracle_half_to_double(W[r * K + g * M + q2]));
                    if (a2 > aq || (a2 == aq && q2 < q))
                        ++beaten;
                }
                mask[r * K + g * M + q] = (uint8_t)(beaten < N ? 1 : 0);
            }
        }
    }
}

/*
 * Score-driven N:M keep-mask: the selection step before packing.  The score
 * of weight (r, k) is |w| in single precision (exact for fp16) and, when
 * scale is given, |w| * scale[k] rounded to single precision; scale is a
 * per-input-channel importance (the activation-weighted magnitude of the
 * Wanda family of pruning methods, the baseline named by the bedrocknews
 * summary of arXiv 2610.12327v1).  Position q of a group is kept iff fewer
 * than N positions beat it, q' beating q when s(q') > s(q), or
 * s(q') == s(q) and q' < q.  With scale NULL this is oracle_topn_mask.
 */
void oracle_select_mask(int64_t rows, int64_t K, int N, int M, const uint16_t *W,
                        const float *scale, uint8_t *mask)
{
    int64_t groups = K / M;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            float sc[8];
            for (int q = 0; q < M; ++q) {
                int64_t k = g * M + q;
                float a = (float)fabs(oracle_half_to_double(W[r * K + k]));
                if (scale) {
                    volatile float prod = a * scale[k]; /* one rounding to single */
                    a = prod;
                }
                sc[q] = a;
            }
            for (int q = 0; q < M; ++q) {
                int beaten = 0;
                for (int q2 = 0; q2 < M; ++q2) {
                    if (q2 == q)
                        continue;
                    if (sc[q2] > sc[q] || (sc[q2] == sc[q] && q2 < q))
                        ++beaten;
                }
                mask[r * K + g * M + q] = (uint8_t)(beaten < N ? 1 : 0);
            }
        }
    }
}

/*
 * Decode-only calibration accumulation, the layer statistic SparseDecoding
 * collects while the dense model generates ("SparseDecoding: Decoding-Aware
 * Pruning for Accurate and Efficient LLM Inference", Abstract):
 * H[i][j] += sum_t x_t[i] x_t[j] over the T token rows of X (fp16 [T][ldx]),
 * in fp64; S[i][j] (if given) receives sum_t |x_t[i] x_t[j]| for the
 * tolerance.  H and S are [K][K].
 */
void oracle_calib_f64(int64_t T, int64_t K, const uint16_t *X, int64_t ldx, double *H, double *S)
{
    for (int64_t i = 0; i < K; ++i) {
        for (int64_t j = 0; j < K; ++j) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                double p = oracle_half_to_double(X[t * ldx + i]) *
                           oracle_half_to_double(X[t * ldx + j]);
                acc += p;
                sabs += fabs(p);
            }
            H[i * K + j] += acc;
            if (S)
                S[i * K + j] = sabs;
        }
    }
}
