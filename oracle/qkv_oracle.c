/*
 * Reference oracle for the RMSNorm + 4-bit Q/K/V projection operator.
 *
 * TEST INFRASTRUCTURE ONLY.  A plain, slow, scalar CPU restatement in double
 * precision.  Only the test-suite, the package smoke check and the
 * CPU-baseline leg of the bench may load it.  It shares no code, header, table
 * or helper with the CUDA library, nor with the other oracle files.
 *
 * Source (web page, cited by title and section):
 *   [QKV] com.microsoft.MatMulNBitsQkv WebGPU kernel manifest (v1): inputs,
 *         outputs, attributes, attributeConstraints, typeConstraints,
 *         derive.* (codesPerByte, codeMask, defaultZero, weightShapeOk,
 *         scaleShapeOk, normContractOk, epsilonValue) and the variants'
 *         passes (MatMulNBitsQkv.RmsNorm, then MatMulNBitsQkv.Projection*).
 *
 * Per row r of the input (rows = product of the leading dimensions of A):
 *   x        = A[r] (+ skip[r] when skip is present)
 *   residual = x                 (the optional input_skip_bias_sum output)
 *   normed   = x / sqrt(mean_k x[k]^2 + epsilon) * norm_scale
 *   Q[r, n]  = sum_k normed[k] * (code_q(n, k) - 8) * q_scales[n, k / block_size]
 *   and K, V likewise with k_B/k_scales and v_B/v_scales (Nkv rows each).
 * Packed weights are [N, kBlocks, blobSize] bytes with kBlocks = ceil(K /
 * block_size) and blobSize = block_size * bits / 8: code j of block b of row n
 * sits in byte j / 2 of blob (n, b), the low nibble holding the even j.
 *
 * Readings taken where the page leaves a step open (each is listed in the
 * design notes of the repository):
 *   - RMSNorm is x * rsqrt(mean(x^2) + epsilon) * norm_scale (the pass name
 *     and the epsilon and norm_scale inputs; no bias, no mean subtraction);
 *   - the zero point is derive.defaultZero = 8 for every block;
 *   - codes of the last block past K (when block_size does not divide K) are
 *     padding and take no part;
 *   - the low nibble of a byte holds the even element (codeMask applied from
 *     bit 0, as in the QMoE manifest's packing).
 *
 * All arithmetic is IEEE double.  Inputs given as double are the caller's
 * float or half values widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define QKV_ORACLE_OK 0
#define QKV_ORACLE_BAD_ARG (-2)
#define QKV_ORACLE_NO_MEMORY (-3)

/* [QKV] derive.codesPerByte = 2, codeMask = 15 for 4-bit codes. */
int oracle_qkv_code(const uint8_t *packed, int64_t n, int64_t k, int64_t kblocks,
                    int64_t block_size)
{
    const int64_t blob = block_size / 2;
    const int64_t b = k / block_size, j = k % block_size;
    const uint8_t byte = packed[(n * kblocks + b) * blob + j / 2];
    return (j % 2 == 0) ? (byte & 15) : (byte >> 4);
}

/* One projection: out[n] = sum_k normed[k] * (code - 8) * scale[n, k / bs]. */
static void project(const double *normed, int64_t K, const uint8_t *B, const double *scales,
                    int64_t N, int64_t block_size, double *out)
{
    const int64_t kblocks = (K + block_size - 1) / block_size;
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const int q = oracle_qkv_code(B, n, k, kblocks, block_size);
            acc += normed[k] * (double)(q - 8) * scales[n * kblocks + k / block_size];
        }
        out[n] = acc;
    }
}

/*
 * The operator for `rows` rows.  A and skip [rows, K] (skip may be NULL),
 * norm_scale [K]; q_B [Nq, kBlocks, blob], q_scales [Nq, kBlocks]; k_B, v_B
 * [Nkv, kBlocks, blob], k_scales, v_scales [Nkv, kBlocks].  Outputs Q
 * [rows, Nq], Kout and V [rows, Nkv]; residual [rows, K] or NULL (needs skip);
 * normed_out [rows, K] or NULL receives the normalised rows.
 */
int oracle_qkv(const double *A, const double *skip, const double *norm_scale, int64_t rows,
               int64_t K, const uint8_t *qB, const double *qS, int64_t Nq, const uint8_t *kB,
               const double *kS, const uint8_t *vB, const double *vS, int64_t Nkv,
               int64_t block_size, double epsilon, double *Q, double *Kout, double *V,
               double *residual, double *normed_out)
{
    if (K <= 0 || Nq <= 0 || Nkv <= 0 || block_size <= 0 || block_size % 2 != 0)
        return QKV_ORACLE_BAD_ARG;
    if (residual && !skip)
        return QKV_ORACLE_BAD_ARG;
    double *x = (double *)malloc((size_t)K * sizeof(double));
    double *normed = (double *)malloc((size_t)K * sizeof(double));
    if (!x || !normed) {
        free(x);
        free(normed);
        return QKV_ORACLE_NO_MEMORY;
    }
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            x[k] = A[r * K + k] + (skip ? skip[r * K + k] : 0.0);
            ss += x[k] * x[k];
        }
        if (residual)
            for (int64_t k = 0; k < K; ++k)
                residual[r * K + k] = x[k];
        const double inv = 1.0 / sqrt(ss / (double)K + epsilon);
        for (int64_t k = 0; k < K; ++k)
            normed[k] = x[k] * inv * norm_scale[k];
        if (normed_out)
            for (int64_t k = 0; k < K; ++k)
                normed_out[r * K + k] = normed[k];
        project(normed, K, qB, qS, Nq, block_size, Q + r * Nq);
        project(normed, K, kB, kS, Nkv, block_size, Kout + r * Nkv);
        project(normed, K, vB, vS, Nkv, block_size, V + r * Nkv);
    }
    free(x);
    free(normed);
    return QKV_ORACLE_OK;
}
