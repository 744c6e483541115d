/*
 * qkv.h -- C ABI of the RMSNorm + 4-bit Q/K/V projection of the GB300
 * (sm_103a) library.  Same library, conventions and status codes as qmoe.h
 * (device pointers owned by the caller, dense row-major layouts, a caller
 * workspace, asynchronous work on the caller's stream, host-side validation
 * before any launch, device conditions in the workspace error word).
 *
 * Operation: the com.microsoft.MatMulNBitsQkv WebGPU kernel manifest (v1),
 * keys inputs, outputs, attributes, attributeConstraints, typeConstraints,
 * derive.* and the variants' passes (MatMulNBitsQkv.RmsNorm followed by
 * MatMulNBitsQkv.Projection).  Per row r of A (rows = product of the leading
 * dimensions):
 *   x        = A[r] (+ skip[r])
 *   residual = x                                   (optional output; needs skip)
 *   normed   = x / sqrt(mean(x^2) + epsilon) * norm_scale
 *   Q[r, n]  = sum_k normed[k] * (code(q_B, n, k) - 8) * q_scales[n, k / 32]
 *   K[r, n], V[r, n] likewise with k_B / k_scales and v_B / v_scales.
 * Packed weights are [N, kBlocks, 16] bytes, kBlocks = ceil(K / 32): code j
 * of block b of row n is in byte j / 2 of blob (n, b), low nibble first; the
 * zero point is 8 (derive.defaultZero).  Codes past K are padding.
 * Arithmetic: fp32 normalisation; the projections run on the tensor cores
 * with fp16 activations and exact integer weights, fp32 block scaling and
 * accumulation (DECODE path), or in fp32 (GENERIC path); outputs in T1.
 */
#ifndef QKV_H
#define QKV_H

#include <stddef.h>
#include <stdint.h>

#include "qmoe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Kernel path.  AUTO picks by shape.
 *   DECODE  : up to 16 rows, K a multiple of 128 (256 with fp16 scales), 16-byte
 *             aligned tensors: one weight-streaming GEMV launch over the three
 *             projections, started while the normalisation kernel runs
 *   GENERIC : scalar fp32 kernels for any valid shape                          */
typedef enum { QKV_PATH_AUTO = 0, QKV_PATH_DECODE = 1, QKV_PATH_GENERIC = 3 } qkv_path;

/*
 * Attributes of the manifest (attributes, attributeConstraints).
 * qkv_attrs_default sets the defaults: bits 4, accuracy_level 0, epsilon
 * 9.999999974752427e-7, path AUTO, and K = Nq = Nkv = block_size = 0, which
 * are required and must be set by the caller.
 */
typedef struct {
    int64_t K;                  /* reduction length, > 0                     */
    int64_t Nq;                 /* rows of q_B, > 0                          */
    int64_t Nkv;                /* rows of k_B and v_B, > 0                  */
    int64_t block_size;         /* must be 32                                */
    int32_t bits;               /* must be 4                                 */
    int32_t accuracy_level;     /* must be 0                                 */
    float epsilon;
    int32_t path;               /* qkv_path                                  */
} qkv_attrs;

void qkv_attrs_default(qkv_attrs *attrs);

/* Workspace bytes matmul_nbits_qkv needs for A's shape, the attributes and T1
 * (QMOE_DT_F32 or QMOE_DT_F16). */
qmoe_status qkv_workspace_size(const int64_t *a_shape, int32_t a_rank, const qkv_attrs *attrs,
                               int32_t dtype, size_t *bytes);

/* The kernel path matmul_nbits_qkv takes for these shapes (never AUTO). */
qmoe_status qkv_choose_path(const int64_t *a_shape, int32_t a_rank, const qkv_attrs *attrs,
                            int32_t dtype, int32_t *path);

/*
 * The operator (manifest inputs aT, skipT, normScaleT, qBT, qScalesT, kBT,
 * kScalesT, vBT, vScalesT; outputs qT, kT, vT, residualT).
 *   A           T1 [rows, K] or [B, S, K]            (a_rank 2 or 3)
 *   skip        T1, the shape of A, or NULL
 *   norm_scale  T1 [K]
 *   q_B         uint8 [Nq, kBlocks, 16]              (q_B_shape[3])
 *   q_scales    T1 [Nq, kBlocks]                     (q_scales_shape[2])
 *   k_B, v_B    uint8 [Nkv, kBlocks, 16]; k_scales, v_scales T1 [Nkv, kBlocks]
 *   Q           T1, A's shape with the last dim Nq
 *   Kout, V     T1, A's shape with the last dim Nkv
 *   residual    T1, the shape of A, or NULL (only with skip)
 * dtype is T1: QMOE_DT_F32 or QMOE_DT_F16.  rows == 0 is a no-op.
 * Errors: INVALID_ARGUMENT for a failed manifest predicate (weightShapeOk,
 * scaleShapeOk, ioShapeOk, normContractOk, required attributes, NULL
 * pointers, residual without skip); NOT_SUPPORTED for bits other than 4,
 * block_size other than 32, accuracy_level other than 0, a T1 other than
 * float32/float16, or a forced path the shape cannot take;
 * WORKSPACE_TOO_SMALL; CUDA for a failed launch.
 */
qmoe_status matmul_nbits_qkv(const void *A, const int64_t *a_shape, int32_t a_rank,
                             const void *skip, const void *norm_scale,
                             const uint8_t *q_B, const int64_t *q_B_shape, const void *q_scales,
                             const int64_t *q_scales_shape,
                             const uint8_t *k_B, const int64_t *k_B_shape, const void *k_scales,
                             const int64_t *k_scales_shape,
                             const uint8_t *v_B, const int64_t *v_B_shape, const void *v_scales,
                             const int64_t *v_scales_shape,
                             void *Q, void *Kout, void *V, void *residual, int32_t dtype,
                             const qkv_attrs *attrs, void *workspace, size_t workspace_bytes,
                             void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* QKV_H */
