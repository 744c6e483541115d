/*
 * moe.h -- C ABI of the float (unquantized) mixture-of-experts layer of the
 * GB300 (sm_103a) library.  Same library, conventions and status codes as
 * qmoe.h (device pointers owned by the caller, dense row-major layouts, a
 * caller workspace, asynchronous work on the caller's stream, host-side
 * validation before any launch, device conditions in the workspace error
 * word read with moe_get_device_error).
 *
 * Operation: the com.microsoft.MoE kernel README (v1), sections Description,
 * Inputs, Outputs, Attributes, Type constraints.  Per token t:
 *   p       = softmax over all E router logits of t;
 *   sel     = the k experts of largest p (descending; equal values to the
 *             lower expert index);
 *   w_i     = p[sel_i], divided by sum_i p[sel_i] when
 *             normalize_routing_weights = 1;
 *   h1      = x_t . W1[e]^T + b1[e]          W1 [E, fusion*I, H]
 *   h3      = x_t . W3[e]^T + b3[e]          W3 [E, I, H] (when consumed)
 *   a       = relu(h1) | gelu(h1) = h1*Phi(h1) | silu(h1) = h1*sigmoid(h1)
 *             (times h3 when FC3 is given) | identity(h1) |
 *             swiglu: a = g*sigmoid(alpha*g)*(u + beta) with (g, u) =
 *             (h1, h3) for swiglu_fusion 0, (h1[2j], h1[2j+1]) for 1,
 *             (h1[j], h1[I+j]) for 2; swiglu_limit clamps g from above and
 *             u on both sides;
 *   o       = a . W2[e]^T + b2[e]            W2 [E, H, I]
 *   y_t     = sum_i w_i * o_i.
 * Arithmetic: every contraction runs on the tensor cores in TF32 (operands
 * with a 10-bit mantissa, fp32 accumulation) on the GROUPED path, in fp32 on
 * the GENERIC path; everything else is fp32.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#include "qmoe.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_ACT_RELU = 0,
    MOE_ACT_GELU = 1,
    MOE_ACT_SILU = 2,
    MOE_ACT_SWIGLU = 3,
    MOE_ACT_IDENTITY = 4
} moe_activation;

/* Kernel path of moe_forward.  AUTO picks by shape.
 *   GROUPED : expert-grouped tcgen05 TF32 GEMMs (H and I multiples of 32,
 *             weight and activation rows 16-byte aligned)
 *   GENERIC : scalar fp32 kernels for any valid shape                       */
typedef enum { MOE_PATH_AUTO = 0, MOE_PATH_GROUPED = 2, MOE_PATH_GENERIC = 3 } moe_path;

/*
 * Attributes of the README's Attributes table.  moe_attrs_default sets its
 * defaults: k 1, activation relu, swiglu_fusion 0, alpha 1, beta 0, no
 * swiglu_limit, normalize_routing_weights 0, use_sparse_mixer 0, path AUTO.
 */
typedef struct {
    int64_t k;                          /* experts per token, 1 <= k <= E         */
    int32_t activation_type;            /* moe_activation                         */
    int32_t swiglu_fusion;              /* 0 (separate FC3), 1 interleaved, 2
                                           concatenated; 1 and 2 only with swiglu */
    float activation_alpha;             /* SwiGLU alpha                           */
    float activation_beta;              /* added to the SwiGLU linear branch      */
    int32_t has_swiglu_limit;           /* 0 = omitted (no clamp)                 */
    float swiglu_limit;
    int32_t normalize_routing_weights;  /* 0 or 1                                 */
    int32_t use_sparse_mixer;           /* must be 0                              */
    int32_t path;                       /* moe_path                               */
} moe_attrs;

void moe_attrs_default(moe_attrs *attrs);

/*
 * Workspace bytes moe_forward needs.  input_shape: [T, H] or [B, S, H]
 * (input_rank 2 or 3); fc1_w_shape: [E, fusion*I, H].  Returns
 * INVALID_ARGUMENT / NOT_SUPPORTED for shapes moe_forward would reject.
 */
qmoe_status moe_workspace_size(const int64_t *input_shape, int32_t input_rank,
                               const int64_t *fc1_w_shape, const moe_attrs *attrs,
                               size_t *bytes);

/* The kernel path moe_forward takes for these shapes (never AUTO). */
qmoe_status moe_choose_path(const int64_t *input_shape, int32_t input_rank,
                            const int64_t *fc1_w_shape, const moe_attrs *attrs, int32_t *path);

/*
 * The float MoE layer (README Inputs and Outputs).
 *   input         fp32 [T,H] or [B,S,H]                (input_rank 2 or 3)
 *   router_probs  fp32 [T,E] router LOGITS             (router_shape[2])
 *   fc1_w         fp32 [E, fusion*I, H]                (fc1_w_shape[3])
 *   fc1_bias      fp32 [E, fusion*I] or NULL
 *   fc2_w         fp32 [E, H, I]                       (fc2_w_shape[3])
 *   fc2_bias      fp32 [E, H] or NULL (added before the routing weight)
 *   fc3_w         fp32 [E, I, H] or NULL               (fc3_w_shape[3] or NULL)
 *   fc3_bias      fp32 [E, I] or NULL (used only with fc3_w)
 *   output        fp32, the shape of input
 * fusion = 2 for swiglu with swiglu_fusion 1 or 2, else 1.  FC3 is read only
 * by swiglu with swiglu_fusion 0 (where it is required) and by silu; other
 * activations ignore it.
 * topk_idx_out (int32 [T,k]) and topk_w_out (fp32 [T,k]) are optional device
 * outputs (NULL to skip): the selected experts in selection order and their
 * routing weights.  T == 0 is a no-op; I == 0 writes sum_i w_i * b2[sel_i]
 * (zeros without fc2_bias).
 * Errors: INVALID_ARGUMENT for ranks and shapes that disagree, k outside
 * [1,E], an unknown activation or swiglu_fusion, swiglu_fusion 1/2 with
 * another activation, swiglu_fusion 0 with swiglu and no fc3_w, NULL
 * required pointers; NOT_SUPPORTED for use_sparse_mixer 1 or a forced path
 * the shape cannot take; WORKSPACE_TOO_SMALL; CUDA for a failed launch.
 */
qmoe_status moe_forward(const float *input, const int64_t *input_shape, int32_t input_rank,
                        const float *router_probs, const int64_t *router_shape,
                        const float *fc1_w, const int64_t *fc1_w_shape, const float *fc1_bias,
                        const float *fc2_w, const int64_t *fc2_w_shape, const float *fc2_bias,
                        const float *fc3_w, const int64_t *fc3_w_shape, const float *fc3_bias,
                        float *output, const moe_attrs *attrs, void *workspace,
                        size_t workspace_bytes, int32_t *topk_idx_out, float *topk_w_out,
                        void *cuda_stream);

/*
 * moe_forward for callers whose activations live in HOST memory: host_input,
 * host_router_probs and host_output are host pointers (page-locked memory
 * gives asynchronous copies); weights and biases are device pointers.  The
 * call enqueues the host-to-device copies into the workspace, the layer, and
 * the device-to-host copy of the output on `cuda_stream`; host_output is
 * valid after the stream synchronizes.  The workspace must hold
 * moe_hostio_workspace_size bytes.
 */
qmoe_status moe_hostio_workspace_size(const int64_t *input_shape, int32_t input_rank,
                                      const int64_t *fc1_w_shape, const moe_attrs *attrs,
                                      size_t *bytes);

qmoe_status moe_forward_hostio(const float *host_input, const int64_t *input_shape,
                               int32_t input_rank, const float *host_router_probs,
                               const int64_t *router_shape, const float *fc1_w,
                               const int64_t *fc1_w_shape, const float *fc1_bias,
                               const float *fc2_w, const int64_t *fc2_w_shape,
                               const float *fc2_bias, const float *fc3_w,
                               const int64_t *fc3_w_shape, const float *fc3_bias,
                               float *host_output, const moe_attrs *attrs, void *workspace,
                               size_t workspace_bytes, void *cuda_stream);

/* Device error word of a workspace used by moe_forward (synchronizes the
 * stream first); same codes as qmoe_get_device_error. */
qmoe_status moe_get_device_error(const void *workspace, void *cuda_stream, int32_t *code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
