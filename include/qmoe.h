/*
 * qmoe.h -- C ABI of the GB300 (sm_103a) QMoE layer library.
 *
 * Two operations, each defined by a web page:
 *
 *  - qmoe_forward: the quantized mixture-of-experts layer of the
 *    com.microsoft.QMoE WebGPU kernel manifest (v1), keys `description`,
 *    `inputs`, `outputs`, `attributes`, `attributeDescriptions`,
 *    `attributeConstraints`, `typeConstraints` and `derive.*`.
 *    Per token t: pick the k largest router logits (descending, ties to the
 *    lower expert index), take the softmax over the k selected logits
 *    (for either value of normalize_routing_weights), run FC1 on the
 *    selected expert's symmetric 4/8-bit weights w = (q - mid) * scale
 *    (mid 8 or 128; column-wise or block-wise scales), apply ReLU or
 *    interleaved SwiGLU (row 2j gate, row 2j+1 linear,
 *    a = g * sigmoid(alpha*g) * (u + beta), optional clamp), run FC2, and sum
 *    the k expert outputs weighted by their routing probabilities.
 *
 *  - grouped_matmul: ONNX "GroupedMatMul - 29", section Summary:
 *    output[m, i] = input[m] @ weights[group_indices[m, i]] (+ bias[g]).
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller, unless a
 *    parameter says "host".  Tensors are dense, row-major, exactly in the
 *    layouts the pages give (last index fastest).
 *  - The library never allocates device memory.  Scratch comes from a
 *    caller-provided device workspace whose size the *_workspace_size
 *    function returns; it must be 256-byte aligned.
 *  - Work is enqueued asynchronously on `cuda_stream` (a cudaStream_t; NULL
 *    means the legacy default stream).  Nothing synchronizes the host
 *    except qmoe_get_device_error and qmoe_profile_end.
 *  - Shape and attribute errors are detected on the host before any launch
 *    and returned as a status; no C++ exception crosses the ABI.
 *  - Conditions only the GPU can see (an out-of-range group index, a
 *    non-finite 16-bit activation, a pipeline wait that timed out) write a
 *    code into the workspace's error word, never trap, and are read back
 *    with qmoe_get_device_error.
 *  - Calls on the same workspace must not overlap on the GPU.
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMOE_OK = 0,
    QMOE_ERR_INVALID_ARGUMENT = 1,   /* a shape, rank or attribute check failed */
    QMOE_ERR_NOT_SUPPORTED = 2,      /* valid ONNX value this layer excludes   */
    QMOE_ERR_WORKSPACE_TOO_SMALL = 3,
    QMOE_ERR_CUDA = 4                /* a CUDA runtime call failed             */
} qmoe_status;

/* Codes written into the workspace error word by the GPU. */
typedef enum {
    QMOE_DEVERR_NONE = 0,
    QMOE_DEVERR_INDEX = 1,           /* grouped_matmul index outside [0, G)    */
    QMOE_DEVERR_NONFINITE = 2,       /* a 16-bit intermediate overflowed       */
    QMOE_DEVERR_TIMEOUT = 3          /* a pipeline wait exceeded its limit     */
} qmoe_device_error;

typedef enum { QMOE_ACT_RELU = 0, QMOE_ACT_SWIGLU = 1 } qmoe_activation;

/* Kernel path of qmoe_forward.  AUTO picks by shape; the others force one
 * path and exist for tests and measurements.
 *   DECODE  : split-K weight-streaming GEMV (tensor-core m16n8k16), for few tokens
 *   GROUPED : expert-grouped tcgen05 GEMMs with TMEM accumulators
 *   GENERIC : scalar fp32 kernels for any valid shape (no alignment needs)   */
typedef enum {
    QMOE_PATH_AUTO = 0,
    QMOE_PATH_DECODE = 1,
    QMOE_PATH_GROUPED = 2,
    QMOE_PATH_GENERIC = 3
} qmoe_path;

/*
 * Attributes of the QMoE manifest (`attributes`, `attributeDescriptions`,
 * `attributeConstraints`).  qmoe_attrs_default sets the manifest defaults:
 * k 1, expert_weight_bits 4, block_size 0 (omitted => column-wise scales),
 * activation relu, swiglu_fusion 0, alpha 1, beta 0, no swiglu_limit,
 * normalize_routing_weights 0, use_sparse_mixer 0, weights_prepacked -1,
 * quant_type "int", path AUTO.
 */
typedef struct {
    int64_t k;                        /* experts per token, 1 <= k <= E          */
    int32_t expert_weight_bits;       /* 4 or 8                                  */
    int32_t activation_type;          /* qmoe_activation                         */
    int64_t block_size;               /* 0 = column-wise; else pow2 >= 16 that
                                         divides hidden and inter               */
    int32_t swiglu_fusion;            /* 0 with relu, 1 with swiglu (interleaved) */
    float activation_alpha;           /* SwiGLU alpha                            */
    float activation_beta;            /* added to the SwiGLU linear branch       */
    int32_t has_swiglu_limit;         /* 0 = omitted (no clamp)                  */
    float swiglu_limit;               /* clamp limit when has_swiglu_limit       */
    int32_t normalize_routing_weights;/* 0 or 1; same routing either way         */
    int32_t use_sparse_mixer;         /* must be 0                               */
    int32_t weights_prepacked;        /* -1 or 0 (raw packed layout)             */
    int32_t quant_type_is_int;        /* must be 1 (quant_type "int")            */
    int32_t path;                     /* qmoe_path                               */
} qmoe_attrs;

void qmoe_attrs_default(qmoe_attrs *attrs);

const char *qmoe_status_string(qmoe_status status);

/*
 * Workspace bytes qmoe_forward needs for these shapes and attributes.
 * input_shape: [T, H] or [B, S, H] (input_rank 2 or 3); fc1_w_shape: the
 * three dims of fc1_experts_weights [E, fusion*I, H/pack].  Returns
 * INVALID_ARGUMENT / NOT_SUPPORTED for shapes qmoe_forward would reject.
 */
qmoe_status qmoe_workspace_size(const int64_t *input_shape, int32_t input_rank,
                                const int64_t *fc1_w_shape, const qmoe_attrs *attrs,
                                size_t *bytes);

/* The kernel path qmoe_forward takes for these shapes (never AUTO). */
qmoe_status qmoe_choose_path(const int64_t *input_shape, int32_t input_rank,
                             const int64_t *fc1_w_shape, const qmoe_attrs *attrs,
                             int32_t *path);

/*
 * The QMoE layer (QMoE manifest: description, inputs[0..5], outputs[0]).
 *   input          fp32 [T,H] or [B,S,H]            (input_rank 2 or 3)
 *   router_probs   fp32 [T,E] router LOGITS          (router_shape[2])
 *   fc1_w          uint8 [E, fusion*I, H/pack]       (fc1_w_shape[3])
 *   fc1_scales     fp32 [E, fusion*I] or [E, fusion*I, H/block_size]
 *   fc2_w          uint8 [E, H, I/pack]              (fc2_w_shape[3])
 *   fc2_scales     fp32 [E, H] or [E, H, I/block_size]
 *   output         fp32, the shape of input
 * pack = 2 for 4-bit (element 2b in the low nibble of byte b) and 1 for 8-bit;
 * fusion = 2 for interleaved SwiGLU, else 1.
 * topk_idx_out (int32 [T,k]) and topk_w_out (fp32 [T,k]) are optional device
 * outputs (NULL to skip) holding the selected experts in selection order and
 * their routing weights.
 * T == 0 is a no-op; inter_size == 0 writes zeros (variant quant_zero_inter).
 * Errors: INVALID_ARGUMENT for a failed manifest predicate (quantContract:
 * ranks, shapes, k outside [1,E], block_size rule, fusion/activation
 * mismatch, NULL pointers); NOT_SUPPORTED for use_sparse_mixer 1,
 * weights_prepacked 1, quant_type other than int, bits other than 4/8;
 * WORKSPACE_TOO_SMALL; CUDA for a failed launch.
 */
qmoe_status qmoe_forward(const float *input, const int64_t *input_shape, int32_t input_rank,
                         const float *router_probs, const int64_t *router_shape,
                         const uint8_t *fc1_w, const int64_t *fc1_w_shape,
                         const float *fc1_scales, const int64_t *fc1_scales_shape,
                         int32_t fc1_scales_rank,
                         const uint8_t *fc2_w, const int64_t *fc2_w_shape,
                         const float *fc2_scales, const int64_t *fc2_scales_shape,
                         int32_t fc2_scales_rank,
                         float *output, const qmoe_attrs *attrs,
                         void *workspace, size_t workspace_bytes,
                         int32_t *topk_idx_out, float *topk_w_out, void *cuda_stream);

/*
 * qmoe_forward for callers whose activations live in HOST memory.
 * host_input, host_router_probs and host_output are host pointers (page-locked
 * memory gives asynchronous copies); the weights and scales are device
 * pointers as in qmoe_forward.  The call enqueues the host-to-device copies
 * into the workspace, the layer, and the device-to-host copy of the output on
 * `cuda_stream`; host_output is valid after the stream synchronizes.
 * When all three buffers are page-locked memory mapped into the device's
 * address space (cudaHostAlloc / cudaHostRegister, or any pinned allocation
 * under unified addressing) and the activations are at most
 * QMOE_HOSTIO_DIRECT_BYTES, no copy is enqueued: the routing and conversion
 * kernels read the inputs and the combine writes the output in place over the
 * host link (decode-sized calls, where each copy's fixed cost exceeds its
 * transfer time).  The results are the same.
 * The workspace must hold qmoe_hostio_workspace_size bytes.
 */
#define QMOE_HOSTIO_DIRECT_BYTES (1u << 20)
qmoe_status qmoe_hostio_workspace_size(const int64_t *input_shape, int32_t input_rank,
                                       const int64_t *fc1_w_shape, const qmoe_attrs *attrs,
                                       size_t *bytes);

qmoe_status qmoe_forward_hostio(const float *host_input, const int64_t *input_shape,
                                int32_t input_rank,
                                const float *host_router_probs, const int64_t *router_shape,
                                const uint8_t *fc1_w, const int64_t *fc1_w_shape,
                                const float *fc1_scales, const int64_t *fc1_scales_shape,
                                int32_t fc1_scales_rank,
                                const uint8_t *fc2_w, const int64_t *fc2_w_shape,
                                const float *fc2_scales, const int64_t *fc2_scales_shape,
                                int32_t fc2_scales_rank,
                                float *host_output, const qmoe_attrs *attrs,
                                void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * qmoe_forward for callers that cannot allocate device memory -- for example
 * an extension hosted by a runtime that owns the whole device memory pool and
 * gives its plugins no allocator, or a latency-critical loop that cannot
 * afford the implicit device synchronization of cudaMalloc.  The operator
 * pages define no such call; it is an addition of this library.
 *
 * Same arguments and results as qmoe_forward, without the workspace: the
 * layer's scratch is a fixed array of qmoe_noalloc_scratch_bytes() (4 MiB)
 * compiled into the library's device image, so every GPU that loads the
 * library holds that memory until the process exits.  The call allocates
 * nothing and calls no allocating routine.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it with
 *    the identity of the current CUDA context; make that first call before
 *    any stream capture.  An address is valid in one context only: when a
 *    later call finds another context current on the device (a host runtime
 *    that runs it in its own context, or a new primary context after
 *    cudaDeviceReset), it looks the address up again in that context, so
 *    that first call in the new context should also come before any capture.
 *  - Shapes whose qmoe_workspace_size exceeds the array are rejected with
 *    QMOE_ERR_WORKSPACE_TOO_SMALL before anything is launched (decode-sized
 *    batches fit; large prefill batches do not).
 *  - Every call uses the same array, which keeps the previous call's
 *    contents (the layer rewrites everything it reads, including the device
 *    error word).  Calls that can overlap on the GPU -- different streams, or
 *    host threads without ordering -- race on it and must be serialized by
 *    the caller.  Their device error word is read with
 *    qmoe_noalloc_get_device_error, not qmoe_get_device_error.
 */
size_t qmoe_noalloc_scratch_bytes(void);

qmoe_status qmoe_forward_noalloc(const float *input, const int64_t *input_shape,
                                 int32_t input_rank,
                                 const float *router_probs, const int64_t *router_shape,
                                 const uint8_t *fc1_w, const int64_t *fc1_w_shape,
                                 const float *fc1_scales, const int64_t *fc1_scales_shape,
                                 int32_t fc1_scales_rank,
                                 const uint8_t *fc2_w, const int64_t *fc2_w_shape,
                                 const float *fc2_scales, const int64_t *fc2_scales_shape,
                                 int32_t fc2_scales_rank,
                                 float *output, const qmoe_attrs *attrs,
                                 int32_t *topk_idx_out, float *topk_w_out, void *cuda_stream);

/*
 * Device error word of the last qmoe_forward_noalloc call(s) on the current
 * device: the kernels record a qmoe_device_error value there (an fp16
 * intermediate out of range, a pipeline wait past its limit) instead of
 * trapping.  The word is read and then cleared in stream order on
 * `cuda_stream` (after the calls enqueued on it before), and the stream is
 * synchronized before *code is set.  Allocates nothing.  Like the calls
 * themselves it shares the fixed array: it must not overlap on the GPU with a
 * qmoe_forward_noalloc call on another stream.  The operator pages have no
 * counterpart to it.
 */
qmoe_status qmoe_noalloc_get_device_error(void *cuda_stream, int32_t *code);

/* Element types of grouped_matmul (GroupedMatMul-29, Type Constraints). */
typedef enum { QMOE_DT_F32 = 0, QMOE_DT_F16 = 1, QMOE_DT_BF16 = 2, QMOE_DT_F64 = 3 } qmoe_dtype;
typedef enum { QMOE_IDX_I32 = 0, QMOE_IDX_I64 = 1 } qmoe_index_dtype;

/* Workspace bytes grouped_matmul needs at least (it holds the device error word). */
qmoe_status grouped_matmul_workspace_size(size_t *bytes);

/*
 * Workspace bytes that let grouped_matmul run on the tensor cores for this
 * shape: f16 or bf16, K a multiple of 64, N a multiple of 8, G <= 8191, with
 * input, weights and output 16-byte aligned.  The workspace then holds the
 * grouping of the (m, i) rows by index and the input rows gathered in group
 * order (about 2 * K * M * S bytes).  For other shapes and types *bytes is the
 * minimum of grouped_matmul_workspace_size.  A smaller workspace is valid: the
 * call then uses the general kernel (fp32 accumulation either way).
 */
qmoe_status grouped_matmul_workspace_size_for(int64_t M, int64_t K, int64_t G, int64_t N,
                                              int64_t S, int32_t dtype, size_t *bytes);

/*
 * GroupedMatMul-29 (Summary, Inputs, Outputs):
 *   input          T [M,K]
 *   weights        T [G,K,N]
 *   group_indices  Tind [M,S] (index_dtype int32 or int64)
 *   bias           T [G,N] or NULL (absent / explicit empty input)
 *   output         T [M,S,N]
 * T is one of qmoe_dtype for input, weights, bias and output alike.
 * Accumulation is fp32 for f32/f16/bf16 and fp64 for f64.
 * M == 0 or S == 0 or N == 0 is a no-op.  K == 0 gives bias (or zeros).
 * An index outside [0,G) is invalid input on the page; here that (m,i) row
 * of the output is written as zeros and the device error word is set to
 * QMOE_DEVERR_INDEX.
 */
qmoe_status grouped_matmul(const void *input, int64_t M, int64_t K,
                           const void *weights, int64_t G, int64_t N,
                           const void *group_indices, int64_t S, int32_t index_dtype,
                           const void *bias, void *output, int32_t dtype,
                           void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Reads (and clears) the device error word of a workspace used by
 * qmoe_forward or grouped_matmul.  Synchronizes `cuda_stream` first.
 * *code receives a qmoe_device_error value.
 */
qmoe_status qmoe_get_device_error(void *workspace, void *cuda_stream, int32_t *code);

/*
 * Upper bound, in nanoseconds, on any single spin-wait inside a kernel
 * (mbarrier or flag).  When a wait exceeds it the kernel records
 * QMOE_DEVERR_TIMEOUT, drains its own copies in flight, releases its tensor
 * memory and returns.  Default 2 s.  Per host thread: it applies to the
 * launches the calling thread makes from its next call on, and leaves other
 * threads' launches at their own setting.
 */
void qmoe_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook for the timeout path (no counterpart on the operator pages).
 * When stage >= 0, the TMA producer of every pipelined kernel launched after
 * this call skips the copies of its pipeline stage number `stage` (counted
 * from 0 per CTA), so the consumers' wait on that stage never completes and
 * must end through the wait limit with QMOE_DEVERR_TIMEOUT.  -1 (the default)
 * turns it off.  Per host thread: only the launches of the calling thread
 * skip the stage, so a hook set by one thread cannot make a layer that another
 * thread runs at the same time wait and fail.
 */
void qmoe_debug_drop_stage(int64_t stage);

/* Kernel identifiers for qmoe_profile_begin. */
typedef enum {
    QMOE_KERNEL_ROUTE = 0,
    QMOE_KERNEL_GROUP = 1,
    QMOE_KERNEL_FC1 = 2,
    QMOE_KERNEL_FC2 = 3,
    QMOE_KERNEL_COMBINE = 4,
    QMOE_KERNEL_GMM = 5              /* grouped_matmul's GEMM                    */
} qmoe_kernel_id;

/*
 * Per-kernel device timing.  After qmoe_profile_begin(id), each launch of
 * kernel `id` is bracketed by CUDA events on the launching stream.  An id
 * outside the enum returns INVALID_ARGUMENT.  The ids name steps of the
 * library's entry points:
 *   qmoe_forward, moe_forward: ROUTE the routing kernel, GROUP the grouping
 *     launches, FC1 / FC2 the two expert projections, COMBINE the weighted sum;
 *   matmul_nbits_qkv (qkv.h): ROUTE the RMSNorm kernel, FC1 the Q/K/V
 *     projection, COMBINE the split-K reduction;
 *   grouped_matmul: GMM its GEMM (the tensor-core kernel or the general one).
 * qmoe_profile_end synchronizes those events and returns how many
 * launches were bracketed and their summed duration in milliseconds, then
 * stops recording.
 */
qmoe_status qmoe_profile_begin(int32_t kernel_id);
qmoe_status qmoe_profile_end(int64_t *launches, double *total_ms);

/* Number of kernels (and memset nodes) this library has enqueued since the
 * process started, summed over all threads. */
uint64_t qmoe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H */
