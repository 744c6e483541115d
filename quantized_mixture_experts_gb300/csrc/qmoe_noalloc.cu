// qmoe_forward_noalloc: the QMoE layer for callers that cannot allocate device
// memory, using a fixed scratch array that lives in the library's own device
// image instead of a caller-provided workspace.
//
// Who needs this: code that must not (or cannot) call cudaMalloc at run time,
// for example an extension hosted by a runtime that owns the whole device
// memory pool and hands its plugins no allocator, or a latency-critical loop
// where the implicit device synchronization of cudaMalloc is not acceptable.
// Such a caller still passes its own input, weight and output tensors; only
// the scratch space the layer needs internally comes from here.
//
// The array below is a file-scope __device__ object: every GPU that loads
// this library holds kNoAllocScratchBytes of it until the process exits.  In
// host code its name is only a host-side stand-in; its device address is
// obtained with cudaGetSymbolAddress (with the device current) and cached per
// device together with the identity of the CUDA context it was obtained in.
// An address belongs to one context: when the current context of a device is
// another one (a host runtime that runs the call in its own context, or a new
// primary context after cudaDeviceReset), the lookup is done again, so a
// stale address from an earlier context is never used.
#include <cuda.h>

#include <mutex>

#include "qmoe_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Context identity through the driver API, resolved once through the runtime
// (the library does not link libcuda).  cuCtxGetId gives an identifier that
// is never reused within the process, unlike a context handle's value.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxApi {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const CtxApi& ctx_api() {
    static CtxApi api;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            api.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            api.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return api;
}

// Identifier of the calling thread's current context; false when there is none
// yet (the runtime creates the primary context lazily) or the query fails.
bool current_ctx_id(unsigned long long* id) {
    const CtxApi& api = ctx_api();
    if (!api.get_current || !api.get_id) return false;
    CUcontext c = nullptr;
    if (api.get_current(&c) != CUDA_SUCCESS || !c) return false;
    return api.get_id(c, id) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
struct Cached {
    unsigned long long ctx_id = 0;
    void* ptr = nullptr;
};
std::mutex g_noalloc_mu;
Cached g_noalloc[kMaxDevices];

// Device address of the scratch array in the current device's current context.
// The first call in a context looks it up (make it before any stream capture).
qmoe_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    unsigned long long id = 0;
    const bool have_id = current_ctx_id(&id);
    if (have_id && g_noalloc[dev].ptr && g_noalloc[dev].ctx_id == id) {
        *out = g_noalloc[dev].ptr;
        return QMOE_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QMOE_ERR_CUDA;
    // the lookup makes the primary context current if nothing was current before
    if (!have_id && !current_ctx_id(&id)) {
        // no context identity available: use the address for this call only
        g_noalloc[dev] = Cached{};
        *out = p;
        return QMOE_OK;
    }
    g_noalloc[dev].ctx_id = id;
    g_noalloc[dev].ptr = p;
    *out = p;
    return QMOE_OK;
}

}  // namespace

extern "C" {

size_t qmoe_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

qmoe_status qmoe_forward_noalloc(const float* input, const int64_t* input_shape,
                                 int32_t input_rank, const float* router_probs,
                                 const int64_t* router_shape, const uint8_t* fc1_w,
                                 const int64_t* fc1_w_shape, const float* fc1_scales,
                                 const int64_t* fc1_scales_shape, int32_t fc1_scales_rank,
                                 const uint8_t* fc2_w, const int64_t* fc2_w_shape,
                                 const float* fc2_scales, const int64_t* fc2_scales_shape,
                                 int32_t fc2_scales_rank, float* output, const qmoe_attrs* attrs,
                                 int32_t* topk_idx_out, float* topk_w_out, void* cuda_stream) {
    size_t need = 0;
    qmoe_status st = qmoe_workspace_size(input_shape, input_rank, fc1_w_shape, attrs, &need);
    if (st != QMOE_OK) return st;
    if (need > kNoAllocScratchBytes) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != QMOE_OK) return st;
    return qmoe_forward(input, input_shape, input_rank, router_probs, router_shape, fc1_w,
                        fc1_w_shape, fc1_scales, fc1_scales_shape, fc1_scales_rank, fc2_w,
                        fc2_w_shape, fc2_scales, fc2_scales_shape, fc2_scales_rank, output, attrs,
                        scratch, kNoAllocScratchBytes, topk_idx_out, topk_w_out, cuda_stream);
}

qmoe_status qmoe_noalloc_get_device_error(void* cuda_stream, int32_t* code) {
    if (!code) return QMOE_ERR_INVALID_ARGUMENT;
    void* scratch = nullptr;
    qmoe_status st = noalloc_scratch(&scratch);
    if (st != QMOE_OK) return st;
    // the error word is the first word of the scratch (the layer's workspace
    // layout); read and clear it in stream order after the calls enqueued before
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), s) != cudaSuccess) return QMOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QMOE_ERR_CUDA;
    *code = v;
    return QMOE_OK;
}

}  // extern "C"
