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
// obtained once per device with cudaGetSymbolAddress (with that device
// current) and cached.
#include <mutex>

#include "qmoe_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device).
qmoe_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QMOE_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
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

}  // extern "C"
