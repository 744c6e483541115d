// Internal declarations shared by the host dispatcher and the kernel files.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "qmoe.h"

namespace qmoe {

// Launch as a programmatic dependent of the previous kernel in the stream: the
// kernel may start while that kernel finishes, and must call griddepcontrol.wait
// before it reads anything the previous kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


// Problem description after host validation (QMoE manifest derive.*).
struct Problem {
    int64_t T = 0;        // derive.numTokens
    int64_t H = 0;        // derive.hiddenSize
    int64_t I = 0;        // derive.interSize
    int64_t E = 0;        // dim(router_probs, 1)
    int64_t k = 0;        // derive.topK
    int bits = 4;         // derive.weightBits
    int pack = 2;         // derive.packSize
    int mid = 8;          // derive.quantMidpoint
    int64_t bs = 0;       // derive.quantBlockSize (0 = column-wise)
    int64_t nb1 = 1;      // derive.fc1ScaleBlocks
    int64_t nb2 = 1;      // derive.fc2ScaleBlocks
    int act = 0;          // 0 relu, 1 swiglu
    int fusion = 1;       // derive.fusionSize
    float alpha = 1.f, beta = 0.f;
    int has_limit = 0;
    float limit = 0.f;
    int path = QMOE_PATH_GENERIC;
    int full_softmax = 0; // routing denominator over every expert (float MoE, unnormalised)
    // device tensors
    const float* x = nullptr;
    const float* logits = nullptr;
    const uint8_t* w1 = nullptr;
    const float* s1 = nullptr;
    const uint8_t* w2 = nullptr;
    const float* s2 = nullptr;
    float* y = nullptr;
};

// Sizes that depend only on the problem shape and path.
struct Plan {
    int64_t slots = 0;          // T * k
    int64_t route_chunks = 0;   // CTAs of the routing kernel (tokens per chunk below)
    int64_t Hp = 0;             // padded row length of the fp16 activations
    int64_t Ip = 0;             // padded row length of the fp16 FC1 output
    int64_t max_tiles = 0;      // expert token-tiles upper bound
    int tile_tokens = 0;        // tokens per expert tile (grouped path)
    int fc2_splits = 1;         // split-K factor of the decode FC2
    int64_t srows = 0;          // grouped path: rows of the K-blocked activation layouts
    size_t bytes = 0;           // total workspace bytes
    // byte offsets into the workspace
    size_t off_ctrl, off_sel, off_pw, off_counts, off_offsets, off_hist, off_rank, off_perm,
        off_inv, off_tiles, off_active, off_x16, off_xs16, off_act, off_slot_out;
};

// Device views of the workspace.
struct Work {
    int32_t* ctrl;        // [0] device error word
    int32_t* sel;         // [T*k] selected experts, selection order
    float* pw;            // [T*k] routing weights
    int32_t* counts;      // [E] slots per expert
    int32_t* offsets;     // [E+1] exclusive scan of counts
    int32_t* hist;        // [route_chunks*E] per-chunk counts, then chunk bases
    int32_t* rank;        // [T*k] stable rank of a slot within its chunk and expert
    int32_t* perm;        // [T*k] sorted position -> slot (t*k+i)
    int32_t* inv;         // [T*k] slot -> sorted position
    int32_t* tiles;       // [4 + 4*max_tiles] header + (expert, row0, rows, expert's first tile)
    int32_t* active;      // [E] experts with at least one slot, ascending
    __half* x16;          // [T*Hp] fp16 copy of the activations (decode path)
    __half* xs16;         // grouped path: fp16 activations in expert-sorted slot order,
                          // K-blocked [Hp/64][srows][64] with the 128-byte swizzle applied
    void* act;            // FC1 output: fp16 [T*k, Ip] (decode), fp32 (generic), or fp16
                          // K-blocked [Ip/64][srows][64] like xs16 (grouped)
    float* slot_out;      // [fc2_splits*T*k*H] per-slot FC2 output (fp32; the grouped path
                          // keeps [T*k*H] fp16 rows weighted by routing weight here)
};

constexpr int kRouteTokensPerChunk = 64;
constexpr int kTileHeader = 4;  // tiles[0] = number of tiles, tiles[1] = active experts

// Tuning constants of the paths.
constexpr int kDecodeMaxTokens = 16;  // AUTO takes the decode path up to this many tokens

// Host-side launch bookkeeping (profiling hooks, launch counter).
// begin=true before the launch(es) of `kernel_id`, begin=false after them with
// the number of kernels launched in between.
void note_launch(int kernel_id, cudaStream_t stream, bool begin, int nkernels = 1);

// Bound on a single in-kernel spin-wait, in nanoseconds, as set by the calling
// host thread (each thread has its own).
uint64_t wait_limit_ns();
// Pipeline stage the producers skip (test hook of the calling host thread), -1
// when off.
int64_t drop_stage();

// ---- launchers (return cudaGetLastError()) ----
// x16_mode: fp16 activation layout (0 natural, 1 4-bit pair order, 2 as 1 with the odd
// elements divided by 16 for the 4-bit decode kernel).
cudaError_t launch_route(const Problem& p, const Plan& pl, const Work& w, int x16_mode,
                         cudaStream_t s);
cudaError_t launch_group(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s);
// Routing and grouping in a single launch for small batches.
constexpr int kSmallRouteSlots = 4096;
bool small_route_ok(const Problem& p, const Plan& pl);
cudaError_t launch_route_group_small(const Problem& p, const Plan& pl, const Work& w,
                                     int x16_mode, cudaStream_t s);
cudaError_t launch_generic_fc1(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s);
cudaError_t launch_generic_fc2(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s);
// Grouping of arbitrary items by group id (shared by the layer and grouped_matmul).
cudaError_t launch_group_items(int32_t* hist, int64_t chunks, int E, int32_t* counts,
                               int32_t* offsets, int32_t* tiles, int32_t* active, int tile_tokens,
                               const int32_t* sel, const int32_t* rank, int64_t slots, int k,
                               int32_t* perm, int32_t* inv, cudaStream_t s);
// grouped_matmul on the tensor cores (f16/bf16): workspace bytes (0 when the
// shape or type does not qualify) and launch.
size_t grouped_matmul_tc_workspace(int64_t M, int64_t K, int64_t G, int64_t N, int64_t S,
                                   int dtype);
cudaError_t launch_grouped_matmul_tc(const void* input, int64_t M, int64_t K, const void* weights,
                                     int64_t G, int64_t N, const void* idx, int64_t S, int idx64,
                                     const void* bias, void* out, int dtype, void* workspace,
                                     cudaStream_t s);
// Grouped path: the FC2 rows are fp16 [T*k, H] and already weighted by routing weight.
cudaError_t launch_combine16(const Problem& p, const Work& w, cudaStream_t s);
cudaError_t launch_combine(const Problem& p, const Plan& pl, const Work& w, int splits,
                           cudaStream_t s);
// Decode path (few tokens): weight-streaming tensor-core GEMV.
bool decode_shape_ok(const Problem& p);
int decode_fc2_splits(const Problem& p);
cudaError_t launch_decode_fc(const Problem& p, const Plan& pl, const Work& w, bool fc1,
                             cudaStream_t s);
// Grouped path (many tokens): tcgen05 expert-grouped GEMMs.
int grouped_tile_tokens();
cudaError_t launch_sort_convert(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s);
bool grouped_shape_ok(const Problem& p);
cudaError_t launch_grouped_fc(const Problem& p, const Plan& pl, const Work& w, bool fc1,
                              cudaStream_t s);
cudaError_t launch_grouped_matmul(const void* input, int64_t M, int64_t K, const void* weights,
                                  int64_t G, int64_t N, const void* idx, int64_t S, int idx64,
                                  const void* bias, void* out, int dtype, int32_t* err,
                                  cudaStream_t s);

}  // namespace qmoe
